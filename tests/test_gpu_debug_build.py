"""The bounds-checked build (libkda_debug.so, KDA_DEBUG): its checks fire on an out-of-range index
without making the access, and the GPU parity suites pass through it with no out-of-bounds access
flagged (every call there ends in check_device_status, which would raise on the bit)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code_or_args, timeout=900):
    env = dict(os.environ, KDA_DEBUG_BUILD="1")
    cmd = [sys.executable] + code_or_args
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_product_build_compiles_the_checks_away():
    import gated_linear_attention_kda_gb300 as kda
    assert not kda.debug_build()
    assert kda.probe_bounds() == [1, 1]
    kda.check_device_status()  # nothing flagged


def test_checked_build_catches_an_out_of_range_index_without_the_access():
    r = _run(["-c", "import gated_linear_attention_kda_gb300 as kda\n"
                    "assert kda.debug_build() and kda.LIB_PATH.endswith('libkda_debug.so')\n"
                    "assert kda.probe_bounds() == [0, 0]\n"
                    "try:\n    kda.check_device_status()\nexcept kda.KDAError as e:\n"
                    "    assert 'out-of-bounds' in str(e), e\nelse:\n    raise SystemExit('no flag')\n"
                    "kda.check_device_status()\nprint('ok')\n"])
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_parity_suites_pass_through_the_checked_build():
    """Every parity test except the full-size ones (their oracle time dominates), including the
    per-step slot checks of the tcgen05 kernel and the shared-preparation kernel's cases, through
    libkda_debug.so."""
    r = _run(["-m", "pytest", "-q", "-x", "-m", "gpu", "-k", "not full", "-p", "no:cacheprovider",
              "tests/test_gpu_parity.py", "tests/test_gpu_chunk32.py", "tests/test_gpu_slot_steps.py",
              "tests/test_gpu_shared_prep.py", "tests/test_gpu_failure_paths.py"], timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    import re
    m = re.search(r"(\d+) passed", r.stdout)
    # the suites ran in full (145 tests at the time of writing, 24 of them the shared-preparation
    # kernel's), not an empty or partial selection
    assert m and int(m.group(1)) >= 140, r.stdout[-2000:]
