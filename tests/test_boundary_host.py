"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__
    __graft_entry__._builder().build_library()
    import gated_linear_attention_kda_gb300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    assert {"kda_fwd", "kda_fwd_flat", "kda_fwd_packed", "kda_fwd_host", "kda_fwd_ex", "kda_decode",
            "kda_decode_ex", "kda_check_device_status", "kda_last_error", "kda_plan", "kda_gate_scale",
            "kda_version", "kda_fwd_ws", "kda_fwd_workspace_bytes", "kda_fwd_static"} <= set(syms)


def test_library_exports_every_declared_symbol(kda):
    lib = ctypes.CDLL(kda.LIB_PATH)
    for s in declared_symbols():
        assert hasattr(lib, s), f"libkda.so does not export {s}"



def test_struct_entry_layout_matches_the_header(kda, tmp_path):
    """The ctypes mirror of kda_fwd_args has the C struct's size and field offsets
    (a C program including the header prints them), and a NULL struct is rejected."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in kda.FwdArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"kda.h\"\nint main(void) {\n"
                   + 'printf("%zu\\n", sizeof(kda_fwd_args));\n'
                   + "".join(f'printf("%zu\\n", offsetof(kda_fwd_args, {f}));\n' for f in fields)
                   + "return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(kda.FwdArgs)
    assert got[1:] == [getattr(kda.FwdArgs, f).offset for f in fields]
    assert kda.library().kda_fwd_packed(None, None) == 1  # KDA_ERR_NULL


def test_gate_scale_matches_the_page_constant(kda):
    # gate_scale = float(lower_bound * 1.4426950408889634): "Conversion to the Gate Scale Factor"
    import numpy as np
    for lb in (-5.0, -2.0, -0.5, 0.0):
        assert kda.gate_scale(lb) == np.float32(lb * 1.4426950408889634)


def test_plan_fills_the_machine(kda):
    assert kda.plan(128, 152) == (1, 128)     # one CTA per state
    assert kda.plan(32, 152) == (4, 128)      # V rows split four ways
    assert kda.plan(16, 152) == (8, 128)
    assert kda.plan(1, 152) == (8, 8)
    assert kda.plan(512, 152) == (1, 512)
    assert kda.plan(0, 152) == (8, 0)
    with pytest.raises(ValueError):
        kda.plan(-1, 152)
    with pytest.raises(ValueError):
        kda.plan(4, 0)


def _call(kda, **over):
    """Direct C-ABI call with dummy (never dereferenced) aligned pointers."""
    args = dict(q=0x1000, k=0x2000, v=0x3000, g=0x4000, beta=0x5000, scale=1.0, out=0x6000, A_log=None,
                dt_bias=None, lb=-5.0, init=None, init_dt=0, fin=None, fin_dt=0, cu=None, N=0,
                B=1, T=16, H=1, K=128, V=128, stream=None)
    args.update(over)
    lib = kda.library()
    return lib.kda_fwd(*[args[x] for x in ("q", "k", "v", "g", "beta", "scale", "out", "A_log", "dt_bias", "lb",
                                           "init", "init_dt", "fin", "fin_dt", "cu", "N", "B", "T", "H", "K",
                                           "V", "stream")])


@pytest.mark.parametrize("over,code", [
    (dict(K=64), 2), (dict(V=256), 2), (dict(H=0), 2), (dict(B=0), 2), (dict(T=-1), 2),
    (dict(cu=0x7000, B=2, N=1), 2), (dict(cu=0x7000, N=0), 2),
    (dict(q=None), 1), (dict(beta=None), 1), (dict(out=None), 1),
    (dict(lb=-5.5), 4), (dict(lb=0.25), 4), (dict(lb=float("nan")), 4), (dict(scale=float("inf")), 4),
    (dict(init=0x8000, init_dt=0), 3), (dict(init=None, init_dt=1), 3), (dict(fin=0x8000, fin_dt=7), 3),
    (dict(init=0x8000, init_dt=1, fin=0x9000000, fin_dt=2), 5),
    (dict(init=0x100000, init_dt=2, fin=0x100000 + 4096, fin_dt=2), 5),
    (dict(q=0x1008), 6), (dict(out=0x6002), 6), (dict(beta=0x5001), 6),
    (dict(init=0x8008, init_dt=2), 6), (dict(cu=0x7004, N=1), 6),
    # the largest problems: a token axis of 2^31 - 32 or more, more than 2^20 heads, more than 2^28 states
    (dict(B=1, T=(1 << 31) - 16), 2), (dict(B=2, T=(1 << 30)), 2), (dict(H=(1 << 20) + 1), 2),
    (dict(B=1 << 20, T=1, H=1 << 9), 2),
])
def test_host_validation_rejects(kda, over, code):
    assert _call(kda, **over) == code
    assert kda.library().kda_last_error()



def test_plain_c_program_uses_the_abi(kda, tmp_path):
    """A C program built against include/kda.h and linked to libkda.so (no Python, no CUDA
    headers) runs the host-side parts of the ABI."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = os.path.join(ROOT, "tests", "c_abi_consumer.c")
    libdir = os.path.dirname(kda.LIB_PATH)
    exe = str(tmp_path / "c_abi_consumer")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                    "-L", libdir, "-lkda", f"-Wl,-rpath,{libdir}", "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 11


@pytest.mark.parametrize("flags", [2, 4, 0x80000000, 3, 6])
def test_unknown_option_bits_are_rejected_on_the_host(kda, flags):
    lib = kda.library()
    if flags & ~3:  # KDA_FLAG_QK_L2NORM and KDA_FLAG_CHUNK32 are the forward pass's bits
        st = lib.kda_fwd_ex(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 0, None, 0,
                            None, 0, 1, 16, 1, 128, 128, flags, None)
        assert st == 4 and b"option bits" in lib.kda_last_error()
    st = lib.kda_decode_ex(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, 0x10000, 2,
                           2, 3, 128, 128, flags, None)
    assert st == 4 and b"option bits" in lib.kda_last_error()


def test_option_entry_points_validate_like_the_plain_ones(kda):
    lib = kda.library()
    assert lib.kda_fwd_ex(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 0, None, 0,
                          None, 0, 1, 16, 1, 64, 128, 1, None) == 2  # K != 128 with the flag set
    assert lib.kda_decode_ex(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 2,
                             2, 3, 128, 128, 1, None) == 1  # state NULL


def test_chunk32_flag_is_validated_on_the_host(kda):
    lib = kda.library()
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 0, None, 0, None, 0, 1, 16, 1)
    assert lib.kda_fwd_ex(*args, 128, 128, 3, None) == 4  # with KDA_FLAG_QK_L2NORM: KDA_ERR_RANGE
    assert b"does not combine" in lib.kda_last_error()
    assert lib.kda_fwd_ex(*args, 64, 128, 2, None) == 2  # K != 128: KDA_ERR_SHAPE, as without the flag
    with pytest.raises(ValueError, match="chunk must be 16 or 32"):
        kda.fwd(*([None] * 7), chunk=64)


def test_bounds_checked_build_exports_every_declared_symbol(kda):
    """libkda_debug.so (the same sources with KDA_DEBUG) builds and exports the whole ABI; it says
    it is the checked build, the product library says it is not."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("_kda_build_t", os.path.join(ROOT, "gated_linear_attention_kda_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = ctypes.CDLL(b.build_library(debug=True))
    for s in declared_symbols():
        assert hasattr(lib, s), f"libkda_debug.so does not export {s}"
    assert lib.kda_debug_build() == 1 and kda.library().kda_debug_build() == 0


def test_wait_timeout_probe_checks_its_arguments_on_the_host(kda):
    lib = kda.library()
    assert lib.kda_probe_wait_timeout(16, None, None) == 1  # KDA_ERR_NULL
    assert lib.kda_probe_wait_timeout(0, 0x1000, None) == 4  # KDA_ERR_RANGE
    assert lib.kda_probe_wait_timeout((1 << 18) + 1, 0x1000, None) == 4


@pytest.mark.parametrize("value", ["3", "0", "16", "x"])
def test_v_split_override_rejects_bad_values(kda, monkeypatch, value):
    monkeypatch.setenv("KDA_V_SPLIT", value)
    assert _call(kda) == 4  # KDA_ERR_RANGE, before anything touches a GPU
    assert b"KDA_V_SPLIT" in kda.library().kda_last_error()


def _decode_call(kda, **over):
    """Direct kda_decode call with dummy (never dereferenced) aligned pointers."""
    args = dict(q=0x1000, k=0x2000, v=0x3000, g=0x4000, beta=0x5000, scale=1.0, out=0x6000, A_log=None,
                dt_bias=None, lb=-5.0, state=0x10000, st_dt=2, S=2, H=3, K=128, V=128, stream=None)
    args.update(over)
    return kda.library().kda_decode(*[args[x] for x in ("q", "k", "v", "g", "beta", "scale", "out", "A_log",
                                                        "dt_bias", "lb", "state", "st_dt", "S", "H", "K", "V",
                                                        "stream")])


@pytest.mark.parametrize("over,code", [
    (dict(K=64), 2), (dict(V=96), 2), (dict(S=0), 2), (dict(H=0), 2),
    (dict(q=None), 1), (dict(state=None), 1), (dict(out=None), 1),
    (dict(st_dt=0), 3), (dict(st_dt=5), 3),
    (dict(lb=-6.0), 4), (dict(lb=1e-3), 4), (dict(scale=float("nan")), 4),
    (dict(q=0x1004), 6), (dict(state=0x10008), 6), (dict(out=0x6001), 6),
])
def test_decode_host_validation_rejects(kda, over, code):
    assert _decode_call(kda, **over) == code
    assert kda.library().kda_last_error()

def test_python_wrapper_rejects_bad_tensors(kda):
    import torch
    q = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16)
    beta = torch.zeros(1, 16, 1, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        kda.fwd(q, q, q, q, beta, 1.0, q.clone())
    with pytest.raises(ValueError, match="CPU tensor|contiguous|bfloat16|shape"):
        kda.fwd_host(q, q, q, q, beta.float(), 1.0, q.clone())
    with pytest.raises(ValueError, match="contiguous"):
        qt = torch.zeros(1, 16, 1, 256, dtype=torch.bfloat16)[..., :128]
        kda.fwd_host(qt, q, q, q, beta, 1.0, q.clone())


def test_python_wrapper_rejects_tensors_on_another_device(kda):
    """Every tensor must live on q's device (the library launches there and dereferences every
    pointer there). The device check is reached on the host path with a tensor on the `meta`
    device standing in for a second device; the decode wrapper shares the same check."""
    import torch
    q = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16)
    beta = torch.zeros(1, 16, 1, dtype=torch.bfloat16)
    other = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16, device="meta")
    for pos in range(1, 4):
        args = [q, q, q, q]
        args[pos] = other
        with pytest.raises(ValueError, match="all tensors must share one device"):
            kda.fwd_host(*args, beta, 1.0, q.clone())
    with pytest.raises(ValueError, match="out is on meta"):
        kda.fwd_host(q, q, q, q, beta, 1.0, other)
    with pytest.raises(ValueError, match="beta is on meta"):
        kda.fwd_host(q, q, q, q, beta.to("meta"), 1.0, q.clone())
    st = torch.zeros(1, 1, 128, 128, dtype=torch.float32)
    with pytest.raises(ValueError, match="final_state is on meta"):
        kda.fwd_host(q, q, q, q, beta, 1.0, q.clone(), initial_state=st, final_state=st.to("meta"))
    kda._same_device(q.device, (("k", q), ("state", st)))  # same device: accepted
    with pytest.raises(ValueError, match="state is on meta"):
        kda._same_device(q.device, (("k", q), ("state", st.to("meta"))))


def test_host_entry_checks_its_host_cu_seqlens_before_any_copy(kda):
    """kda_fwd_host reads cu_seqlens on the host (to cut the call into pieces): bounds that do not
    rise from 0 to T are KDA_ERR_SHAPE before any CUDA call."""
    import ctypes
    import numpy as np
    lib = kda.library()
    for bad in ([0, 5, 3, 8], [1, 4, 8], [0, 4, 9], [0, 4, 7]):
        cu = np.array(bad, dtype=np.int64)
        st = lib.kda_fwd_host(None, None, None, None, None, 1.0, None, None, None, -5.0, None, 0, None, 0,
                              cu.ctypes.data_as(ctypes.c_void_p), len(bad) - 1, 1, 8, 2, 128, 128, None)
        assert st == 2, bad  # KDA_ERR_SHAPE
        assert b"cu_seqlens" in lib.kda_last_error()


def test_workspace_entry_points_validate_on_the_host(kda):
    """kda_fwd_ws checks its workspace's alignment and then every argument as kda_fwd_ex does;
    kda_fwd_workspace_bytes rejects a NULL result pointer and bad sizes. No GPU is touched."""
    lib = kda.library()
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 0, None, 0, None, 0, 1, 16, 1)
    assert lib.kda_fwd_ws(*args, 128, 128, 0, 0x7001, 1 << 20, None) == 6  # misaligned workspace: KDA_ERR_ALIGN
    assert b"workspace" in lib.kda_last_error()
    assert lib.kda_fwd_ws(*args, 64, 128, 0, 0x7000, 1 << 20, None) == 2  # K != 128: KDA_ERR_SHAPE
    assert lib.kda_fwd_ws(*args, 128, 128, 4, 0x7000, 1 << 20, None) == 4  # unknown option bit: KDA_ERR_RANGE
    assert lib.kda_fwd_workspace_bytes(1, 1, 0, None) == 1
    n = ctypes.c_size_t(7)
    assert lib.kda_fwd_workspace_bytes(-1, 1, 0, ctypes.byref(n)) == 2
    assert lib.kda_fwd_workspace_bytes(1, 0, 0, ctypes.byref(n)) == 2
    assert n.value == 7  # untouched on error


def test_static_entry_point_validates_like_fwd_ex(kda):
    """kda_fwd_static reports argument errors exactly as kda_fwd_ex does (no GPU touched), and
    its scratch limit matches the header's."""
    lib = kda.library()
    args = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -5.0, None, 0, None, 0, None, 0, 1, 16, 1)
    assert lib.kda_fwd_static(*args, 64, 128, 0, None) == 2  # K != 128: KDA_ERR_SHAPE
    assert lib.kda_fwd_static(*args, 128, 128, 4, None) == 4  # unknown option bit: KDA_ERR_RANGE
    assert b"option bits" in lib.kda_last_error()
    assert lib.kda_fwd_static(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1.0, 0x6000, None, None, -6.0, None, 0, None,
                              0, None, 0, 1, 16, 1, 128, 128, 0, None) == 4  # lower_bound outside [-5, 0]
    hdr = open(HEADER).read()
    assert re.search(r"#define KDA_STATIC_SCRATCH_STATES (\d+)", hdr).group(1) == str(kda.STATIC_SCRATCH_STATES)
