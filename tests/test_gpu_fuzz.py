"""Seeded random combinations of the call's options, each against the fp64 oracle with the parity
tolerance: batch or varlen (with empty and ragged sequences), lengths around chunk boundaries, head
counts that pick either forward kernel and every V split, lower_bound anywhere in [-5, 0], gate
parameters on or off, no / bf16 / fp32 states (in place or not), CHUNK = 16 or 32, and q/k
normalised in the kernel."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

CASES = 64


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.choice([1, 2, 3, 5, 8, 40, 80]))
    varlen = rng.random() < 0.35
    lb = float(rng.choice([0.0, -5.0, rng.uniform(-5.0, 0.0)]))
    chunk = 32 if rng.random() < 0.3 else 16
    qkn = chunk == 16 and rng.random() < 0.25
    state = str(rng.choice(["none", "bf16", "fp32"]))
    in_place = state != "none" and rng.random() < 0.3
    if varlen:
        n = int(rng.integers(1, 7))
        lengths = [int(x) for x in rng.integers(0, 90, n)]
        if sum(lengths) == 0:
            lengths[0] = 1
        d = W.make("varlen_n16_h32", lengths=lengths, H=H, seed=seed, raw_qk=qkn)
        nseq = n
    else:
        B = int(rng.integers(1, 4))
        T = int(rng.choice([1, 15, 16, 17, 31, 32, 33, int(rng.integers(1, 200))]))
        d = W.make("b2_t128_h8", B=B, T=T, H=H, seed=seed, raw_qk=qkn)
        nseq = B
    if rng.random() < 0.5:
        d["A_log"], d["dt_bias"] = None, None
    if state == "none":
        d["initial_state"] = None
    else:
        dt = torch.bfloat16 if state == "bf16" else torch.float32
        d["initial_state"] = (torch.randn(nseq, H, 128, 128, generator=torch.Generator().manual_seed(seed)) * 0.02).to(dt)
    final = None if state == "none" and rng.random() < 0.3 else ("bf16" if state == "bf16" else "fp32")
    return d, dict(lower_bound=lb, chunk=chunk, qk_l2norm=qkn, in_place=in_place, final_dtype=final)


@pytest.mark.parametrize("seed", range(CASES))
def test_random_option_combinations_match_the_oracle(seed):
    d, kw = _case(seed)
    heads = None if d["q"].shape[2] < 8 else [0, d["q"].shape[2] - 1]
    o, s = run_gpu(d, final_dtype=kw["final_dtype"], in_place=kw["in_place"], lower_bound=kw["lower_bound"],
                   qk_l2norm=kw["qk_l2norm"], chunk=kw["chunk"])
    o_ref, s_ref = run_oracle(d, heads=heads, lower_bound=kw["lower_bound"], qk_l2norm=kw["qk_l2norm"])
    if heads is not None:
        o, s = o[:, :, heads], (None if s is None else s[:, heads])
    assert_close(f"out ({kw})", o, o_ref)
    if s is not None:
        assert_close(f"final_state ({kw})", s, s_ref)
