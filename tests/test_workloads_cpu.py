"""The seeded workload recipe and the benchmark's algorithmic byte count (CPU only)."""
import math

import torch

import bench
import workloads as W


def test_raw_qk_keeps_every_other_draw():
    a = W.make("b2_t128_h8", T=40)
    b = W.make("b2_t128_h8", T=40, raw_qk=True)
    for name in ("v", "g", "beta", "A_log", "dt_bias", "initial_state"):
        assert torch.equal(a[name], b[name]), name
    na = a["k"].float().norm(dim=-1)
    nb = b["k"].float().norm(dim=-1)
    assert torch.allclose(na, torch.ones_like(na), atol=1e-2)
    assert nb.mean() > 8.0                                   # raw N(0, 1) rows: norm near sqrt(128)
    # the normalised draw is the raw draw divided by its norm (before the bf16 rounding)
    ratio = b["k"].float() / nb[..., None]
    assert torch.allclose(ratio, a["k"].float(), atol=1e-2)


def test_benchmark_workload_bytes():
    d = W.make("b8_t4096_h16")
    nbytes, flops = bench.algorithmic("b8_t4096_h16", d)
    assert nbytes == 1282 * 8 * 4096 * 16 + 8 * 16 * 128 * 128 * 4 == 680525824
    assert flops == 8 * 16 * math.ceil(4096 / 16) * bench.FLOPS_PER_CHUNK_HEAD


def test_varlen_lengths_are_ragged_and_seeded():
    d1, d2 = W.make("varlen_n16_h32", H=1), W.make("varlen_n16_h32", H=1)
    cu = d1["cu_seqlens"]
    assert torch.equal(cu, d2["cu_seqlens"]) and int(cu[0]) == 0 and cu.numel() == 17
    lens = cu[1:] - cu[:-1]
    assert bool((lens % 16 != 0).all()) and bool((lens >= 1).all()) and bool((lens <= 8192).all())
    assert d1["q"].shape[1] == int(cu[-1])
