"""GPU parity of the 32-token-chunk forward pass (KDA_FLAG_CHUNK32, the chunk-size ablation of
"How FlashKDA's CHUNK Size of 16 Improves Numerical Stability Over CHUNK 64" -- "Why CHUNK Size
Determines Numerical Stability") against the fp64 oracle, with the tolerance of every other
parity test (relative L2 <= 5e-3, |err| <= 2e-2 + 2e-2 |ref|). The oracle has no chunks, so the
same expected values hold for CHUNK = 16 and 32."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

# H = 3 splits each state's V rows over CTAs (NS = 1, 2 or 4 scan warps); H = 80 fills the
# machine with whole-state CTAs (eight scan warps).
HEADS = [pytest.param(3, id="split"), pytest.param(80, id="whole")]


def _check(d, final_dtype="fp32", heads=None, **kw):
    o, s = run_gpu(d, final_dtype=final_dtype, chunk=32, **kw)
    o_ref, s_ref = run_oracle(d, heads=heads, lower_bound=kw.get("lower_bound"), scale=kw.get("scale"))
    if heads is not None:
        o, s = o[:, :, heads], (None if s is None else s[:, heads])
    rel = assert_close("out", o, o_ref)
    if s is not None:
        assert_close("final_state", s, s_ref)
    return rel


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("T", [1, 16, 17, 31, 32, 33, 45, 100])
def test_chunk32_ragged_lengths(T, H):
    _check(W.make("b2_t128_h8", T=T, H=H, B=1), heads=None if H < 8 else [0, 41, 79])


@pytest.mark.parametrize("H", HEADS)
@pytest.mark.parametrize("lb", [0.0, -0.5, -5.0])
def test_chunk32_lower_bound_range(lb, H):
    """lower_bound -5 puts the exponent factors at their widest span (2^{+-115} around the
    mid-chunk reference); 0 keeps every gate at 1."""
    _check(W.make("b2_t128_h8", B=1, H=H, T=133), lower_bound=lb, heads=None if H < 8 else [1, 50])


@pytest.mark.parametrize("H", HEADS)
def test_chunk32_saturated_gates_and_betas(H):
    d = W.make("b2_t128_h8", B=1, H=H, T=70)
    gen = torch.Generator().manual_seed(7)
    sat = lambda t: torch.where(torch.rand(t.shape, generator=gen) < 0.5, t.float() * 30.0, t.float()).to(torch.bfloat16)
    d["g"] = sat(d["g"])
    d["beta"] = sat(d["beta"])
    _check(d, heads=None if H < 8 else [0, 41, 79])


@pytest.mark.parametrize("H", HEADS)
def test_chunk32_varlen_with_empty_and_ragged_sequences(H):
    d = W.make("varlen_n16_h32", lengths=[5, 37, 16, 1, 0, 23, 64, 40, 33], H=H)
    _check(d, final_dtype="bf16", heads=None if H < 8 else [0, 33, 79])


@pytest.mark.parametrize("H", HEADS)
def test_chunk32_no_gate_parameters_bf16_states(H):
    d = W.make("b8_t4096_h16", B=1, T=200, H=H)
    d["initial_state"] = (torch.randn(1, H, 128, 128, generator=torch.Generator().manual_seed(9)) * 0.02).to(torch.bfloat16)
    _check(d, final_dtype="bf16", heads=None if H < 8 else [2, 77])


@pytest.mark.parametrize("vs", [1, 2, 4, 8])
def test_chunk32_forced_v_split(vs, monkeypatch):
    monkeypatch.setenv("KDA_V_SPLIT", str(vs))
    _check(W.make("b2_t128_h8", T=77))


@pytest.mark.parametrize("H", HEADS)
def test_chunk32_deterministic_and_close_to_chunk16(H):
    d = W.make("b2_t128_h8", T=99, H=H, B=1)
    a = run_gpu(d, chunk=32)
    b = run_gpu(d, chunk=32)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = run_gpu(d, chunk=16)
    assert_close("out (32 vs 16)", a[0], c[0], rel_l2=1e-2)


def test_chunk32_struct_entry_point():
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", T=50)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    outs = []
    for entry in (kda.fwd, kda.fwd_packed):
        out = torch.empty_like(c["v"])
        fin = torch.empty_like(c["initial_state"])
        entry(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
              d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"], chunk=32)
        outs.append((out, fin))
    kda.check_device_status()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def _full(name, final_dtype, heads):
    import gated_linear_attention_kda_gb300 as kda
    d = W.make(name)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    H = d["q"].shape[2]
    nseq = d["q"].shape[0] if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    out = torch.full_like(c["v"], float("nan"))
    fin = torch.full((nseq, H, 128, 128), float("nan"), device="cuda",
                     dtype=torch.float32 if final_dtype == "fp32" else torch.bfloat16)
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"], chunk=32)
    kda.check_device_status()
    o_ref, s_ref = run_oracle(d, heads=heads)
    assert_close("out", out[:, :, heads].float().cpu().double().numpy(), o_ref)
    assert_close("final_state", fin[:, heads].float().cpu().double().numpy(), s_ref)


def test_chunk32_full_b8_t4096_h16():
    """The benchmark workload (V rows whole: eight scan warps per CTA), four heads of every sequence."""
    _full("b8_t4096_h16", "fp32", [0, 5, 10, 15])


def test_chunk32_full_long_context():
    """B=1, T=131072, H=32 (V rows split four ways), four heads."""
    _full("b1_t131072_h32", "fp32", [0, 9, 22, 31])
