"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and compare them with the stated tolerance."""
import numpy as np
import torch

import oracle
import workloads as W

REL_L2 = 5e-3          # relative L2 error on out and final_state
ABS, REL = 2e-2, 2e-2  # elementwise |err| <= ABS + REL * |ref|

_DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


def to_dev(d, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run_gpu(d, final_dtype="fp32", in_place=False, lower_bound=None, scale=None, qk_l2norm=False, chunk=16):
    import gated_linear_attention_kda_gb300 as kda
    c = to_dev(d)
    out = torch.full_like(c["v"], float("nan"))
    nseq = (c["cu_seqlens"].numel() - 1) if c["cu_seqlens"] is not None else c["q"].shape[0]
    H = c["q"].shape[2]
    fin = None
    init = c["initial_state"]
    if in_place:
        fin = init
    elif final_dtype:
        fin = torch.full((nseq, H, 128, 128), float("nan"), dtype=_DT[final_dtype], device="cuda")
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"] if scale is None else scale, out,
            c["A_log"], c["dt_bias"], d["lower_bound"] if lower_bound is None else lower_bound, init, fin,
            c["cu_seqlens"], qk_l2norm=qk_l2norm, chunk=chunk)
    kda.check_device_status()
    o = out.float().cpu().double().numpy()
    s = None if fin is None else fin.float().cpu().double().numpy()
    return o, s


def run_oracle(d, heads=None, lower_bound=None, scale=None, qk_l2norm=False):
    """fp64 oracle; ``heads`` restricts the run to those heads (heads are independent)."""
    sel = (lambda x: x) if heads is None else (lambda x: x[:, :, heads])
    bits = {k: W.bf16_bits(sel(d[k]).contiguous()) for k in ("q", "k", "v", "g")}
    bb = W.bf16_bits(d["beta"][:, :, heads].contiguous() if heads is not None else d["beta"])
    A = None if d["A_log"] is None else (d["A_log"] if heads is None else d["A_log"][heads]).numpy()
    db = None if d["dt_bias"] is None else (d["dt_bias"] if heads is None else d["dt_bias"][heads]).numpy()
    init = d["initial_state"]
    if init is not None and heads is not None:
        init = init[:, heads].contiguous()
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].numpy()
    return oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bb,
                      d["scale"] if scale is None else scale, A, db,
                      d["lower_bound"] if lower_bound is None else lower_bound, W.state_f64(init), cu,
                      qk_l2norm=qk_l2norm)


def assert_close(name, got, ref, rel_l2=REL_L2):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (den if den > 0 else 1.0)
    bad = np.abs(got - ref) > ABS + REL * np.abs(ref)
    assert rel <= rel_l2, f"{name}: relative L2 error {rel:.3e} > {rel_l2}"
    assert not bad.any(), f"{name}: {int(bad.sum())} elements outside {ABS} + {REL}|ref| (max {np.abs(got - ref).max():.3e})"
    return rel
