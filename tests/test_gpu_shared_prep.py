"""kda_fwd_ws: the split-state kernel whose CTAs share each chunk's preparation through a
workspace. Its prepared operands are the same bytes the warp-MMA kernel's prep lanes make, so at
every split (2, 4, 8) its output and final state equal kda_fwd's at the same split bit for bit;
one case is also checked against the fp64 oracle. Lengths cover a single token, fewer chunks than
CTAs in the cluster, ragged tails, many passes over the 16-entry workspace ring, and varlen with
empty sequences."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu

SPLITS = (2, 4, 8)
SHAPES = {
    "t1": dict(B=1, T=1, H=2),
    "t20": dict(B=2, T=20, H=3),           # two chunks: some CTAs prepare none
    "t663": dict(B=2, T=16 * 41 + 7, H=3),  # ragged tail
    "t2050": dict(B=1, T=2050, H=1),        # 129 chunks: 8 passes over the 16-entry workspace ring
    "varlen": dict(lengths=[0, 5, 16, 300, 33, 1000, 0, 17], H=2),
}


def _inputs(shape, seed):
    kw = dict(SHAPES[shape])
    if "lengths" in kw:
        return W.make("varlen_n16_h32", lengths=kw["lengths"], H=kw["H"], seed=seed)
    return W.make("b2_t128_h8", B=kw["B"], T=kw["T"], H=kw["H"], seed=seed)


def _run(d, ws_mode, state="fp32", in_place=False):
    import gated_linear_attention_kda_gb300 as kda
    c = to_dev(d)
    nseq = (c["cu_seqlens"].numel() - 1) if c["cu_seqlens"] is not None else c["q"].shape[0]
    H = c["q"].shape[2]
    out = torch.full_like(c["v"], float("nan"))
    dt = {"fp32": torch.float32, "bf16": torch.bfloat16}[state]
    init = None if c["initial_state"] is None else c["initial_state"].to(dt)
    fin = init.clone() if in_place else torch.full((nseq, H, 128, 128), float("nan"), dtype=dt, device="cuda")
    if in_place:
        init = fin
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], init, fin, c["cu_seqlens"])
    if ws_mode is None:
        kda.fwd(*args)
    else:
        nb = kda.workspace_bytes(nseq, H)
        # garbage contents: the workspace needs no initialisation
        ws = torch.full((max(nb, 16) + 16 * (ws_mode == "again"),), 0xA5, dtype=torch.uint8, device="cuda")
        kda.fwd_ws(*args, workspace=ws)
        if ws_mode == "again":  # a second call reusing the same workspace
            if in_place:
                return None
            out2 = torch.full_like(out, float("nan"))
            fin2 = torch.full_like(fin, float("nan"))
            kda.fwd_ws(*args[:6], out2, *args[7:11], fin2, args[12], workspace=ws)
            kda.check_device_status()
            assert torch.equal(out, out2) and torch.equal(fin, fin2), "second call with the same workspace differs"
    kda.check_device_status()
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("split", SPLITS)
def test_shared_prep_bitwise(shape, split, monkeypatch):
    monkeypatch.setenv("KDA_V_SPLIT", str(split))
    d = _inputs(shape, seed=50 + split)
    ref_o, ref_s = _run(d, None)
    got_o, got_s = _run(d, "again")
    assert torch.equal(got_o, ref_o), f"out differs in {int((got_o != ref_o).sum())} elements"
    assert torch.equal(got_s, ref_s), f"final state differs in {int((got_s != ref_s).sum())} elements"


@pytest.mark.parametrize("split", SPLITS)
def test_shared_prep_bf16_state_in_place(split, monkeypatch):
    monkeypatch.setenv("KDA_V_SPLIT", str(split))
    d = _inputs("varlen", seed=7)
    ref_o, ref_s = _run(d, None, state="bf16", in_place=True)
    got_o, got_s = _run(d, "once", state="bf16", in_place=True)
    assert torch.equal(got_o, ref_o) and torch.equal(got_s, ref_s)


def test_shared_prep_no_gate_parameters(monkeypatch):
    monkeypatch.setenv("KDA_V_SPLIT", "4")
    d = _inputs("t663", seed=3)
    d["A_log"], d["dt_bias"], d["lower_bound"] = None, None, -1.25
    ref_o, ref_s = _run(d, None)
    got_o, got_s = _run(d, "once")
    assert torch.equal(got_o, ref_o) and torch.equal(got_s, ref_s)


def test_shared_prep_oracle_parity(monkeypatch):
    monkeypatch.setenv("KDA_V_SPLIT", "4")
    d = _inputs("t663", seed=11)
    o, s = _run(d, "once")
    ref_o, ref_s = run_oracle(d)
    assert_close("out", o.float().double().numpy(), ref_o)
    assert_close("final_state", s.double().numpy(), ref_s)


def test_workspace_bytes(monkeypatch):
    import gated_linear_attention_kda_gb300 as kda
    per_state = 16 * 15104
    monkeypatch.setenv("KDA_V_SPLIT", "4")
    assert kda.workspace_bytes(3, 5) == 15 * per_state
    assert kda.workspace_bytes(3, 5, qk_l2norm=True) == 0
    assert kda.workspace_bytes(3, 5, chunk=32) == 0
    monkeypatch.setenv("KDA_V_SPLIT", "1")
    assert kda.workspace_bytes(3, 5) == 0
    monkeypatch.delenv("KDA_V_SPLIT")
    # the planned split
    vs32, _ = kda.plan(32, torch.cuda.get_device_properties(0).multi_processor_count)
    assert kda.workspace_bytes(1, 32) == (32 * per_state if vs32 > 1 else 0)


def test_workspace_errors(monkeypatch):
    import gated_linear_attention_kda_gb300 as kda
    monkeypatch.setenv("KDA_V_SPLIT", "2")
    d = to_dev(_inputs("t663", seed=5))
    nb = kda.workspace_bytes(2, 3)
    out = torch.empty_like(d["v"])
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"], d["lower_bound"])
    small = torch.empty(nb - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="KDA_ERR_RANGE"):
        kda.fwd_ws(*args, workspace=small)
    big = torch.empty(nb + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError, match="KDA_ERR_ALIGN"):
        kda.fwd_ws(*args, workspace=big[1:])
    kda.check_device_status()


@pytest.mark.parametrize("qkn", [False, True])
def test_workspace_ignored_off_the_shared_path(qkn, monkeypatch):
    """With an option bit, or without a split, the call is kda_fwd_ex's and leaves the workspace alone."""
    import gated_linear_attention_kda_gb300 as kda
    monkeypatch.setenv("KDA_V_SPLIT", "4" if qkn else "1")
    d = to_dev(W.make("b2_t128_h8", B=1, T=100, H=2, seed=9, raw_qk=qkn))
    outs = []
    ws = torch.full((16 * 15104 * 2,), 0x5A, dtype=torch.uint8, device="cuda")
    for use in (False, True):
        out = torch.empty_like(d["v"])
        args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], out, d["A_log"], d["dt_bias"], d["lower_bound"])
        if use:
            kda.fwd_ws(*args, qk_l2norm=qkn, workspace=ws)
        else:
            kda.fwd(*args, qk_l2norm=qkn)
        outs.append(out)
    kda.check_device_status()
    assert torch.equal(outs[0], outs[1])
    assert bool((ws == 0x5A).all())
