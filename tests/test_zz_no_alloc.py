"""kda_fwd_static, the entry point that allocates nothing: the shared chunk preparation of
kda_fwd_ws on the library's own file-scope scratch. Collected last, and also run alone: it must
pass either way. Two calls in a row each equal kda_fwd's result bit for bit (the scratch keeps the
previous call's contents and needs no clearing), the device's free memory does not move across
calls, and a request larger than the scratch is refused with a message naming the limit."""
import pytest
import torch

import workloads as W
from tests.kda_harness import to_dev

pytestmark = pytest.mark.gpu


def _call(kda, fn, c, d, out, fin):
    fn(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"], d["lower_bound"],
       c["initial_state"], fin, c["cu_seqlens"])


def _pair(kda, d, nseq):
    c = to_dev(d)
    H = c["q"].shape[2]
    sdt = torch.float32 if c["initial_state"] is None else c["initial_state"].dtype
    bufs = [(torch.full_like(c["v"], float("nan")),
             torch.full((nseq, H, 128, 128), float("nan"), dtype=sdt, device="cuda")) for _ in range(3)]
    _call(kda, kda.fwd, c, d, *bufs[0])
    _call(kda, kda.fwd_static, c, d, *bufs[1])
    _call(kda, kda.fwd_static, c, d, *bufs[2])  # second call in a row, same scratch
    kda.check_device_status()
    return bufs


@pytest.mark.parametrize("shape", [dict(B=1, T=1500, H=8),      # 8 states: split 8
                                   dict(B=2, T=16 * 43 + 9, H=12),  # 24 states: split 4
                                   dict(lengths=[700, 0, 33, 1200], H=4)])  # varlen, 16 states
def test_static_equals_fwd_on_two_calls_in_a_row(shape, monkeypatch):
    import gated_linear_attention_kda_gb300 as kda
    monkeypatch.delenv("KDA_V_SPLIT", raising=False)
    if "lengths" in shape:
        d = W.make("varlen_n16_h32", lengths=shape["lengths"], H=shape["H"], seed=21)
        nseq = len(shape["lengths"])
    else:
        d = W.make("b2_t128_h8", B=shape["B"], T=shape["T"], H=shape["H"], seed=22)
        nseq = shape["B"]
    assert kda.workspace_bytes(nseq, d["q"].shape[2]) > 0, "the plan must split these states"
    (o0, s0), (o1, s1), (o2, s2) = _pair(kda, d, nseq)
    for o, s in ((o1, s1), (o2, s2)):
        assert torch.equal(o, o0) and torch.equal(s, s0)


def test_static_allocates_nothing(monkeypatch):
    import gated_linear_attention_kda_gb300 as kda
    monkeypatch.setenv("KDA_V_SPLIT", "4")
    d = W.make("b2_t128_h8", B=1, T=900, H=6, seed=23)
    c = to_dev(d)
    out = torch.empty_like(c["v"])
    fin = torch.empty(1, 6, 128, 128, device="cuda")
    _call(kda, kda.fwd_static, c, d, out, fin)  # first call: per-device set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        _call(kda, kda.fwd_static, c, d, out, fin)
    torch.cuda.synchronize()
    kda.check_device_status()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_refuses_more_states_than_its_scratch(monkeypatch):
    import gated_linear_attention_kda_gb300 as kda
    H = kda.STATIC_SCRATCH_STATES + 16
    d = W.make("b2_t128_h8", B=1, T=40, H=H, seed=24)
    c = to_dev(d)
    out = torch.empty_like(c["v"])
    fin = torch.empty(1, H, 128, 128, device="cuda")
    monkeypatch.setenv("KDA_V_SPLIT", "2")  # forced split: this call would need the scratch
    with pytest.raises(ValueError, match="KDA_ERR_RANGE.*static scratch holds 80 states"):
        _call(kda, kda.fwd_static, c, d, out, fin)
    monkeypatch.setenv("KDA_V_SPLIT", "1")  # unsplit: no scratch, no limit
    ref_o, ref_s = torch.empty_like(out), torch.empty_like(fin)
    _call(kda, kda.fwd, c, d, ref_o, ref_s)
    _call(kda, kda.fwd_static, c, d, out, fin)
    kda.check_device_status()
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_s)
