"""GPU parity: the CUDA path against the fp64 oracle on the same seeded
inputs, element by element, with the stated tolerance (relative L2 <= 5e-3,
|err| <= 2e-2 + 2e-2 |ref|) on ``out`` and ``final_state``."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _check(d, final_dtype="fp32", heads=None, **kw):
    o, s = run_gpu(d, final_dtype=final_dtype, **kw)
    o_ref, s_ref = run_oracle(d, heads=heads, lower_bound=kw.get("lower_bound"), scale=kw.get("scale"),
                              qk_l2norm=kw.get("qk_l2norm", False))
    if heads is not None:
        o, s = o[:, :, heads], (None if s is None else s[:, heads])
    rel = assert_close("out", o, o_ref)
    if s is not None:
        assert_close("final_state", s, s_ref)
    return rel


def test_small_one_head_four_chunks():
    _check(W.make("b1_t64_h1"))


def test_state_carry_case_fp32_states():
    _check(W.make("b2_t128_h8"))


def test_split_call_equals_one_call():
    """T = 128 as 64 + 64 through final_state -> initial_state."""
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8")
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    half = lambda x, a, b: x[:, a:b].contiguous()
    out1 = torch.empty_like(half(c["v"], 0, 64))
    out2 = torch.empty_like(out1)
    mid = torch.empty_like(c["initial_state"])
    fin = torch.empty_like(c["initial_state"])
    args = lambda a, b: [half(c[x], a, b) for x in ("q", "k", "v", "g", "beta")]
    kda.fwd(*args(0, 64), d["scale"], out1, c["A_log"], c["dt_bias"], d["lower_bound"], c["initial_state"], mid)
    kda.fwd(*args(64, 128), d["scale"], out2, c["A_log"], c["dt_bias"], d["lower_bound"], mid, fin)
    kda.check_device_status()
    o_ref, s_ref = run_oracle(d)
    assert_close("out", torch.cat([out1, out2], 1).float().cpu().double().numpy(), o_ref)
    assert_close("final_state", fin.cpu().double().numpy(), s_ref)


# H = 3 / 4 runs the split-V-row warp-MMA kernel; H = 80 fills the machine
# with whole-state CTAs and runs the tensor-memory (tcgen05) kernel.
KERNEL_HEADS = [pytest.param(3, id="mma"), pytest.param(80, id="tcgen05")]


def test_head_counts_select_both_kernels():
    import gated_linear_attention_kda_gb300 as kda
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    assert kda.plan(3, nsm)[0] > 1 and kda.plan(80, nsm)[0] == 1


@pytest.mark.parametrize("H", KERNEL_HEADS)
@pytest.mark.parametrize("T", [1, 15, 16, 17, 37, 100])
def test_ragged_lengths(T, H):
    _check(W.make("b2_t128_h8", T=T, H=H, B=1), heads=None if H < 8 else [0, 41, 79])


@pytest.mark.parametrize("H", KERNEL_HEADS)
@pytest.mark.parametrize("lb", [0.0, -0.5, -5.0])
def test_lower_bound_range(lb, H):
    _check(W.make("b2_t128_h8", B=1, H=H, T=70), lower_bound=lb, heads=None if H < 8 else [1, 50])



@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_saturated_gates_and_betas_and_larger_values(H):
    """Gate and beta logits pushed into saturation (|logit| up to 30: decay exp(lower_bound) or none,
    beta 0 or 1, where the tanh form of the sigmoid is at its limits) and values 20 times larger."""
    d = W.make("b2_t128_h8", B=1, H=H, T=70)
    gen = torch.Generator().manual_seed(7)
    sat = lambda t: torch.where(torch.rand(t.shape, generator=gen) < 0.5, t.float() * 30.0, t.float()).to(torch.bfloat16)
    d["g"] = sat(d["g"])
    d["beta"] = sat(d["beta"])
    d["v"] = (d["v"].float() * 20.0).to(torch.bfloat16)
    _check(d, heads=None if H < 8 else [0, 41, 79])

@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_no_gate_parameters_bf16_states(H):
    d = W.make("b8_t4096_h16", B=1, T=200, H=H)
    d["initial_state"] = (torch.randn(1, H, 128, 128, generator=torch.Generator().manual_seed(9)) * 0.02).to(torch.bfloat16)
    _check(d, final_dtype="bf16", heads=None if H < 8 else [2, 77])


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_in_place_state_equals_out_of_place(H):
    d = W.make("b2_t128_h8", T=77, H=H, B=1)
    o1, s1 = run_gpu(d)
    o2, s2 = run_gpu(d, in_place=True)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_deterministic_repeats(H):
    d = W.make("b2_t128_h8", T=99, H=H, B=1)
    a = run_gpu(d)
    b = run_gpu(d)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("case", ["lb0", "varlen"])
def test_ten_repeats_bitwise_identical_and_within_tolerance(case):
    """The whole-state (tcgen05) kernel ten times on the same inputs: every repeat bitwise equal to
    the first and within tolerance of the oracle. lower_bound 0 keeps every cross-chunk correction
    term at full weight; the varlen case mixes ragged sequences in one launch."""
    if case == "lb0":
        d = W.make("b2_t128_h8", B=1, T=133, H=80)
        kw = {"lower_bound": 0.0}
        fdt = "fp32"
    else:
        d = W.make("varlen_n16_h32", lengths=[5, 37, 16, 1, 0, 23, 64, 40, 200, 17], H=12)
        kw = {}
        fdt = "bf16"
    first = run_gpu(d, final_dtype=fdt, **kw)
    for _ in range(9):
        again = run_gpu(d, final_dtype=fdt, **kw)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    heads = [0, 41, 79] if case == "lb0" else None
    o_ref, s_ref = run_oracle(d, heads=heads, lower_bound=kw.get("lower_bound"))
    o, s = first
    if heads is not None:
        o, s = o[:, :, heads], s[:, heads]
    assert_close("out", o, o_ref)
    assert_close("final_state", s, s_ref)


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_no_final_state_and_zero_scale(H):
    d = W.make("b1_t64_h1", H=H)
    o, s = run_gpu(d, final_dtype=None, scale=0.0)
    assert s is None and np.all(o == 0)


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_varlen_small_with_empty_and_ragged_sequences(H):
    d = W.make("varlen_n16_h32", lengths=[5, 37, 16, 1, 0, 23, 64, 40], H=H)
    _check(d, final_dtype="bf16", heads=None if H < 8 else [0, 33, 79])


@pytest.mark.parametrize("N", [64, 65])
def test_varlen_many_sequences_both_orders(N):
    """64 sequences take the longest-first CTA order of the whole-state kernel, 65 the plain order
    (lengths 0..40, so empty, single-chunk and ragged sequences all occur); H = 3 gives 192 / 195
    states, more than the SMs, so every state is one CTA."""
    gen = torch.Generator().manual_seed(11 + N)
    lens = torch.randint(0, 41, (N,), generator=gen).tolist()
    d = W.make("varlen_n16_h32", lengths=lens, H=3)
    _check(d, final_dtype="bf16")


@pytest.mark.parametrize("H", [2, 80])
def test_varlen_equals_separate_calls(H):
    lens = [19, 48, 3, 33]
    d = W.make("varlen_n16_h32", lengths=lens, H=H)
    o, s = run_gpu(d, final_dtype="bf16")
    cu = d["cu_seqlens"]
    for i in range(len(lens)):
        a, b = int(cu[i]), int(cu[i + 1])
        di = dict(d)
        for k in ("q", "k", "v", "g", "beta"):
            di[k] = d[k][:, a:b].contiguous()
        di["initial_state"] = d["initial_state"][i:i + 1].contiguous()
        di["cu_seqlens"] = None
        oi, si = run_gpu(di, final_dtype="bf16")
        assert np.array_equal(oi, o[:, a:b]) and np.array_equal(si[0], s[i])


def test_bad_cu_seqlens_flags_device_error_without_fault():
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("varlen_n16_h32", lengths=[50, 10, 40], H=2)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    c["cu_seqlens"] = torch.tensor([0, 50, 30, 100], dtype=torch.int64, device="cuda")  # decreasing bound
    out = torch.zeros_like(c["v"])
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], None, c["cu_seqlens"])
    with pytest.raises(kda.KDAError, match="KDA_ERR_DEVICE"):
        kda.check_device_status()
    kda.check_device_status()  # the word is cleared after it was reported
    torch.cuda.synchronize()   # the context is still healthy


@pytest.mark.parametrize("states", ["none", "initial_only", "final_only", "both", "in_place"])
def test_empty_call_passes_the_state_through(states):
    """T = 0: no forward kernel runs; final_state receives initial_state, or zeros without one."""
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", T=0)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    init = c["initial_state"] if states in ("initial_only", "both", "in_place") else None
    fin = None
    if states in ("final_only", "both"):
        fin = torch.full_like(c["initial_state"], float("nan"))
    elif states == "in_place":
        fin = init
    before = None if init is None else init.clone()
    out = torch.empty_like(c["v"])
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], init, fin)
    kda.check_device_status()
    if fin is not None:
        assert torch.equal(fin, before if before is not None else torch.zeros_like(fin))
    if init is not None:
        assert torch.equal(init, before)


def test_empty_varlen_call_and_its_cu_seqlens_check():
    """Varlen with every sequence empty: the bf16 final states equal the initial ones; a nonzero
    cu_seqlens entry in an empty call is flagged on the device, without a fault."""
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("varlen_n16_h32", lengths=[0, 0, 0], H=2)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    fin = torch.full_like(c["initial_state"], float("nan"))
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])
    kda.check_device_status()
    assert torch.equal(fin, c["initial_state"])
    bad = torch.tensor([0, 5, 5, 5], dtype=torch.int64, device="cuda")
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin, bad)
    with pytest.raises(kda.KDAError, match="KDA_ERR_DEVICE"):
        kda.check_device_status(bad)
    kda.check_device_status(bad.device)  # reported once, then cleared
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", ["b2", "b8_four_pieces", "varlen_pieces", "empty"])
def test_host_entry_point_matches_device_entry_point(case):
    """kda_fwd_host (pinned host buffers, the call cut into pieces on their own streams) gives
    kda_fwd's results bit for bit: the pieces run the V-row split of the whole call."""
    import gated_linear_attention_kda_gb300 as kda
    fdt = "fp32"
    if case == "b2":
        d = W.make("b2_t128_h8", T=45)
    elif case == "b8_four_pieces":
        d = W.make("b2_t128_h8", B=8, T=70, H=12)
    elif case == "varlen_pieces":
        d = W.make("varlen_n16_h32", lengths=[5, 37, 16, 1, 0, 23, 64, 40, 200, 17], H=12)
        fdt = "bf16"
    else:
        d = W.make("b2_t128_h8", B=3, T=0)
    o_dev, s_dev = run_gpu(d, final_dtype=fdt)
    out = torch.full_like(d["v"], float("nan")).pin_memory()
    fin = torch.full_like(d["initial_state"], float("nan")).pin_memory()
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    kda.fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], d["scale"], out, pin["A_log"],
                 pin["dt_bias"], d["lower_bound"], pin["initial_state"], fin, pin["cu_seqlens"])
    assert np.array_equal(out.float().double().numpy(), o_dev)
    assert np.array_equal(fin.float().double().numpy(), s_dev)


@pytest.mark.parametrize("entry", ["fwd_flat", "fwd_packed"])
def test_flat_and_struct_entry_points_match_kda_fwd(entry):
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", T=45)
    o_dev, s_dev = run_gpu(d)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.full_like(c["v"], float("nan"))
    fin = torch.full_like(c["initial_state"], float("nan"))
    getattr(kda, entry)(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
                        d["lower_bound"], c["initial_state"], fin)
    kda.check_device_status()
    assert np.array_equal(out.float().cpu().double().numpy(), o_dev)
    assert np.array_equal(fin.cpu().double().numpy(), s_dev)



@pytest.mark.parametrize("vs", [1, 2, 4, 8])
def test_forced_v_split_matches_oracle(vs, monkeypatch):
    """Every split of the V rows (1: the tcgen05 kernel; 2, 4, 8: the warp-MMA kernel) on the same
    ragged inputs, against the oracle."""
    monkeypatch.setenv("KDA_V_SPLIT", str(vs))
    _check(W.make("b2_t128_h8", T=45))


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_no_writes_outside_out_and_final_state(H):
    """Canaries on both sides of out and final_state survive the call (varlen, ragged lengths)."""
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("varlen_n16_h32", lengths=[5, 16, 33], H=H)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    pad = 64

    def padded(like):
        n = like.numel()
        big = torch.empty(n + 2 * pad, dtype=like.dtype, device="cuda")
        big.view(torch.int16 if like.element_size() == 2 else torch.int32).fill_(0x5A5A)
        return big, big[pad:pad + n].view(like.shape)

    obig, out = padded(c["v"])
    fbig, fin = padded(c["initial_state"])
    before_o, before_f = obig.clone(), fbig.clone()
    kda.fwd(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])
    kda.check_device_status()
    for big, ref in ((obig, before_o), (fbig, before_f)):
        assert torch.equal(big[:pad], ref[:pad]) and torch.equal(big[-pad:], ref[-pad:])


# ------------------------------------------------------------ full-size workloads

def _check_every_head(name, final_dtype, group, workspace=False):
    """A full-size workload in the launch configuration the benchmark times, compared with the
    oracle on EVERY token of EVERY head. The oracle runs in head groups (heads are independent)
    to bound host memory; the relative L2 error is accumulated over the whole tensor and the
    elementwise bound is checked in every group. ``workspace`` runs the call through kda_fwd_ws
    (the planned split with the preparation shared by each state's cluster)."""
    import gated_linear_attention_kda_gb300 as kda
    from tests.kda_harness import ABS, REL, REL_L2
    d = W.make(name)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    H = d["q"].shape[2]
    nseq = d["q"].shape[0] if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    out = torch.full_like(c["v"], float("nan"))
    fin = torch.full((nseq, H, 128, 128), float("nan"), device="cuda",
                     dtype=torch.float32 if final_dtype == "fp32" else torch.bfloat16)
    args = (c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
            d["lower_bound"], c["initial_state"], fin, c["cu_seqlens"])
    if workspace:
        nbytes = kda.workspace_bytes(nseq, H)
        assert nbytes > 0, "the planned split must share the preparation here"
        kda.fwd_ws(*args, workspace=torch.empty(nbytes, dtype=torch.uint8, device="cuda"))
    else:
        kda.fwd(*args)
    kda.check_device_status()
    out_h, fin_h = out.cpu(), fin.cpu()
    del c, out, fin
    acc = {"out": [0.0, 0.0], "final_state": [0.0, 0.0]}
    for h0 in range(0, H, group):
        heads = list(range(h0, min(H, h0 + group)))
        o_ref, s_ref = run_oracle(d, heads=heads)
        for key, got_t, ref in (("out", out_h[:, :, heads], o_ref), ("final_state", fin_h[:, heads], s_ref)):
            got = got_t.float().double().numpy()
            assert got.shape == ref.shape and np.isfinite(got).all(), key
            err = got - ref
            acc[key][0] += float(np.sum(err * err))
            acc[key][1] += float(np.sum(ref * ref))
            bad = np.abs(err) > ABS + REL * np.abs(ref)
            assert not bad.any(), f"{key} heads {heads[0]}..{heads[-1]}: {int(bad.sum())} elements out of bound"
    for key, (e2, r2) in acc.items():
        rel = math.sqrt(e2 / r2)
        assert rel <= REL_L2, f"{key}: relative L2 error {rel:.3e} over all heads"


def test_full_b8_t4096_h16_every_head():
    """B=8, T=4096, H=16, fp32 final state: all 16 heads of all 8 sequences."""
    _check_every_head("b8_t4096_h16", "fp32", group=16)


def test_full_varlen_n16_h32_every_head():
    """16 packed sequences (66 217 tokens), H=32, bf16 initial and final states: all heads."""
    _check_every_head("varlen_n16_h32", "bf16", group=8)


def test_full_long_context_every_head():
    """B=1, T=131072, H=32, fp32 initial and final states: all 32 heads."""
    _check_every_head("b1_t131072_h32", "fp32", group=16)


def test_full_long_context_every_head_shared_preparation():
    """The same through kda_fwd_ws (split 4, each state's cluster sharing the preparation)."""
    _check_every_head("b1_t131072_h32", "fp32", group=16, workspace=True)


# ------------------------------------------------------------ per-step parity (one chunk)

@pytest.mark.parametrize("name,b,h,chunk,rows", [
    ("b1_t64_h1", 0, 0, 0, 16), ("b1_t64_h1", 0, 0, 1, 16), ("b1_t64_h1", 0, 0, 3, 16), ("b1_t64_h1", 0, 0, 2, 5),
    ("b2_t128_h8", 0, 0, 0, 16), ("b2_t128_h8", 1, 5, 7, 16), ("b2_t128_h8", 0, 3, 4, 11),
])
def test_chunk_steps_match_the_fp64_chunk_terms(name, b, h, chunk, rows):
    """Gate cumsum (log2), beta, A, P and T = (I + A)^-1 of one chunk, through the kernels' own
    per-chunk device code (kda_probe_chunk), against oracle.chunk_ref.chunk_terms in fp64.
    G2 and beta may differ by the tanh.approx sigmoid: |d sigma| <= 2.5e-4 per token, so
    |d G2_r| <= (r + 1) |lower_bound| log2(e) 2.5e-4; A, P, T use the parity tolerance."""
    import oracle
    import oracle.chunk_ref as chunk_ref
    import gated_linear_attention_kda_gb300 as kda
    d = W.make(name)
    sl = slice(16 * chunk, 16 * chunk + 16)
    tiles = {x: d[x][b, sl, h].contiguous() for x in ("q", "k", "g")}
    bt = d["beta"][b, sl, h].contiguous()
    A_log = None if d["A_log"] is None else d["A_log"][h:h + 1].contiguous()
    dt = None if d["dt_bias"] is None else d["dt_bias"][h].contiguous()
    lb = d["lower_bound"]
    o = kda.probe_chunk(tiles["q"].cuda(), tiles["k"].cuda(), tiles["g"].cuda(), bt.cuda(),
                        None if A_log is None else A_log.cuda(), None if dt is None else dt.cuda(), lb, rows)
    torch.cuda.synchronize()
    f64 = lambda t: oracle.bf16_bits_to_f64(W.bf16_bits(t))
    L = rows
    G2, beta, A, P, T = chunk_ref.chunk_terms(f64(tiles["q"])[:L], f64(tiles["k"])[:L], f64(tiles["g"])[:L],
                                              f64(bt)[:L], None if A_log is None else float(A_log[0]),
                                              None if dt is None else dt.double().numpy(), lb)
    got = {n: t.cpu().double().numpy() for n, t in o.items()}
    bound = (np.arange(L)[:, None] + 1) * abs(lb) * math.log2(math.e) * 2.5e-4 + 1e-5
    assert np.all(np.abs(got["G2"][:L] - G2) <= bound)
    assert np.all(np.abs(got["beta"][:L] - beta) <= 2.5e-4 + 1e-6)
    assert np.all(got["beta"][L:] == 0.0)
    for n, ref in (("A", A), ("P", P), ("T", T)):
        assert_close(n, got[n][:L, :L], ref)



# ------------------------------------------------------------ q/k L2 normalisation in the kernel

@pytest.mark.parametrize("H", KERNEL_HEADS)
@pytest.mark.parametrize("T", [37, 128])
def test_qk_l2norm_in_kernel_matches_oracle(T, H):
    """Raw N(0, 1) q and k (norms near sqrt(128)), normalised inside the kernel
    (KDA_FLAG_QK_L2NORM), against the oracle with the same normalisation; both kernels."""
    d = W.make("b2_t128_h8", B=1, T=T, H=H, raw_qk=True)
    _check(d, heads=None if H < 8 else [0, 41, 79], qk_l2norm=True)


@pytest.mark.parametrize("H", KERNEL_HEADS)
def test_qk_l2norm_varlen_ragged_and_empty(H):
    d = W.make("varlen_n16_h32", lengths=[0, 19, 64, 1, 33], H=H, raw_qk=True)
    _check(d, final_dtype="bf16", heads=None if H < 8 else [3, 77], qk_l2norm=True)


def test_qk_l2norm_flag_through_struct_entry():
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", B=1, T=45, H=80, raw_qk=True)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    outs = []
    for fn in (kda.fwd, kda.fwd_packed):
        out = torch.full_like(c["v"], float("nan"))
        fin = torch.full_like(c["initial_state"], float("nan"))
        fn(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, c["A_log"], c["dt_bias"],
           d["lower_bound"], c["initial_state"], fin, qk_l2norm=True)
        outs.append((out, fin))
    kda.check_device_status()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_unknown_option_bits_are_rejected():
    import ctypes
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b1_t64_h1")
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = kda.library().kda_fwd_ex(P(c["q"]), P(c["k"]), P(c["v"]), P(c["g"]), P(c["beta"]), d["scale"], P(out),
                                  P(c["A_log"]), P(c["dt_bias"]), d["lower_bound"], None, 0, None, 0, None, 0,
                                  1, 64, 1, 128, 128, 6, None)
    assert st == 4  # KDA_ERR_RANGE


# ------------------------------------------------------------ single-token steps (decode)

@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate_params", [True, False])
def test_decode_step_matches_oracle(state_dtype, gate_params):
    """One token per (sequence, head) with the state updated in place, against the oracle's
    one-token call from the same initial state."""
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", B=3, T=1, H=5)
    d["initial_state"] = d["initial_state"].to(state_dtype)
    if not gate_params:
        d["A_log"], d["dt_bias"] = None, None
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.full_like(c["v"], float("nan"))
    state = c["initial_state"].clone()
    kda.decode(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, state, c["A_log"], c["dt_bias"],
               d["lower_bound"])
    kda.check_device_status()
    o_ref, s_ref = run_oracle(d)
    assert_close("out", out.float().cpu().double().numpy(), o_ref)
    assert_close("state", state.float().cpu().double().numpy(), s_ref)


def test_decode_step_qk_l2norm_matches_oracle():
    import gated_linear_attention_kda_gb300 as kda
    d = W.make("b2_t128_h8", B=3, T=1, H=5, raw_qk=True)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.full_like(c["v"], float("nan"))
    state = c["initial_state"].clone()
    kda.decode(c["q"], c["k"], c["v"], c["g"], c["beta"], d["scale"], out, state, c["A_log"], c["dt_bias"],
               d["lower_bound"], qk_l2norm=True)
    kda.check_device_status()
    o_ref, s_ref = run_oracle(d, qk_l2norm=True)
    assert_close("out", out.float().cpu().double().numpy(), o_ref)
    assert_close("state", state.float().cpu().double().numpy(), s_ref)


def test_decode_steps_continue_the_chunked_pass():
    """kda_fwd over the first 37 tokens, then ten single-token steps on its final state: the
    step outputs and the final state match the oracle over all 47 tokens."""
    import gated_linear_attention_kda_gb300 as kda
    T0, n = 37, 10
    d = W.make("b2_t128_h8", T=T0 + n)
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    out = torch.empty_like(c["v"])
    state = torch.empty_like(c["initial_state"])
    head = {x: c[x][:, :T0].contiguous() for x in ("q", "k", "v", "g", "beta")}
    out0 = torch.empty_like(head["v"])
    kda.fwd(head["q"], head["k"], head["v"], head["g"], head["beta"], d["scale"], out0,
            c["A_log"], c["dt_bias"], d["lower_bound"], c["initial_state"], state)
    out[:, :T0] = out0
    for t in range(T0, T0 + n):
        o_t = torch.empty_like(c["v"][:, t].contiguous())
        kda.decode(c["q"][:, t].contiguous(), c["k"][:, t].contiguous(), c["v"][:, t].contiguous(),
                   c["g"][:, t].contiguous(), c["beta"][:, t].contiguous(), d["scale"], o_t, state,
                   c["A_log"], c["dt_bias"], d["lower_bound"])
        out[:, t] = o_t
    kda.check_device_status()
    o_ref, s_ref = run_oracle(d)
    assert_close("out", out.float().cpu().double().numpy(), o_ref)
    assert_close("state", state.cpu().double().numpy(), s_ref)
