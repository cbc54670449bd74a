"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test fixes a property that the KDA forward pass must have by its
definition (the gated delta rule with per-channel decay, the gate of
"FlashKDA lower_bound Parameter: Controlling Exponentiation Precision in
Selective State Space Models", the state carry and varlen contract of
"FlashKDA Input Tensor Shapes and DTypes"), chosen so that a dropped term, a
wrong sign or index, or a transposed operand in the oracle fails at least one.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import oracle.chunk_ref as chunk_ref
import workloads as W

rng = np.random.default_rng(1234)


def _bits(x):
    """float array -> bf16 bit patterns (values must already be bf16-exact or are rounded)."""
    return W.bf16_bits(torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def _inputs(name, **kw):
    d = W.make(name, **kw)
    bits = {k: W.bf16_bits(d[k]) for k in ("q", "k", "v", "g", "beta")}
    A = None if d["A_log"] is None else d["A_log"].numpy()
    db = None if d["dt_bias"] is None else d["dt_bias"].numpy()
    init = W.state_f64(d["initial_state"])
    cu = None if d["cu_seqlens"] is None else d["cu_seqlens"].numpy()
    return d, bits, A, db, init, cu


def _run(bits, d, A, db, init, cu):
    return oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], d["scale"], A, db,
                      d["lower_bound"], init, cu)


# ---------------------------------------------------------------- closed forms

def test_single_token_from_zero_state():
    """T=1, S0=0: S = beta v k^T and o = scale beta (k.q) v."""
    K, V = 5, 3
    q, k = rng.standard_normal((1, 1, 1, K)), rng.standard_normal((1, 1, 1, K))
    v = rng.standard_normal((1, 1, 1, V))
    alpha = rng.uniform(0.1, 1.0, (1, 1, 1, K))
    beta = np.array([[[0.37]]])
    out, fin = oracle.core(q, k, v, alpha, beta, 0.5)
    np.testing.assert_allclose(fin[0, 0], 0.37 * np.outer(v[0, 0, 0], k[0, 0, 0]), rtol=1e-14, atol=1e-15)
    expect = 0.5 * 0.37 * np.dot(k[0, 0, 0], q[0, 0, 0]) * v[0, 0, 0]
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=1e-13, atol=1e-15)


def test_single_token_with_state_matrix_form():
    """T=1, S0 given: S = S0 Diag(alpha) (I - beta k k^T) + beta v k^T, o = scale S q."""
    K, V = 4, 6
    S0 = rng.standard_normal((1, 1, V, K))
    q, k = rng.standard_normal((1, 1, 1, K)), rng.standard_normal((1, 1, 1, K))
    v = rng.standard_normal((1, 1, 1, V))
    alpha = rng.uniform(0.1, 1.0, (1, 1, 1, K))
    b = 0.8
    out, fin = oracle.core(q, k, v, alpha, np.array([[[b]]]), 1.25, initial_state=S0)
    kk = k[0, 0, 0]
    S = S0[0, 0] @ np.diag(alpha[0, 0, 0]) @ (np.eye(K) - b * np.outer(kk, kk)) + b * np.outer(v[0, 0, 0], kk)
    np.testing.assert_allclose(fin[0, 0], S, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(out[0, 0, 0], 1.25 * S @ q[0, 0, 0], rtol=1e-13, atol=1e-14)


def test_beta_zero_is_pure_decay():
    """beta logits = -inf: S_t = S0 Diag(prod_{s<=t} alpha_s), o_t = scale S0 (q_t * prod alpha)."""
    B, T, H, K = 1, 9, 2, 128
    S0 = rng.standard_normal((1, H, K, K)) * 0.1
    g = _bits(rng.standard_normal((B, T, H, K)))
    q = _bits(rng.standard_normal((B, T, H, K)) * 0.1)
    k = _bits(rng.standard_normal((B, T, H, K)) * 0.1)
    v = _bits(rng.standard_normal((B, T, H, K)))
    beta = _bits(np.full((B, T, H), -np.inf))
    A_log = np.array([0.3, -0.2], np.float32)
    dt = (rng.standard_normal((H, K)) * 0.1).astype(np.float32)
    lb = -1.5
    out, fin = oracle.fwd(q, k, v, g, beta, 0.7, A_log, dt, lb, S0, None)
    x = np.exp(A_log.astype(np.float64))[None, None, :, None] * (_f64(g) + dt.astype(np.float64))
    alpha = np.exp(lb / (1.0 + np.exp(-x)))
    cum = np.cumprod(alpha, axis=1)
    for h in range(H):
        np.testing.assert_allclose(fin[0, h], S0[0, h] * cum[0, -1, h][None, :], rtol=1e-12, atol=1e-15)
        for t in range(T):
            exp_o = 0.7 * S0[0, h] @ (_f64(q)[0, t, h] * cum[0, t, h])
            np.testing.assert_allclose(out[0, t, h], exp_o, rtol=1e-11, atol=1e-14)


def test_delta_rule_storage_orthonormal_keys():
    """lower_bound=0 (no decay), beta=1, orthonormal keys: S_n = S0 (I - sum k k^T) + sum v k^T,
    so S_n k_j = v_j, and a query equal to the current key reads back scale * v_t."""
    K = V = 128
    n = 40
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:, :n].T                                    # n orthonormal rows
    vals = rng.standard_normal((n, V))
    S0 = rng.standard_normal((1, 1, V, K)) * 0.05
    alpha = np.ones((1, n, 1, K))
    beta = np.ones((1, n, 1))
    q = keys[None, :, None, :]
    out, fin = oracle.core(q, keys[None, :, None, :], vals[None, :, None, :], alpha, beta, 2.0,
                           initial_state=S0)
    S = fin[0, 0]
    np.testing.assert_allclose(S @ keys.T, vals.T, rtol=1e-10, atol=1e-11)
    expect = S0[0, 0] @ (np.eye(K) - keys.T @ keys) + vals.T @ keys
    np.testing.assert_allclose(S, expect, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(out[0, :, 0], 2.0 * vals, rtol=1e-10, atol=1e-11)


def test_delta_rule_storage_through_full_gate():
    """Same storage law through the library-facing entry: lower_bound=0 makes alpha == 1 for any g,
    beta logit +inf gives beta == 1 (bf16 keys are exact powers-of-two scaled unit vectors)."""
    K = V = 128
    n = 16
    keys = np.zeros((n, K))
    for j in range(n):
        keys[j, 3 * j] = 1.0                               # orthonormal and bf16-exact
    vals = _f64(_bits(rng.standard_normal((n, V))))
    g = _bits(rng.standard_normal((1, n, 1, K)) * 3)
    out, fin = oracle.fwd(_bits(keys[None, :, None]), _bits(keys[None, :, None]), _bits(vals[None, :, None]), g,
                          _bits(np.full((1, n, 1), np.inf)), 1.0, None, None, 0.0, None, None)
    np.testing.assert_allclose(fin[0, 0] @ keys.T, vals.T, rtol=0, atol=0)
    np.testing.assert_allclose(out[0, :, 0], vals, rtol=0, atol=0)


# ---------------------------------------------------------------- in-kernel q/k normalisation

def test_qk_l2norm_invariant_to_power_of_two_input_scale():
    """With q and k L2-normalised first, multiplying every q by 4 and every k by 1/2 (exact in
    bf16) leaves the forward pass unchanged up to the 1e-6 inside the square root; without the
    normalisation the same rescaling changes it."""
    d, bits, A, db, init, cu = _inputs("b2_t128_h8", T=40, H=2, raw_qk=True)
    q, k = _f64(bits["q"]), _f64(bits["k"])
    scaled = dict(bits, q=_bits(4.0 * q), k=_bits(0.5 * k))
    np.testing.assert_array_equal(_f64(scaled["q"]), 4.0 * q)   # the rescaling is exact
    np.testing.assert_array_equal(_f64(scaled["k"]), 0.5 * k)
    args = (d["scale"], A, db, d["lower_bound"], init, cu)
    o1, s1 = oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], *args, qk_l2norm=True)
    o2, s2 = oracle.fwd(scaled["q"], scaled["k"], bits["v"], bits["g"], bits["beta"], *args, qk_l2norm=True)
    np.testing.assert_allclose(o2, o1, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(s2, s1, rtol=1e-6, atol=1e-9)
    o3, _ = oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], *args)
    o4, _ = oracle.fwd(scaled["q"], scaled["k"], bits["v"], bits["g"], bits["beta"], *args)
    assert np.abs(o4 - o3).max() > 1e-2


def test_qk_l2norm_delta_rule_storage_with_scaled_one_hot_keys():
    """lower_bound = 0 (no decay), beta = 1, keys c_j e_j on distinct channels: the normalised
    key is a_j e_j with a_j = c_j / sqrt(c_j^2 + 1e-6), so the delta rule leaves S e_j = a_j v_j,
    and a later query d_j e_j (with k = 0, which the normalisation keeps at 0) reads
    scale * a_j * b_j * v_j with b_j = d_j / sqrt(d_j^2 + 1e-6)."""
    K = V = 128
    n = 12
    keys = np.zeros((2 * n, K))
    qrys = np.zeros((2 * n, K))
    for j in range(n):
        keys[j, 5 * j + 1] = (2.0, 8.0, 16.0)[j % 3]
        qrys[n + j, 5 * j + 1] = (4.0, 0.5, 32.0)[j % 3]
        qrys[j, 0] = 1.0
    vals = _f64(_bits(rng.standard_normal((2 * n, V))))
    g = _bits(rng.standard_normal((1, 2 * n, 1, K)))
    out, fin = oracle.fwd(_bits(qrys[None, :, None]), _bits(keys[None, :, None]), _bits(vals[None, :, None]), g,
                          _bits(np.full((1, 2 * n, 1), np.inf)), 0.5, None, None, 0.0, None, None, qk_l2norm=True)
    c = keys[:n].sum(axis=1)
    dq = qrys[n:].sum(axis=1)
    a = c / np.sqrt(c * c + 1e-6)
    b = dq / np.sqrt(dq * dq + 1e-6)
    np.testing.assert_allclose(out[0, n:, 0], 0.5 * (a * b)[:, None] * vals[:n], rtol=1e-12, atol=1e-14)
    unit = (keys[:n] != 0).astype(np.float64)
    np.testing.assert_allclose(fin[0, 0] @ unit.T, (a[:, None] * vals[:n]).T, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- gate

def test_gate_special_points():
    """lower_bound * sigmoid(exp(A_log) (g + dt_bias)) at points with known sigmoid values."""
    H, K = 3, 128
    g = np.zeros((1, H, K), np.float32)
    g[0, 0, :] = 1.0                    # with dt_bias = -1: argument 0 -> sigmoid 1/2
    g[0, 1, :] = 0.5                    # A_log = ln 2, no bias: argument ~1 -> sigmoid(1)
    g[0, 2, :] = 2.0                    # A_log = 0, bias 0: sigmoid(2)
    dt = np.zeros((H, K), np.float32)
    dt[0, :] = -1.0
    A_log = np.array([0.0, math.log(2.0), 0.0], np.float32)
    lb = -4.0
    a = oracle.gate(_bits(g), A_log, dt, lb)
    np.testing.assert_allclose(a[0, 0], lb / 2, rtol=0, atol=0)
    x1 = math.exp(float(np.float32(math.log(2.0)))) * 0.5
    np.testing.assert_allclose(a[0, 1], lb / (1 + math.exp(-x1)), rtol=1e-15)
    np.testing.assert_allclose(a[0, 1], lb * 0.7310585786300049, rtol=1e-7)
    np.testing.assert_allclose(a[0, 2], lb * 0.8807970779778823, rtol=1e-15)
    # no A_log / dt_bias: lower_bound * sigmoid(g)
    b = oracle.gate(_bits(g), None, None, lb)
    np.testing.assert_allclose(b[0, 0], lb * 0.7310585786300049, rtol=1e-15)


def test_gate_range_and_bf16_bound():
    """The gate lies in (lower_bound, 0) and a 16-token in-chunk cumsum stays within 16*|lower_bound|
    nats, so exp(+-cumsum) at lower_bound=-5 stays inside bf16 range ("Bounding the bf16
    Representable Range"; "bf16 Dynamic Range and Exponential Terms")."""
    g = _bits(rng.standard_normal((64, 4, 128)) * 4)
    a = oracle.gate(g, None, None, -5.0)
    assert np.all(a < 0) and np.all(a > -5.0)
    cs = np.cumsum(a.reshape(4, 16, 4, 128), axis=1)
    assert np.abs(cs).max() <= 80.0
    assert 80.0 / math.log(2) < 127                       # 2^{115.4} < bf16 max ~ 2^128


# ---------------------------------------------------------------- exact arithmetic

def _exact_recurrence(q, k, v, alpha, beta, scale, S0):
    """Token-by-token gated delta rule over Fractions; lists of lists, [v][c] state."""
    T, K = len(q), len(q[0])
    V = len(v[0])
    S = [row[:] for row in S0]
    outs = []
    for t in range(T):
        for r in range(V):
            for c in range(K):
                S[r][c] *= alpha[t][c]
        pred = [sum(S[r][c] * k[t][c] for c in range(K)) for r in range(V)]
        for r in range(V):
            e = beta[t] * (v[t][r] - pred[r])
            for c in range(K):
                S[r][c] += e * k[t][c]
        outs.append([scale * sum(S[r][c] * q[t][c] for c in range(K)) for r in range(V)])
    return outs, S


@pytest.mark.parametrize("K,V,T", [(2, 3, 20), (3, 2, 17), (4, 4, 12)])
def test_exact_rational_brute_force(K, V, T):
    r = np.random.default_rng(K * 100 + V * 10 + T)
    fr = lambda lo, hi: Fraction(int(r.integers(lo, hi)), 8)
    q = [[fr(-8, 9) for _ in range(K)] for _ in range(T)]
    k = [[fr(-8, 9) for _ in range(K)] for _ in range(T)]
    v = [[fr(-16, 17) for _ in range(V)] for _ in range(T)]
    alpha = [[Fraction(int(r.integers(1, 9)), 8) for _ in range(K)] for _ in range(T)]
    beta = [Fraction(int(r.integers(0, 9)), 8) for _ in range(T)]
    S0 = [[fr(-4, 5) for _ in range(K)] for _ in range(V)]
    scale = Fraction(3, 4)
    outs, S = _exact_recurrence(q, k, v, alpha, beta, scale, S0)
    to = lambda x: np.array(x, dtype=np.float64)
    out, fin = oracle.core(to(q)[None, :, None], to(k)[None, :, None], to(v)[None, :, None],
                           to(alpha)[None, :, None], to(beta)[None, :, None], float(scale),
                           initial_state=to(S0)[None, None])
    ex_o, ex_s = to([[float(x) for x in row] for row in outs]), to([[float(x) for x in row] for row in S])
    np.testing.assert_allclose(out[0, :, 0], ex_o, rtol=1e-12, atol=1e-12 * np.abs(ex_o).max())
    np.testing.assert_allclose(fin[0, 0], ex_s, rtol=1e-12, atol=1e-12 * np.abs(ex_s).max())


# ---------------------------------------------------------------- independent chunked evaluation

@pytest.mark.parametrize("name,kw", [("b1_t64_h1", {}), ("b2_t128_h8", {}),
                                     ("varlen_n16_h32", dict(lengths=[5, 37, 16, 1, 23], H=2))])
@pytest.mark.parametrize("chunk", [16, 7, 1])
def test_chunked_wy_agrees(name, kw, chunk):
    d, bits, A, db, init, cu = _inputs(name, **kw)
    o1, s1 = _run(bits, d, A, db, init, cu)
    o2, s2 = chunk_ref.fwd(*(_f64(bits[x]) for x in ("q", "k", "v", "g", "beta")), d["scale"], A, db,
                           d["lower_bound"], init, cu, chunk=chunk)
    assert np.abs(o1 - o2).max() <= 1e-10 * np.abs(o1).max()
    assert np.abs(s1 - s2).max() <= 1e-10 * np.abs(s1).max()


# ---------------------------------------------------------------- invariants

def test_split_call_state_carry():
    """T=128 in one call equals 64 + 64 with final_state -> initial_state ("Initial and Final States")."""
    d, bits, A, db, init, cu = _inputs("b2_t128_h8")
    o, s = _run(bits, d, A, db, init, None)
    first = {k: v[:, :64] for k, v in bits.items()}
    second = {k: v[:, 64:] for k, v in bits.items()}
    o1, s1 = _run(first, d, A, db, init, None)
    o2, s2 = _run(second, d, A, db, s1, None)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(s2, s, rtol=1e-12, atol=1e-14)


def test_final_state_is_affine_in_the_initial_state_and_segments_compose():
    """Each token maps S to S A_t + B_t (A_t = Diag(alpha_t)(I - beta_t k_t k_t^T), B_t = beta_t v_t
    k_t^T), so a segment maps S0 to S0 M + C with M the final state from S0 = I and v = 0 and C the
    final state from S0 = 0; two segments compose to one call. (The algebra a segment-parallel scan
    over a long sequence would rest on.)"""
    K = V = 6
    T = 50
    q = rng.standard_normal((1, T, 1, K))
    k = rng.standard_normal((1, T, 1, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, 1, V))
    alpha = rng.uniform(0.6, 1.0, (1, T, 1, K))
    beta = rng.uniform(0.0, 1.0, (1, T, 1))

    def seg(t0, t1, S0, vv):
        return oracle.core(q[:, t0:t1], k[:, t0:t1], vv[:, t0:t1], alpha[:, t0:t1], beta[:, t0:t1], 1.0,
                           initial_state=S0)[1][0, 0]

    eye = np.eye(K)[None, None]
    zero_v = np.zeros_like(v)
    M1, C1 = seg(0, 20, eye, zero_v), seg(0, 20, None, v)
    M2, C2 = seg(20, T, eye, zero_v), seg(20, T, None, v)
    S0 = rng.standard_normal((1, 1, V, K))
    _, full = oracle.core(q, k, v, alpha, beta, 1.0, initial_state=S0)
    np.testing.assert_allclose(S0[0, 0] @ M1 + C1, seg(0, 20, S0, v), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose((S0[0, 0] @ M1 + C1) @ M2 + C2, full[0, 0], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S0[0, 0] @ (M1 @ M2) + (C1 @ M2 + C2), full[0, 0], rtol=1e-11, atol=1e-12)


def test_varlen_equals_separate_calls():
    """Packed sequences with cu_seqlens equal separate per-sequence calls ("Variable-Length Mode")."""
    lens = [5, 37, 16, 1, 23, 0, 40]
    d, bits, A, db, init, cu = _inputs("varlen_n16_h32", lengths=lens, H=3)
    o, s = _run(bits, d, A, db, init, cu)
    for i in range(len(lens)):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        sub = {k: v[:, t0:t1] for k, v in bits.items()}
        oi, si = _run(sub, d, A, db, init[i:i + 1], None)
        assert np.array_equal(oi, o[:, t0:t1])
        assert np.array_equal(si[0], s[i])
    # an empty sequence hands its initial state through unchanged
    assert np.array_equal(s[5], init[5])


def test_contraction_bound():
    """With ||k||=1, beta in [0,1], alpha <= 1: ||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t||."""
    d, bits, A, db, init, cu = _inputs("b2_t128_h8", B=1, H=2, T=40)
    S = init
    beta = 1 / (1 + np.exp(-_f64(bits["beta"])))
    for t in range(40):
        sub = {k: v[:, t:t + 1] for k, v in bits.items()}
        _, S1 = _run(sub, d, A, db, S, None)
        for h in range(2):
            vn = np.linalg.norm(_f64(bits["v"])[0, t, h])
            assert np.linalg.norm(S1[0, h]) <= np.linalg.norm(S[0, h]) + beta[0, t, h] * vn + 1e-12
        S = S1


def test_scale_is_linear_on_output_only():
    """scale multiplies the output and never the state ("Global Scaling Factor")."""
    d, bits, A, db, init, cu = _inputs("b2_t128_h8", B=1, H=2, T=33)
    o1, s1 = oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], 1.0, A, db, -2.0, init)
    o2, s2 = oracle.fwd(bits["q"], bits["k"], bits["v"], bits["g"], bits["beta"], 0.25, A, db, -2.0, init)
    np.testing.assert_allclose(o2, 0.25 * o1, rtol=1e-15, atol=0)
    assert np.array_equal(s1, s2)


# ------------------------------------------------------------ per-chunk terms (step checks)

def test_chunk_terms_against_the_gate_and_closed_forms():
    """chunk_terms: its gate cumsum is the cumsum of the oracle's gate (log2 units), T inverts
    I + A, and with lower_bound = 0 (no decay) A and P reduce to beta-scaled and plain dot
    products (the decay-free chunk matrices)."""
    d = W.make("b1_t64_h1")
    sl = slice(16, 32)
    qb, kb, gb = (W.bf16_bits(d[x][0, sl, 0].contiguous()) for x in ("q", "k", "g"))
    bl = _f64(W.bf16_bits(d["beta"][0, sl, 0].contiguous()))
    A_log, dt = float(d["A_log"][0]), d["dt_bias"][0].double().numpy()
    q, k, g = _f64(qb), _f64(kb), _f64(gb)
    G2, beta, A, P, T = chunk_ref.chunk_terms(q, k, g, bl, A_log, dt, -5.0)
    ga = oracle.gate(gb[:, None, :], d["A_log"][:1].numpy(), d["dt_bias"][:1].numpy(), -5.0)[:, 0, :]
    assert np.allclose(G2, np.cumsum(ga, axis=0) / math.log(2.0), rtol=0, atol=1e-12)
    assert np.allclose(T @ (np.eye(16) + A), np.eye(16), rtol=0, atol=1e-12)
    assert np.allclose(beta, 1.0 / (1.0 + np.exp(-bl)))
    G2z, _, Az, Pz, _ = chunk_ref.chunk_terms(q, k, g, bl, A_log, dt, 0.0)
    assert np.all(G2z == 0.0)
    assert np.allclose(Az, np.tril(beta[:, None] * (k @ k.T), -1), rtol=0, atol=1e-13)
    assert np.allclose(Pz, np.tril(q @ k.T), rtol=0, atol=1e-13)
