"""Per-step parity of the tcgen05 kernel's own chunk operands: the prep slot of every chunk, as
the tensor core reads it (kda_probe_slots), decoded and compared with fp64 values built from
oracle.chunk_ref.chunk_terms and the chunk algebra of the kernel:
  Z' = [K Gamma ; Q Gamma] Diag(gamma_{n-1}),  Kbar = K 2^(G_end - G),  gamma = 2^G_end,
  TM = [T' ; s M],  Phi = [[-T', 0], [-s M, s I]],  T' = (I + A)^-1 diag(beta),  M = P T',
  (H Phi^T)^T with H = Kbar_{n-1} [K Gamma ; Q Gamma]^T,  H''^T with H'' = Kbar_{n-2} Diag(gamma_{n-1}) [K Gamma ; Q Gamma]^T
(G: the gate's in-chunk cumsum in log2 units, Gamma = 2^G; "FlashKDA lower_bound Parameter ..."
-- "Conversion to the Gate Scale Factor", "How FlashKDA's CHUNK Size of 16 ..." -- "Efficient 16x16
Matrix Inversion").

Tolerances. With lower_bound = 0 every gate is exactly 0 (Gamma = gamma = 1), so Z', Kbar, V and
gamma are exact roundings of the inputs (bf16, f16) and are compared bit for bit. With lower_bound
!= 0 the kernel's gate uses tanh.approx: |d sigma| <= 2.5e-4 per token, so |d G| <= 16
|lower_bound| log2(e) 2.5e-4 = eps_G over a chunk and every factor 2^(+-G) is within
dg = 2^eps_G - 1 (relative) of the fp64 value; bf16 rounding adds 2^-8, f16 2^-11. T' and M carry
the parity tolerance of the forward pass (their fp16 Neumann products). The cross-chunk products
are sums over 128 channels, so they are bounded against the sums of absolute values of their
terms: (H Phi^T)^T within 2e-2 (T', M) + 3 dg of |Kbar_{n-1}| |Z|^T |Phi|^T, H''^T within 2^-9 +
3 dg of |Kbar_{n-2}| Diag(gamma) |Z|^T. Their f16 operands (Kbar, K Gamma, Q Gamma and gamma) lose
at most 2^-25 absolute each where they fall below f16's normal range, so every term a b of such a
sum is off by at most 2^-25 (|a| + |b| + |a| |b|) beyond the relative part; the bound adds 2^-24
times those sums (before the product with Phi for (H Phi^T)^T), and the f16 rounding of the
stored result itself adds 2^-25 absolute (f16 subnormal spacing 2^-24) on top of 2^-11 relative.
(H Phi^T)^T is formed from H^w rounded to f16 once more (the A operand of its MMA), which adds
2^-25 sum_k |Phi_mk| absolute to row m."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close

pytestmark = pytest.mark.gpu

SLOT_LAYOUT = {"Z": 0, "V": 8192, "KB": 12288, "PHI": 16384, "TM": 20480, "CC": 21504, "HP": 22528, "GAM": 23552}


def _sw128(rows):
    """byte offset of (row, col) in a 16-bit tile of `rows` rows x 128 columns stored as two
    64-column blocks of 128-byte rows with the 128-byte swizzle"""
    r = np.arange(rows)[:, None]
    c = np.arange(128)[None, :]
    return (c >> 6) * (rows * 128) + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2


def _cm16(n_rows):
    n = np.arange(n_rows)[:, None]
    k = np.arange(16)[None, :]
    return (n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2


def _cm32():
    n = np.arange(32)[:, None]
    k = np.arange(32)[None, :]
    return (n >> 3) * 1024 + (k >> 2) * 128 + (n & 7) * 16 + (k & 3) * 4


def _u16(slot, base, off):
    b = slot[base + off[..., None] + np.array([0, 1])]
    return (b[..., 0].astype(np.uint16) | (b[..., 1].astype(np.uint16) << 8))


def _bf16(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f16(bits):
    return bits.view(np.float16).astype(np.float64)


def _f32(slot, base, off):
    b = slot[base + off[..., None] + np.arange(4)]
    return b.astype(np.uint8).copy().view(np.float32)[..., 0].astype(np.float64)


def decode(slot):
    L = SLOT_LAYOUT
    return {
        "Z": _bf16(_u16(slot, L["Z"], _sw128(32))),
        "V": _f16(_u16(slot, L["V"], _sw128(16))),
        "KB": _f16(_u16(slot, L["KB"], _sw128(16))),
        "PHI": _f32(slot, L["PHI"], _cm32()),
        "TM": _f16(_u16(slot, L["TM"], _cm16(32))),
        "CC": _f16(_u16(slot, L["CC"], _cm16(32))),
        "HP": _f16(_u16(slot, L["HP"], _cm16(32))),
        "GAM": slot[L["GAM"]:L["GAM"] + 512].copy().view(np.float32).astype(np.float64),
    }


def reference(d, lb, T):
    """fp64 slot contents of every chunk of head 0 of batch row 0 (rows past T are zero keys and
    queries, beta 0 and no gate, as the kernel pads them)."""
    import oracle.chunk_ref as chunk_ref
    f64 = lambda t: t.double().numpy()
    q, k, v, g = (f64(d[x][0, :T, 0]) for x in ("q", "k", "v", "g"))
    bl = f64(d["beta"][0, :T, 0])
    A_log = None if d["A_log"] is None else float(d["A_log"][0])
    dt = None if d["dt_bias"] is None else d["dt_bias"][0].double().numpy()
    s = d["scale"]
    out = []
    for n in range((T + 15) // 16):
        a, e = 16 * n, min(16 * n + 16, T)
        L = e - a
        G2, beta, A, P, Tm = chunk_ref.chunk_terms(q[a:e], k[a:e], g[a:e], bl[a:e], A_log, dt, lb)
        pad = lambda x, fill: np.concatenate([x, np.repeat(fill, 16 - L, axis=0)]) if L < 16 else x
        G = pad(G2, G2[-1:])
        kc, qc = pad(k[a:e], np.zeros((1, 128))), pad(q[a:e], np.zeros((1, 128)))
        vc = pad(v[a:e], np.zeros((1, 128)))
        bt = np.concatenate([beta, np.zeros(16 - L)])
        Tf = np.eye(16); Tf[:L, :L] = Tm
        Pf = np.zeros((16, 16)); Pf[:L, :L] = P
        Gam = np.exp2(G)
        Tp = Tf * bt[None, :]
        M = Pf @ Tp
        out.append(dict(G=G, Gam=Gam, gam=Gam[15], KG=kc * Gam, QG=qc * Gam, KB=kc * np.exp2(G[15] - G), V=vc,
                        V16=vc.astype(np.float16).astype(np.float64),
                        TM=np.concatenate([Tp, s * M]),
                        PHI=np.block([[-Tp, np.zeros((16, 16))], [-s * M, s * np.eye(16)]])))
    for n, c in enumerate(out):
        gp = out[n - 1]["gam"] if n >= 1 else np.ones(128)
        Zf = np.concatenate([c["KG"], c["QG"]])
        c["Z"] = Zf * gp[None, :]
        c["KB16"] = c["KB"].astype(np.float16).astype(np.float64)
        # sum_c (|a_c| + |b_c| + |a_c| |b_c|) for every (row of a, row of b): the f16 underflow term
        under = lambda a, b: (np.ones_like(a) @ np.abs(b).T + np.abs(a) @ np.ones_like(b).T
                              + np.abs(a) @ np.abs(b).T)
        if n >= 1:
            kb = out[n - 1]["KB"]
            H = kb @ Zf.T                                     # [16 j][32]
            c["CC"] = (H @ c["PHI"].T).T                      # [32][16]
            c["CC_abs"] = (np.abs(kb) @ np.abs(Zf).T @ np.abs(c["PHI"]).T).T
            c["CC_abs1"] = (under(kb, Zf) @ np.abs(c["PHI"]).T).T
            c["CC_phi1"] = np.repeat(np.abs(c["PHI"]).sum(axis=1)[:, None], 16, axis=1)   # [32 m][16 j]
        if n >= 2:
            kb = out[n - 2]["KB"]
            c["HP"] = ((kb * gp[None, :]) @ Zf.T).T
            c["HP_abs"] = ((np.abs(kb) * gp[None, :]) @ np.abs(Zf).T).T
            c["HP_abs1"] = under(kb, Zf).T
    return out


def _run(d, lb, T):
    import gated_linear_attention_kda_gb300 as kda
    cu = lambda t: t.contiguous().cuda()
    A_log = None if d["A_log"] is None else cu(d["A_log"][0:1])
    dt = None if d["dt_bias"] is None else cu(d["dt_bias"][0])
    dump, _ = kda.probe_slots(cu(d["q"][0, :T, 0]), cu(d["k"][0, :T, 0]), cu(d["v"][0, :T, 0]), cu(d["g"][0, :T, 0]),
                              cu(d["beta"][0, :T, 0]), d["scale"], A_log, dt, lb)
    kda.check_device_status()
    return [decode(row) for row in dump.cpu().numpy()]


def _within(name, got, ref, rel, abs_=0.0, scale=None):
    """|got - ref| <= abs_ + rel * (scale if given else |ref|), elementwise"""
    sc = np.abs(ref) if scale is None else scale
    tol = abs_ + rel * sc
    bad = np.abs(got - ref) > tol
    if bad.any():
        i = np.unravel_index(np.argmax(np.abs(got - ref) / np.maximum(tol, 1e-300)), got.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements off; worst at {i}: got {got[i]:.6e} "
                             f"ref {ref[i]:.6e} tol {tol[i] if np.ndim(tol) else tol:.3e}")


def test_slot_operands_without_decay_are_exact_roundings():
    """lower_bound 0: Gamma = gamma = 1, so Z' and Kbar are the bf16 / f16 inputs themselves."""
    d = W.make("b1_t64_h1")
    T, lb = 64, 0.0
    got, ref = _run(d, lb, T), reference(d, lb, T)
    for n, (gs, rs) in enumerate(zip(got, ref)):
        assert np.array_equal(gs["Z"], rs["Z"]), f"chunk {n}: Z'"
        assert np.array_equal(gs["KB"], rs["KB16"]), f"chunk {n}: Kbar"
        assert np.array_equal(gs["V"], rs["V16"]), f"chunk {n}: V"
        assert np.array_equal(gs["GAM"], rs["gam"]), f"chunk {n}: gamma"
        assert_close(f"chunk {n}: TM", gs["TM"], rs["TM"])
        assert_close(f"chunk {n}: Phi", gs["PHI"], rs["PHI"])
        if n >= 1:
            _within(f"chunk {n}: (H Phi^T)^T", gs["CC"], rs["CC"], 2e-2, abs_=2.0 ** -25 + 2.0 ** -24 * rs["CC_phi1"],
                    scale=rs["CC_abs"] + 2.0 ** -19 * rs["CC_abs1"])
        if n >= 2:
            _within(f"chunk {n}: H''^T", gs["HP"], rs["HP"], 2.0 ** -9, abs_=2.0 ** -25,
                    scale=rs["HP_abs"] + 2.0 ** -15 * rs["HP_abs1"])


@pytest.mark.parametrize("name,lb,T", [("b1_t64_h1", -5.0, 64), ("b2_t128_h8", -2.0, 45), ("b2_t128_h8", -0.5, 64)])
def test_slot_operands_match_the_chunk_algebra(name, lb, T):
    d = W.make(name)
    got, ref = _run(d, lb, T), reference(d, lb, T)
    eps_g = 16 * abs(lb) * math.log2(math.e) * 2.5e-4
    dg = 2.0 ** eps_g - 1.0                 # one factor 2^(+-G) from the tanh.approx gate
    for n, (gs, rs) in enumerate(zip(got, ref)):
        _within(f"chunk {n}: gamma", gs["GAM"], rs["gam"], dg + 2.0 ** -20, abs_=1e-38)
        _within(f"chunk {n}: Z'", gs["Z"], rs["Z"], (1 + dg) ** 2 * (1 + 2.0 ** -8) - 1, abs_=1e-38)
        _within(f"chunk {n}: Kbar", gs["KB"], rs["KB"], dg + 2.0 ** -10, abs_=2.0 ** -24)
        assert np.array_equal(gs["V"], rs["V16"]), f"chunk {n}: V"
        assert_close(f"chunk {n}: TM", gs["TM"], rs["TM"])
        assert_close(f"chunk {n}: Phi", gs["PHI"], rs["PHI"])
        if n >= 1:
            rel = 2e-2 + 3 * dg
            _within(f"chunk {n}: (H Phi^T)^T", gs["CC"], rs["CC"], rel, abs_=2.0 ** -25 + 2.0 ** -24 * rs["CC_phi1"],
                    scale=rs["CC_abs"] + 2.0 ** -24 / rel * rs["CC_abs1"])
        if n >= 2:
            rel = 2.0 ** -9 + 3 * dg
            _within(f"chunk {n}: H''^T", gs["HP"], rs["HP"], rel, abs_=2.0 ** -25,
                    scale=rs["HP_abs"] + 2.0 ** -24 / rel * rs["HP_abs1"])
