"""CHUNK = 16 against 32 and 64 on the numerics of the chunk products (CPU, no GPU).

"How FlashKDA's CHUNK Size of 16 Improves Numerical Stability Over CHUNK 64" -- "bf16 Dynamic
Range and Exponential Terms": the factors K 2^{G - G_ref} and K 2^{G_ref - G} of the chunk matrix
must stay inside bf16's range. At lower_bound = -5 the in-chunk cumsum of the gate reaches
C |lower_bound| log2(e) bits over C tokens. With the exponent reference at the chunk start the
factors span 2^{+-115} for C = 16 but 2^{+-462} for C = 64; the mid-chunk reference halves that.
These tests build the bf16 factors of worst-case and random chunks, count factors that leave
bf16's finite normal range, and compare A = tril(beta K_l K_r^T) (fp32 accumulation of bf16
products) with the fp64 value."""
import math

import numpy as np
import pytest
import torch

LOG2E = 1.0 / math.log(2.0)
BF16_MAX_EXP, BF16_MIN_NORMAL_EXP = 127, -126


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def chunk_factors(C, lower_bound, ref, seed=0, saturate=True, K=64):
    """One chunk of C tokens: unit-norm keys, gate saturated at lower_bound (the worst case) or
    random; returns (G in log2 units [C, K], k [C, K], beta [C])."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((C, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    sig = np.ones((C, K)) if saturate else 1.0 / (1.0 + np.exp(-rng.standard_normal((C, K))))
    G = np.cumsum(lower_bound * sig, axis=0) * LOG2E
    Gref = np.zeros(K) if ref == "start" else G[(C - 1) // 2]
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    return G, Gref, k, beta


def factor_exponent_span(C, lower_bound, ref):
    G, Gref, _, _ = chunk_factors(C, lower_bound, ref)
    return float(np.max(np.abs(G - Gref)))


@pytest.mark.parametrize("C,ref,fits", [(16, "start", True), (16, "mid", True), (32, "start", False),
                                        (32, "mid", True), (64, "start", False), (64, "mid", False)])
def test_exponent_span_against_bf16_range(C, ref, fits):
    span = factor_exponent_span(C, -5.0, ref)
    expect = (C if ref == "start" else C - (C - 1) // 2 - 1) * 5.0 * LOG2E
    assert span == pytest.approx(expect, rel=1e-12)
    # K 2^{-span} must stay a normal bf16 for |k| ~ 2^-4 (unit norm over 64 channels)
    assert (span + 4 <= -BF16_MIN_NORMAL_EXP) == fits


def chunk_matrix_error(C, lower_bound, ref, seed):
    """Relative Frobenius error of A built from bf16 factors (fp32 accumulation) against fp64;
    inf if a factor overflowed or the product is not finite."""
    G, Gref, k, beta = chunk_factors(C, lower_bound, ref, seed, saturate=False)
    with np.errstate(over="ignore", invalid="ignore"):
        kl = _bf16(k * np.exp2(G - Gref))
        kr = _bf16(k * np.exp2(Gref - G))
        A16 = np.tril(beta[:, None] * (kl.astype(np.float32) @ kr.T.astype(np.float32)), -1).astype(np.float64)
    ratio = np.exp2(G[:, None, :] - G[None, :, :])
    A = np.tril(beta[:, None] * np.einsum("rc,jc,rjc->rj", k, k, ratio), -1)
    if not np.all(np.isfinite(A16)):
        return math.inf
    return float(np.linalg.norm(A16 - A) / np.linalg.norm(A))


def test_chunk_16_products_are_accurate_and_chunk_64_breaks_without_rescaling():
    errs = {(C, ref): max(chunk_matrix_error(C, -5.0, ref, s) for s in range(4))
            for C in (16, 32, 64) for ref in ("start", "mid")}
    # CHUNK = 16: bf16 factors give the chunk matrix to bf16 accuracy with either reference
    assert errs[(16, "start")] < 1e-2 and errs[(16, "mid")] < 1e-2
    # CHUNK = 64 at lower_bound = -5: the start-referenced factors overflow bf16
    assert math.isinf(errs[(64, "start")])
