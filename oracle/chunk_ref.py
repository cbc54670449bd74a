"""Test infrastructure only: an independent fp64 chunked (WY) evaluation of
the KDA forward pass, used to pin the per-token oracle in ``kda_oracle.c``.

It shares no code with that oracle: the recurrence is reached here through the
chunked form instead of token by token. For one (sequence, head) and one chunk
of rows r = 1..L starting from state S0 (V x K):

* Gamma_r = prod_{s<=r} alpha_s (per channel), gamma = Gamma_L;
* A[r, j] = beta_r * sum_c k_r[c] k_j[c] Gamma_r[c] / Gamma_j[c]   for j < r;
* (I + A) E = diag(beta) V - diag(beta) (K * Gamma) S0^T, solved by forward
  substitution (E has the written rows e_r of the delta rule);
* o_r = scale * (S0 (q_r * Gamma_r) + sum_{j<=r} P[r, j] e_j) with
  P[r, j] = sum_c q_r[c] k_j[c] Gamma_r[c] / Gamma_j[c];
* S_L = S0 Diag(gamma) + sum_j e_j (k_j * gamma / Gamma_j)^T.

These identities follow by unrolling the gated delta rule inside the chunk.
The chunk size is a free parameter: any size must give the per-token result.
The same chunked form underlies "How FlashKDA's CHUNK Size of 16 Improves
Numerical Stability Over CHUNK 64" (16-token chunks, the unit-lower chunk
matrix and its inverse); here it is evaluated in fp64 with natural exponents.
"""
from __future__ import annotations

import numpy as np


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _chunk_matrices(qc, kc, Gam, bc):
    """A[r, j] = beta_r sum_c k_r k_j Gamma_r / Gamma_j for j < r and P[r, j] = sum_c q_r k_j
    Gamma_r / Gamma_j for j <= r (zero elsewhere), for one chunk's rows."""
    L = kc.shape[0]
    A = np.zeros((L, L))
    P = np.zeros((L, L))
    for r in range(L):
        for j in range(r + 1):
            ratio = Gam[r] / Gam[j]
            if j < r:
                A[r, j] = bc[r] * np.dot(kc[r] * kc[j], ratio)
            P[r, j] = np.dot(qc[r] * kc[j], ratio)
    return A, P


def chunk_terms(q, k, g, beta_logit, A_log=None, dt_bias=None, lower_bound=-5.0):
    """The per-chunk quantities of one chunk of one head, for step-by-step checks (rows
    r = 0..L-1, inputs float64 widened from bf16: q, k, g [L, K], beta_logit [L], A_log a
    scalar or None, dt_bias [K] or None). Returns the gate's inclusive in-chunk cumsum in
    log2 units [L, K], beta [L], A and P as in the chunked form, and T = (I + A)^-1."""
    a = 1.0 if A_log is None else np.exp(float(A_log))
    b = 0.0 if dt_bias is None else np.asarray(dt_bias, np.float64)
    G = np.cumsum(lower_bound * _sigmoid(a * (g + b)), axis=0)   # natural-log gate, summed
    beta = _sigmoid(beta_logit)
    A, P = _chunk_matrices(q, k, np.exp(G), beta)
    T = np.linalg.inv(np.eye(k.shape[0]) + A)
    return G / np.log(2.0), beta, A, P, T


def chunk_unit(q, k, v, alpha, beta, scale, S0, chunk):
    """One (sequence, head) unit. ``q, k, alpha``: [L_tot, K]; ``v``: [L_tot, V];
    ``beta``: [L_tot] activated; ``S0``: [V, K]. Returns (out [L_tot, V], S)."""
    Ltot = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((Ltot, v.shape[1]), np.float64)
    for s in range(0, Ltot, chunk):
        e = min(s + chunk, Ltot)
        L = e - s
        Gam = np.cumprod(alpha[s:e], axis=0)          # [L, K]
        kc, qc, vc, bc = k[s:e], q[s:e], v[s:e], beta[s:e]
        A, P = _chunk_matrices(qc, kc, Gam, bc)
        rhs = bc[:, None] * (vc - (kc * Gam) @ S.T)   # [L, V]
        E = np.zeros_like(rhs)
        for r in range(L):                             # forward substitution
            E[r] = rhs[r] - A[r, :r] @ E[:r]
        out[s:e] = scale * ((qc * Gam) @ S.T + P @ E)
        gam = Gam[-1]
        S = S * gam[None, :] + E.T @ (kc * (gam[None, :] / Gam))
    return out, S


def fwd(q, k, v, g, beta_logit, scale, A_log=None, dt_bias=None, lower_bound=-5.0,
        initial_state=None, cu_seqlens=None, chunk=16):
    """Chunked fp64 forward on float64 arrays (already widened from bf16).

    Shapes as the library: q, k, g [B,T,H,K]; v [B,T,H,V]; beta_logit [B,T,H];
    initial_state [B|N,H,V,K]. Returns (out, final_state)."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    a = np.ones(H) if A_log is None else np.exp(np.asarray(A_log, np.float64))
    b = np.zeros((H, K)) if dt_bias is None else np.asarray(dt_bias, np.float64)
    alpha = np.exp(lower_bound * _sigmoid(a[None, None, :, None] * (g + b[None, None])))
    beta = _sigmoid(beta_logit)
    if cu_seqlens is not None:
        spans = [(0, int(cu_seqlens[i]), int(cu_seqlens[i + 1])) for i in range(len(cu_seqlens) - 1)]
    else:
        spans = [(bb, 0, T) for bb in range(B)]
    out = np.zeros((B, T, H, V))
    fin = np.zeros((len(spans), H, V, K))
    for n, (bb, t0, t1) in enumerate(spans):
        for h in range(H):
            S0 = np.zeros((V, K)) if initial_state is None else initial_state[n, h]
            o, S = chunk_unit(q[bb, t0:t1, h], k[bb, t0:t1, h], v[bb, t0:t1, h],
                              alpha[bb, t0:t1, h], beta[bb, t0:t1, h], scale, S0, chunk)
            out[bb, t0:t1, h] = o
            fin[n, h] = S
    return out, fin
