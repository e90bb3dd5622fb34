"""Independent fp64 chunked formulation of the gated delta rule (TEST INFRASTRUCTURE).

This is a second, different algorithm for the function ``gdn_ref.c`` defines;
tests use it only to pin the token recurrence. It is written from the
chunked closed form, derived by unrolling the recurrence inside one chunk:

With chunk-start state S (dk x dv), in-chunk cumulative log-decay
G_i = sum_{j<=i} g_j, gamma_i = exp(G_i) and x_i = beta_i * delta_i (the
corrected value written by token i),

    (I + A) X = diag(beta) V - diag(beta * gamma) K S,
    A_ij = beta_i * (gamma_i / gamma_j) * k_i . k_j   for j < i, else 0,
    o_i  = scale * [gamma_i * S^T q_i + sum_{j<=i} (gamma_i / gamma_j)(q_i . k_j) x_j],
    S'   = gamma_L * S + sum_j (gamma_L / gamma_j) k_j x_j^T     (L = last row).

That is the two-phase split of "Optimizing GDN Chunk Prefill on Intel AMX
CPU" (section 4: A, its triangular solve, w and u; section 5: the state
contribution, the local attention output and the state update), with the
plus sign of (I + A) fixed by the derivation. The triangular system is
solved with SciPy's ``solve_triangular`` (a library primitive); nothing is
blocked, fused or reordered beyond the closed form above.

Per-channel gates (g of shape [T, Hv, dk]): G_i becomes a vector over the key
dimension and every scalar ratio gamma_i / gamma_j moves inside the dot
products, one factor per key channel d:

    A_ij = beta_i * sum_d k_id k_jd exp(G_id - G_jd)        for j < i,
    (I + A) X = diag(beta) V - diag(beta) (exp(G) * K) S,
    o_i  = scale * [(exp(G_i) * q_i)^T S + sum_{j<=i} (sum_d q_id k_jd exp(G_id - G_jd)) x_j],
    S'   = diag(exp(G_L)) S + (exp(G_L - G) * K)^T X,

which reduces to the scalar form when all channels carry the same gate.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def chunked_forward(q, k, v, g, beta, scale=None, initial_state=None,
                    cu_seqlens=None, chunk_size=64, qk_l2norm=False, eps=1e-6):
    """Chunked fp64 evaluation. Same shapes and conventions as
    ``oracle.recurrent_forward``. Returns (out [T,Hv,dv], final [N,Hv,dv,dk])."""
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    HG = Hv // H
    if scale is None or not (scale > 0):
        scale = 1.0 / np.sqrt(dk)
    if qk_l2norm:
        q = q / np.sqrt((q * q).sum(-1, keepdims=True) + eps)
        k = k / np.sqrt((k * k).sum(-1, keepdims=True) + eps)
    cu = (np.array([0, T]) if cu_seqlens is None
          else np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu")
                          else cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    s0 = _f64(initial_state)
    out = np.zeros((T, Hv, dv))
    final = np.zeros((N, Hv, dv, dk))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for hv in range(Hv):
            h = hv // HG
            S = np.zeros((dk, dv)) if s0 is None else s0[n, hv].T.copy()
            for c0 in range(t0, t1, chunk_size):
                c1 = min(c0 + chunk_size, t1)
                K = k[c0:c1, h]              # [L, dk]
                Q = q[c0:c1, h]
                V = v[c0:c1, hv]             # [L, dv]
                b = beta[c0:c1, hv]          # [L]
                L = c1 - c0
                if g.ndim == 3:
                    S, o, X = _channel_chunk(K, Q, V, b, g[c0:c1, hv], S)
                    out[c0:c1, hv] = scale * o
                    continue
                G = np.cumsum(g[c0:c1, hv])  # inclusive, within the chunk
                ii, jj = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
                ratio = np.exp(np.where(jj <= ii, G[:, None] - G[None, :], -np.inf))
                A = np.where(jj < ii, b[:, None] * ratio * (K @ K.T), 0.0)
                rhs = b[:, None] * V - (b * np.exp(G))[:, None] * (K @ S)
                X = solve_triangular(np.eye(L) + A, rhs, lower=True, unit_diagonal=True)
                o = np.exp(G)[:, None] * (Q @ S) + (ratio * (Q @ K.T)) @ X
                out[c0:c1, hv] = scale * o
                S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * K).T @ X
            final[n, hv] = S.T
    return out, final


def _channel_chunk(K, Q, V, b, g, S):
    """One chunk with per-channel gates g [L, dk]; returns (S', o / scale, X)."""
    L = K.shape[0]
    G = np.cumsum(g, axis=0)                                  # [L, dk]
    ii, jj = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
    diff = np.where((jj <= ii)[:, :, None], G[:, None, :] - G[None, :, :], -np.inf)
    ratio = np.exp(diff)                                      # [L, L, dk], 0 above the diagonal
    KK = np.einsum("id,jd,ijd->ij", K, K, ratio)
    QK = np.einsum("id,jd,ijd->ij", Q, K, ratio)
    A = np.where(jj < ii, b[:, None] * KK, 0.0)
    rhs = b[:, None] * V - b[:, None] * ((np.exp(G) * K) @ S)
    X = solve_triangular(np.eye(L) + A, rhs, lower=True, unit_diagonal=True)
    o = (np.exp(G) * Q) @ S + QK @ X
    S = np.exp(G[-1])[:, None] * S + (np.exp(G[-1][None, :] - G) * K).T @ X
    return S, o, X
