"""fp64 oracle of the gated-DeltaNet front end (TEST INFRASTRUCTURE ONLY).

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may import it;
the product path never does.

The front end turns the qkv projection output into q, k, v, following the
llama.cpp page (PrismML-Eng/llama.cpp pull 399, "What", item 1, and "How
(exactness)"): a causal depthwise convolution of width d_conv over each
channel, whose inputs are the d_conv - 1 inputs saved from before the
sequence (the conv state) followed by the sequence's own rows, then SiLU, then
the per-head L2 norm of q and k. With xx the concatenation [state, x] of one
channel,

    y_t = SiLU( sum_{j=0}^{d_conv-1} w[j] * xx[t + j] )      (no bias)

so w[d_conv-1] multiplies the current token. The new conv state is the last
d_conv - 1 entries of xx (old state entries when the sequence is shorter), and
snapshot s (for rolling a speculative batch back) is the state after the
sequence's token s: xx[s + 1 .. s + d_conv - 1].

Channel order of the projection output: q (H heads x dk), then k (H x dk),
then v (Hv x dv). The L2 norm divides each q and k head row by
sqrt(sum x^2 + eps).

Written as plain loops over sequences and taps with NumPy arithmetic in fp64;
no blocking or reordering beyond the definition above.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def silu(x):
    return x / (1.0 + np.exp(-x))


def conv_front(x, w, H, Hv, dk=128, dv=128, conv_state=None, cu_seqlens=None,
               l2norm=False, eps=1e-6, n_snapshots=0):
    """x [T, C] (C = 2*H*dk + Hv*dv), w [C, d_conv], conv_state [N, C, d_conv-1]
    or None (zeros), cu_seqlens [N+1] or None (one sequence of T rows).

    Returns q [T,H,dk], k [T,H,dk], v [T,Hv,dv], new conv state [N, C, d_conv-1]
    and, if n_snapshots > 0, snapshots [N, n_snapshots, C, d_conv-1] (entries for
    tokens past a sequence's end keep the state after its last token)."""
    x = _f64(x)
    w = _f64(w)
    T, C = x.shape
    d = w.shape[1]
    assert C == 2 * H * dk + Hv * dv
    cu = [0, T] if cu_seqlens is None else [int(a) for a in np.asarray(cu_seqlens).tolist()]
    N = len(cu) - 1
    s0 = np.zeros((N, C, d - 1)) if conv_state is None else _f64(conv_state)
    y = np.zeros((T, C))
    s1 = np.zeros((N, C, d - 1))
    snaps = np.zeros((N, n_snapshots, C, d - 1)) if n_snapshots else None
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        xx = np.concatenate([s0[n].T, x[a:b]], axis=0)  # [d-1+len, C]
        L = b - a
        for t in range(L):
            acc = np.zeros(C)
            for j in range(d):
                acc = acc + w[:, j] * xx[t + j]
            y[a + t] = silu(acc)
        s1[n] = xx[L:L + d - 1].T
        for s in range(n_snapshots):
            e = min(s, L - 1) + 1 if L > 0 else 0  # state after token min(s, L-1)
            snaps[n, s] = xx[e:e + d - 1].T
    q = y[:, :H * dk].reshape(T, H, dk)
    k = y[:, H * dk:2 * H * dk].reshape(T, H, dk)
    v = y[:, 2 * H * dk:].reshape(T, Hv, dv)
    if l2norm:
        q = q / np.sqrt((q * q).sum(-1, keepdims=True) + eps)
        k = k / np.sqrt((k * k).sum(-1, keepdims=True) + eps)
    return q, k, v, s1, snaps
