"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each pin takes an oracle library handle (so that the mutation tests can run
the same pins on deliberately broken copies of the oracle) and raises
AssertionError when the oracle disagrees with what the mathematics fixes:

* exact-rational brute force on tiny inputs, written in the transition-matrix
  form S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
  (a different arrangement of the same recurrence, evaluated without rounding);
* the independent chunked fp64 formulation (oracle/chunked.py);
* closed form 1: mutually orthonormal keys turn the delta rule into decayed
  causal linear attention, a masked (Q K^T * D) V product;
* closed form 2: beta = 1 with unit keys makes S_t^T k_t = v_t exactly;
* invariants: beta = 0 leaves the state to decay only (S_t = exp(cum g) S_0);
* per-channel gates: exact rationals, the chunked form, uniform gates = scalar
  gates, and beta = 0 decaying each key row by its own cumulative gate;
* GQA pairing h = hv / (Hv / H) against explicitly repeated key heads;
* split/resume and varlen isolation (bitwise);
* L2-norm prologue against pre-normalised inputs; the default scale.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle
from oracle.chunked import chunked_forward


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = math.sqrt(float((b * b).mean())) if b.size else 1.0
    return float(np.abs(a - b).max() / den) if a.size else 0.0


def rand_case(rng, T, H, Hv, dk, dv, N=1, init=True, lengths=None, unit_keys=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, Hv, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((T, Hv)) + 2.0)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, Hv))))
    if lengths is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    n = len(cu) - 1
    s0 = 0.1 * rng.standard_normal((n, Hv, dv, dk)) if init else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0, cu_seqlens=cu,
                scale=1.0 / math.sqrt(dk))


def run(lib, c, **kw):
    args = dict(c)
    args.update(kw)
    return oracle.recurrent_forward(args["q"], args["k"], args["v"], args["g"], args["beta"],
                                    args.get("scale"), args.get("initial_state"),
                                    args.get("cu_seqlens"),
                                    qk_l2norm=args.get("qk_l2norm", False),
                                    eps=args.get("eps", 1e-6), lib=lib,
                                    out_init=args.get("out_init"))


# ---------------------------------------------------------------- exact rationals
def _exact_lane(q, k, v, alpha, beta, s0, scale):
    """Transition-matrix form in exact rationals: S_t = alpha (I - b k k^T) S + b k v^T."""
    dk, dv = len(k[0]), len(v[0])
    S = [[s0[i][j] for j in range(dv)] for i in range(dk)]
    outs = []
    for t in range(len(k)):
        a, b, kt, vt, qt = alpha[t], beta[t], k[t], v[t], q[t]
        P = [[a * ((1 if i == m else 0) - b * kt[i] * kt[m]) for m in range(dk)] for i in range(dk)]
        S = [[sum(P[i][m] * S[m][j] for m in range(dk)) + b * kt[i] * vt[j] for j in range(dv)]
             for i in range(dk)]
        outs.append([scale * sum(S[i][j] * qt[i] for i in range(dk)) for j in range(dv)])
    return outs, S


def pin_exact_rationals(lib):
    rng = np.random.default_rng(5)
    H, Hv, dk, dv = 1, 2, 4, 3
    lengths = [5, 3]
    T = sum(lengths)
    dy = lambda: Fraction(int(rng.integers(-8, 9)), 8)   # dyadic: exact in fp64
    q = [[[dy() for _ in range(dk)] for _ in range(H)] for _ in range(T)]
    k = [[[dy() for _ in range(dk)] for _ in range(H)] for _ in range(T)]
    v = [[[dy() for _ in range(dv)] for _ in range(Hv)] for _ in range(T)]
    alphas = [Fraction(1, 2), Fraction(3, 4), Fraction(7, 8), Fraction(1, 1), Fraction(5, 8)]
    alpha = [[alphas[int(rng.integers(0, len(alphas)))] for _ in range(Hv)] for _ in range(T)]
    beta = [[Fraction(int(rng.integers(0, 9)), 8) for _ in range(Hv)] for _ in range(T)]
    s0 = [[[[dy() for _ in range(dk)] for _ in range(dv)] for _ in range(Hv)] for _ in lengths]
    scale = Fraction(1, 2)
    f = lambda x: np.array(x, dtype=np.float64)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    out, fin = oracle.recurrent_forward(
        f(q), f(k), f(v), np.log(f(alpha)), f(beta), float(scale), f(s0), cu, lib=lib)
    for n in range(len(lengths)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for hv in range(Hv):
            h = hv // (Hv // H)
            s0_kv = [[s0[n][hv][j][i] for j in range(dv)] for i in range(dk)]
            outs, S = _exact_lane([q[t][h] for t in range(t0, t1)], [k[t][h] for t in range(t0, t1)],
                                  [v[t][hv] for t in range(t0, t1)],
                                  [alpha[t][hv] for t in range(t0, t1)],
                                  [beta[t][hv] for t in range(t0, t1)], s0_kv, scale)
            for t in range(t0, t1):
                for j in range(dv):
                    ex = float(outs[t - t0][j])
                    assert abs(out[t, hv, j] - ex) <= 1e-13 * max(1.0, abs(ex)), (t, hv, j)
            for i in range(dk):
                for j in range(dv):
                    ex = float(S[i][j])
                    assert abs(fin[n, hv, j, i] - ex) <= 1e-13 * max(1.0, abs(ex)), (n, hv, i, j)


# ---------------------------------------------------------------- chunked formulation
def pin_chunked(lib):
    rng = np.random.default_rng(11)
    for T in (1, 63, 64, 65, 200):
        c = rand_case(rng, T, 2, 4, 16, 8)
        o1, f1 = run(lib, c)
        o2, f2 = chunked_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                 c["initial_state"], c["cu_seqlens"])
        assert rel(o1, o2) <= 1e-12 and rel(f1, f2) <= 1e-12, T
    lengths = [70, 1, 64, 129, 3]
    c = rand_case(rng, sum(lengths) + 5, 2, 4, 16, 8, lengths=lengths)
    o1, f1 = run(lib, c)
    o2, f2 = chunked_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                             c["initial_state"], c["cu_seqlens"])
    assert rel(o1, o2) <= 1e-12 and rel(f1, f2) <= 1e-12


# ---------------------------------------------------------------- closed forms
def pin_orthonormal_keys(lib):
    """S_0 = 0 and mutually orthonormal keys: every correction term vanishes."""
    rng = np.random.default_rng(3)
    T, dk, dv = 24, 32, 16
    basis, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = basis[:, :T].T.reshape(T, 1, dk)                  # T orthonormal rows
    c = rand_case(rng, T, 1, 2, dk, dv, init=False)
    c["k"] = k
    out, _ = run(lib, c)
    for hv in range(2):
        G = np.cumsum(c["g"][:, hv])
        D = np.tril(np.exp(G[:, None] - G[None, :]))
        W = (c["q"][:, 0] @ k[:, 0].T) * D * c["beta"][None, :, hv]
        expect = c["scale"] * W @ c["v"][:, hv]
        assert rel(out[:, hv], expect) <= 1e-12, hv


def pin_overwrite(lib):
    """beta = 1, |k_t| = 1, q_t = k_t, scale = 1 => o_t = v_t for any history."""
    rng = np.random.default_rng(4)
    c = rand_case(rng, 40, 2, 4, 16, 8, lengths=[17, 23])
    c["beta"] = np.ones_like(c["beta"])
    c["q"] = c["k"].copy()
    out, _ = run(lib, c, scale=1.0)
    assert np.abs(out - c["v"]).max() <= 1e-12


def pin_beta_zero(lib):
    """beta = 0: the state only decays, S_t = exp(sum_{s<=t} g_s) S_0 (g = 0 gives S_t = S_0)."""
    rng = np.random.default_rng(6)
    lengths = [9, 14]
    c = rand_case(rng, 23, 2, 4, 8, 6, lengths=lengths)
    c["beta"] = np.zeros_like(c["beta"])
    out, fin = run(lib, c)
    cu = c["cu_seqlens"]
    for n in range(2):
        t0, t1 = cu[n], cu[n + 1]
        for hv in range(4):
            h = hv // 2
            cum = np.cumsum(c["g"][t0:t1, hv])
            S0 = c["initial_state"][n, hv]                 # [dv, dk]
            expect = c["scale"] * np.exp(cum)[:, None] * (c["q"][t0:t1, h] @ S0.T)
            assert rel(out[t0:t1, hv], expect) <= 1e-12
            assert rel(fin[n, hv], np.exp(cum[-1]) * S0) <= 1e-12
    c["g"] = np.zeros_like(c["g"])
    out, fin = run(lib, c)
    assert np.array_equal(fin, c["initial_state"])


def pin_gqa_pairing(lib):
    """H key heads serving Hv = HG * H value heads equals repeating each key head HG times."""
    rng = np.random.default_rng(8)
    c = rand_case(rng, 30, 2, 6, 8, 8)
    out, fin = run(lib, c)
    rep = dict(c, q=np.repeat(c["q"], 3, axis=1), k=np.repeat(c["k"], 3, axis=1))
    out2, fin2 = run(lib, rep)
    assert np.array_equal(out, out2) and np.array_equal(fin, fin2)


def pin_split_resume(lib):
    rng = np.random.default_rng(9)
    c = rand_case(rng, 150, 1, 2, 8, 8)
    out, fin = run(lib, c)
    for t1 in (64, 77):
        a = dict(c, cu_seqlens=np.array([0, t1]))
        oa, fa = run(lib, a)
        b = dict(c, cu_seqlens=np.array([t1, 150]), initial_state=fa)
        ob, fb = run(lib, b)
        assert np.array_equal(oa[:t1], out[:t1]) and np.array_equal(ob[t1:], out[t1:])
        assert np.array_equal(fb, fin)


def pin_varlen_isolation(lib):
    rng = np.random.default_rng(10)
    lengths = [5, 0, 70, 33]
    c = rand_case(rng, 120, 2, 4, 8, 8, lengths=lengths)
    canary = np.full((120, 4, 8), 7.25)
    out, fin = run(lib, c, out_init=canary)
    cu = c["cu_seqlens"]
    assert np.array_equal(out[cu[-1]:], canary[cu[-1]:])
    assert np.array_equal(fin[1], c["initial_state"][1])        # empty sequence
    for n in range(len(lengths)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        sub = dict(c, q=c["q"][t0:t1], k=c["k"][t0:t1], v=c["v"][t0:t1], g=c["g"][t0:t1],
                   beta=c["beta"][t0:t1], initial_state=c["initial_state"][n:n + 1],
                   cu_seqlens=np.array([0, t1 - t0]))
        o1, f1 = run(lib, sub)
        assert np.array_equal(o1, out[t0:t1]) and np.array_equal(f1[0], fin[n])


def pin_l2norm_and_scale(lib):
    rng = np.random.default_rng(12)
    c = rand_case(rng, 20, 1, 2, 16, 8, unit_keys=False)
    c["q"] *= 3.0
    c["k"] *= 0.5
    o_on, f_on = run(lib, c, qk_l2norm=True, eps=0.0)
    nq = c["q"] / np.linalg.norm(c["q"], axis=-1, keepdims=True)
    nk = c["k"] / np.linalg.norm(c["k"], axis=-1, keepdims=True)
    o_off, f_off = run(lib, dict(c, q=nq, k=nk))
    assert rel(o_on, o_off) <= 1e-13 and rel(f_on, f_off) <= 1e-13
    o_def, _ = run(lib, dict(c, q=nq, k=nk, scale=None))
    o_nan, _ = run(lib, dict(c, q=nq, k=nk, scale=float("nan")))
    o_exp, _ = run(lib, dict(c, q=nq, k=nk, scale=1.0 / 4.0))
    assert np.array_equal(o_def, o_exp) and np.array_equal(o_nan, o_exp)


# ---------------------------------------------------------------- per-channel gates
def channel_gates(rng, T, Hv, dk):
    """Log-decays per key channel, each channel with its own typical magnitude."""
    mu = rng.uniform(-1.0, 4.0, size=dk)
    return -np.log1p(np.exp(-(rng.standard_normal((T, Hv, dk)) + mu)))


def _exact_lane_channel(q, k, v, alpha, beta, s0, scale):
    """S_t = (I - b k k^T) diag(alpha_t) S + b k v^T in exact rationals."""
    dk, dv = len(k[0]), len(v[0])
    S = [[s0[i][j] for j in range(dv)] for i in range(dk)]
    outs = []
    for t in range(len(k)):
        a, b, kt, vt, qt = alpha[t], beta[t], k[t], v[t], q[t]
        D = [[a[i] * S[i][j] for j in range(dv)] for i in range(dk)]
        S = [[D[i][j] - b * kt[i] * sum(kt[m] * D[m][j] for m in range(dk)) + b * kt[i] * vt[j]
              for j in range(dv)] for i in range(dk)]
        outs.append([scale * sum(S[i][j] * qt[i] for i in range(dk)) for j in range(dv)])
    return outs, S


def pin_channel_exact_rationals(lib):
    rng = np.random.default_rng(15)
    H, Hv, dk, dv = 1, 2, 4, 3
    lengths = [4, 3]
    T = sum(lengths)
    dy = lambda: Fraction(int(rng.integers(-8, 9)), 8)
    q = [[[dy() for _ in range(dk)] for _ in range(H)] for _ in range(T)]
    k = [[[dy() for _ in range(dk)] for _ in range(H)] for _ in range(T)]
    v = [[[dy() for _ in range(dv)] for _ in range(Hv)] for _ in range(T)]
    alphas = [Fraction(1, 4), Fraction(1, 2), Fraction(3, 4), Fraction(7, 8), Fraction(1, 1)]
    alpha = [[[alphas[int(rng.integers(0, len(alphas)))] for _ in range(dk)] for _ in range(Hv)]
             for _ in range(T)]
    beta = [[Fraction(int(rng.integers(0, 9)), 8) for _ in range(Hv)] for _ in range(T)]
    s0 = [[[[dy() for _ in range(dk)] for _ in range(dv)] for _ in range(Hv)] for _ in lengths]
    scale = Fraction(3, 4)
    f = lambda x: np.array(x, dtype=np.float64)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    out, fin = oracle.recurrent_forward(
        f(q), f(k), f(v), np.log(f(alpha)), f(beta), float(scale), f(s0), cu, lib=lib)
    for n in range(len(lengths)):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for hv in range(Hv):
            h = hv // (Hv // H)
            s0_kv = [[s0[n][hv][j][i] for j in range(dv)] for i in range(dk)]
            outs, S = _exact_lane_channel(
                [q[t][h] for t in range(t0, t1)], [k[t][h] for t in range(t0, t1)],
                [v[t][hv] for t in range(t0, t1)], [alpha[t][hv] for t in range(t0, t1)],
                [beta[t][hv] for t in range(t0, t1)], s0_kv, scale)
            for t in range(t0, t1):
                for j in range(dv):
                    ex = float(outs[t - t0][j])
                    assert abs(out[t, hv, j] - ex) <= 1e-13 * max(1.0, abs(ex)), (t, hv, j)
            for i in range(dk):
                for j in range(dv):
                    ex = float(S[i][j])
                    assert abs(fin[n, hv, j, i] - ex) <= 1e-13 * max(1.0, abs(ex)), (n, hv, i, j)


def pin_channel_chunked(lib):
    rng = np.random.default_rng(16)
    for T in (1, 63, 64, 65, 130):
        c = rand_case(rng, T, 2, 4, 16, 8)
        c["g"] = channel_gates(rng, T, 4, 16)
        o1, f1 = run(lib, c)
        o2, f2 = chunked_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                 c["initial_state"], c["cu_seqlens"])
        assert rel(o1, o2) <= 1e-12 and rel(f1, f2) <= 1e-12, T
    lengths = [70, 1, 0, 66]
    c = rand_case(rng, sum(lengths) + 3, 1, 2, 8, 12, lengths=lengths)
    c["g"] = channel_gates(rng, c["q"].shape[0], 2, 8)
    o1, f1 = run(lib, c)
    o2, f2 = chunked_forward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                             c["initial_state"], c["cu_seqlens"])
    assert rel(o1, o2) <= 1e-12 and rel(f1, f2) <= 1e-12


def pin_channel_uniform_is_scalar(lib):
    """The same gate on every key channel is the scalar gate."""
    rng = np.random.default_rng(17)
    c = rand_case(rng, 50, 2, 4, 8, 6, lengths=[20, 30])
    o1, f1 = run(lib, c)
    o2, f2 = run(lib, dict(c, g=np.repeat(c["g"][:, :, None], 8, axis=2)))
    assert rel(o1, o2) <= 1e-13 and rel(f1, f2) <= 1e-13


def pin_channel_beta_zero(lib):
    """beta = 0: key row d of the state decays by exp(sum of its own gates)."""
    rng = np.random.default_rng(18)
    c = rand_case(rng, 21, 1, 2, 8, 5)
    c["beta"] = np.zeros_like(c["beta"])
    c["g"] = channel_gates(rng, 21, 2, 8)
    out, fin = run(lib, c)
    for hv in range(2):
        cum = np.cumsum(c["g"][:, hv], axis=0)              # [T, dk]
        S0 = c["initial_state"][0, hv]                      # [dv, dk]
        expect = c["scale"] * (np.exp(cum) * c["q"][:, 0]) @ S0.T
        assert rel(out[:, hv], expect) <= 1e-12
        assert rel(fin[0, hv], S0 * np.exp(cum[-1])[None, :]) <= 1e-12


ALL_PINS = [pin_exact_rationals, pin_chunked, pin_orthonormal_keys, pin_overwrite,
            pin_beta_zero, pin_gqa_pairing, pin_split_resume, pin_varlen_isolation,
            pin_l2norm_and_scale, pin_channel_exact_rationals, pin_channel_chunked,
            pin_channel_uniform_is_scalar, pin_channel_beta_zero]


# ---------------------------------------------------------------- backward
def _loss_and_grads(lib, c, do, dfin):
    grads = oracle.recurrent_backward(c["q"], c["k"], c["v"], c["g"], c["beta"], c["scale"],
                                      c["initial_state"], c["cu_seqlens"], do, dfin, lib=lib)

    def loss(**over):
        a = dict(c)
        a.update(over)
        out, fin = run(lib, a)
        return float((out * do).sum() + (fin * dfin).sum())

    return grads, loss


def pin_backward_finite_differences(lib):
    """Every gradient entry against a central difference of L = <do, out> + <dfin, final>."""
    rng = np.random.default_rng(21)
    c = rand_case(rng, 9, 1, 2, 3, 2, lengths=[5, 4])
    do = rng.standard_normal(c["v"].shape)
    dfin = rng.standard_normal(c["initial_state"].shape)
    grads, loss = _loss_and_grads(lib, c, do, dfin)
    eps = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("initial_state", "d_initial")):
        base = c[name]
        for idx in np.ndindex(base.shape):
            plus, minus = base.copy(), base.copy()
            plus[idx] += eps
            minus[idx] -= eps
            fd = (loss(**{name: plus}) - loss(**{name: minus})) / (2 * eps)
            got = grads[key][idx]
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx, got, fd)


def _torch_token_loss(q, k, v, g, beta, s0, scale, cu, H, Hv, do, dfin):
    """The token recurrence written as a plain torch loop (for autograd)."""
    import torch
    HG = Hv // H
    loss = torch.zeros((), dtype=torch.float64)
    for n in range(len(cu) - 1):
        for hv in range(Hv):
            h = hv // HG
            S = s0[n, hv].T
            for t in range(int(cu[n]), int(cu[n + 1])):
                a = torch.exp(g[t, hv])
                pred = a * (S.T @ k[t, h])
                S = a * S + beta[t, hv] * torch.outer(k[t, h], v[t, hv] - pred)
                loss = loss + scale * ((S.T @ q[t, h]) * do[t, hv]).sum()
            loss = loss + (S.T * dfin[n, hv]).sum()
    return loss


def pin_backward_autograd(lib):
    """The adjoint against torch autograd of an independently written token loop."""
    import torch
    rng = np.random.default_rng(22)
    c = rand_case(rng, 70, 2, 4, 8, 6, lengths=[66, 0, 4])
    do = rng.standard_normal(c["v"].shape)
    dfin = rng.standard_normal(c["initial_state"].shape)
    grads, _ = _loss_and_grads(lib, c, do, dfin)
    names = ("q", "k", "v", "g", "beta", "initial_state")
    ts = {n: torch.tensor(c[n], dtype=torch.float64, requires_grad=True) for n in names}
    loss = _torch_token_loss(ts["q"], ts["k"], ts["v"], ts["g"], ts["beta"], ts["initial_state"],
                             c["scale"], c["cu_seqlens"], 2, 4, torch.tensor(do),
                             torch.tensor(dfin))
    loss.backward()
    for n, key in zip(names, ("dq", "dk", "dv", "dg", "dbeta", "d_initial")):
        assert rel(grads[key], ts[n].grad.numpy()) <= 1e-12, n


def pin_backward_closed_forms(lib):
    """beta = 0 and g = 0: out = scale S0^T q, so dq = scale S0 do, dS0 = scale sum q do^T
    + dfin, dk = dv = 0; and dbeta = k^T dS (v - S0^T k) at every token."""
    rng = np.random.default_rng(23)
    c = rand_case(rng, 12, 1, 1, 4, 3)
    c["beta"] = np.zeros_like(c["beta"])
    c["g"] = np.zeros_like(c["g"])
    do = rng.standard_normal(c["v"].shape)
    dfin = rng.standard_normal(c["initial_state"].shape)
    grads, _ = _loss_and_grads(lib, c, do, dfin)
    S0 = c["initial_state"][0, 0]          # [dv, dk]
    q, k, v = c["q"][:, 0], c["k"][:, 0], c["v"][:, 0]
    np.testing.assert_allclose(grads["dq"][:, 0], c["scale"] * do[:, 0] @ S0, atol=1e-13)
    assert np.abs(grads["dk"]).max() <= 1e-13 and np.abs(grads["dv"]).max() <= 1e-13
    dS = dfin[0, 0] + c["scale"] * do[:, 0].T @ q          # [dv, dk], constant in t
    np.testing.assert_allclose(grads["d_initial"][0, 0], dS, atol=1e-12)
    # the state never changes, so the gradient into token t's state is the sum of
    # the reads from t onwards plus dfin
    for t in range(12):
        dSt = dfin[0, 0] + c["scale"] * do[t:, 0].T @ q[t:]   # [dv, dk]
        delta = v[t] - S0 @ k[t]
        np.testing.assert_allclose(grads["dbeta"][t, 0], delta @ dSt @ k[t], atol=1e-12)


BACKWARD_PINS = [pin_backward_finite_differences, pin_backward_autograd,
                 pin_backward_closed_forms]
