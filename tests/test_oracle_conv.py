"""Pins of the front-end oracle (no GPU): closed forms, a hand-worked example and
properties any correct causal convolution with a carried state must have."""
import numpy as np
import pytest

from oracle.conv_front import conv_front, silu

H, HV, DK = 1, 1, 4   # small heads: C = 2*1*4 + 1*4 = 12 channels


def rand(rng, T, d, n_state=1):
    C = 2 * H * DK + HV * DK
    return (rng.standard_normal((T, C)), rng.standard_normal((C, d)),
            rng.standard_normal((n_state, C, d - 1)))


def run(x, w, s=None, cu=None, **kw):
    return conv_front(x, w, H, HV, DK, DK, conv_state=s, cu_seqlens=cu, **kw)


def cat(q, k, v):
    T = q.shape[0]
    return np.concatenate([q.reshape(T, H * DK), k.reshape(T, H * DK), v.reshape(T, HV * DK)],
                          axis=1)


def test_silu_identities():
    x = np.linspace(-30, 30, 121)
    assert silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(silu(x) - silu(-x), x, atol=1e-12)   # x s(x) + x s(-x) = x
    np.testing.assert_allclose(silu(np.array([40.0])), [40.0], rtol=1e-15)


def test_hand_worked_example():
    """d_conv = 2, one channel of interest: w = [0.5, 2], state 4, x = [1, 3]:
    y0 = SiLU(0.5*4 + 2*1) = SiLU(4), y1 = SiLU(0.5*1 + 2*3) = SiLU(6.5); new state 3."""
    C = 2 * H * DK + HV * DK
    x = np.zeros((2, C)); x[:, 0] = [1.0, 3.0]
    w = np.zeros((C, 2)); w[0] = [0.5, 2.0]
    s = np.zeros((1, C, 1)); s[0, 0, 0] = 4.0
    q, k, v, s1, _ = run(x, w, s)
    y = cat(q, k, v)
    np.testing.assert_allclose(y[:, 0], [4.0 / (1 + np.exp(-4.0)), 6.5 / (1 + np.exp(-6.5))],
                               rtol=1e-15)
    assert s1[0, 0, 0] == 3.0


def test_width_one_is_elementwise():
    rng = np.random.default_rng(1)
    x, w, _ = rand(rng, 7, 1)
    q, k, v, s1, _ = run(x, w)
    np.testing.assert_allclose(cat(q, k, v), silu(x * w[:, 0]), rtol=1e-14)
    assert s1.shape[-1] == 0


@pytest.mark.parametrize("d", [2, 3, 4, 5])
def test_impulse_response_reads_weights_backwards(d):
    """A unit input at t0 (zero state) gives y[t0 + m] = SiLU(w[d-1-m]) for m < d and
    SiLU(0) = 0 elsewhere: pins the tap order and the causal offset."""
    rng = np.random.default_rng(d)
    _, w, _ = rand(rng, 1, d)
    C = w.shape[0]
    T, t0 = 12, 4
    x = np.zeros((T, C)); x[t0] = 1.0
    y = cat(*run(x, w)[:3])
    for t in range(T):
        m = t - t0
        expect = silu(w[:, d - 1 - m]) if 0 <= m < d else np.zeros(C)
        np.testing.assert_allclose(y[t], expect, rtol=1e-14, atol=0)


@pytest.mark.parametrize("d", [2, 4, 5])
def test_state_carries_across_calls(d):
    """One call over T rows == calls over pieces with the state carried (pieces
    shorter than d - 1 included): pins the state window."""
    rng = np.random.default_rng(10 + d)
    x, w, s = rand(rng, 23, d)
    q, k, v, s_end, _ = run(x, w, s)
    ys, st = [], s
    for a, b in [(0, 1), (1, 3), (3, 10), (10, 11), (11, 23)]:
        qq, kk, vv, st, _ = run(x[a:b], w, st)
        ys.append(cat(qq, kk, vv))
    np.testing.assert_allclose(np.concatenate(ys), cat(q, k, v), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st, s_end, rtol=0, atol=0)


def test_varlen_sequences_are_independent():
    rng = np.random.default_rng(3)
    d = 4
    C = 2 * H * DK + HV * DK
    x = rng.standard_normal((17, C))
    w = rng.standard_normal((C, d))
    s = rng.standard_normal((3, C, d - 1))
    cu = [0, 5, 5, 17]
    q, k, v, s1, _ = run(x, w, s, cu)
    y = cat(q, k, v)
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        qq, kk, vv, sn, _ = run(x[a:b], w, s[n:n + 1])
        np.testing.assert_allclose(y[a:b], cat(qq, kk, vv), rtol=0, atol=0)
        np.testing.assert_allclose(s1[n], sn[0], rtol=0, atol=0)
    np.testing.assert_array_equal(s1[1], s[1])   # empty sequence keeps its state


def test_snapshots_are_prefix_states():
    rng = np.random.default_rng(4)
    d = 4
    x, w, s = rand(rng, 6, d)
    *_, snaps = run(x, w, s, n_snapshots=8)
    for i in range(8):
        n_tok = min(i + 1, 6)
        *_, s_pref, _ = run(x[:n_tok], w, s)
        np.testing.assert_array_equal(snaps[0, i], s_pref[0])


def test_l2norm_gives_unit_heads():
    rng = np.random.default_rng(5)
    x, w, s = rand(rng, 9, 4)
    q, k, v, _, _ = run(x, w, s, l2norm=True, eps=0.0)
    q0, k0, v0, _, _ = run(x, w, s)
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(k, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(q, q0 / np.linalg.norm(q0, axis=-1, keepdims=True), rtol=1e-13)
    np.testing.assert_array_equal(v, v0)
