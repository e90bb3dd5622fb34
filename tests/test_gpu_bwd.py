"""Backward pass (gdn_chunk_bwd) through the C ABI against the oracle's fp64 adjoint
of the token recurrence, gradient by gradient, as max|x - x_ref| / rms(x_ref).

fp32 inputs: the kernels compute in fp32 from the same stored inputs the oracle reads,
so every gradient is held to 2e-4 (fp32 rounding accumulated over the chunk products and
the reverse scan). bf16 inputs: the forward recompute runs on the tensor-core kernels
and the reverse scan reads their bridge (w as one bf16 rounding, M as a bf16 hi/lo pair,
k as fp16), so the gradients carry the forward path's operand precision and are held to
the bf16 bar, 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs

from gpu_helpers import ratio, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-4
TOL_BF16 = 1e-2
KEYS = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")


def upstream(x, seed, out_dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(x["T"], x["Hv"], x["dv"], generator=g, dtype=torch.float64)
    dfin = torch.randn(x["N"], x["Hv"], x["dv"], x["dk"], generator=g, dtype=torch.float64)
    return do.to(out_dtype), dfin.float()


def run_pair(x, do, dfin, **kw):
    d = to_dev(x)
    got = B.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do.cuda(), x["scale"],
                          d.get("initial_state"), d["cu_seqlens"],
                          None if dfin is None else dfin.cuda(), **kw)
    ref = oracle.recurrent_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                    x.get("initial_state"), x["cu_seqlens"], do, dfin)
    ref["d_initial_state"] = ref.pop("d_initial")
    return got, ref


def check(x, got, ref, tol=None):
    tol = tol or (TOL if x["dtype"] == "f32" else TOL_BF16)
    cu = x["cu_seqlens"].numpy()
    rows = np.arange(int(cu[0]), int(cu[-1]))
    for key in KEYS:
        a, r = got[key], ref[key]
        if key != "d_initial_state":
            a, r = a[rows], r[rows]
        e = ratio(a, r)
        print(f"{x['dtype']} d{x['dk']} {key} {e:.2e}")
        assert e <= tol, (key, e)


CASES = [
    dict(T=1), dict(T=63), dict(T=64), dict(T=65), dict(T=200),
    dict(lengths=[5, 0, 70, 33], H=2, Hv=4),
    dict(lengths=[129, 1, 64], H=1, Hv=3),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_small_grid(case, d, dtype):
    kw = dict(H=2, Hv=4)
    kw.update(case)
    x = make_inputs(2, seed=51, dtype=dtype, d=d, with_initial_state=True, **kw)
    do, dfin = upstream(x, 7)
    check(x, *run_pair(x, do, dfin))


def test_no_final_state_gradient_and_zero_initial_state():
    x = make_inputs(8, seed=52, T=150, H=2, Hv=2, with_initial_state=False)
    do, _ = upstream(x, 8)
    got, ref = run_pair(x, do, None)
    check(x, got, ref)


def test_bf16_upstream_gradient():
    x = make_inputs(2, seed=53, T=130, H=2, Hv=4)
    do, dfin = upstream(x, 9, out_dtype=torch.bfloat16)
    check(x, *run_pair(x, do, dfin))


def test_varlen_packed_equals_each_sequence_alone_bitwise():
    x = make_inputs(2, seed=54, lengths=[70, 0, 1, 129], H=2, Hv=4, d=64)
    do, dfin = upstream(x, 10)
    d = to_dev(x)
    full = B.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do.cuda(), x["scale"],
                           d["initial_state"], d["cu_seqlens"], dfin.cuda())
    cu = x["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if a == b:  # an empty sequence passes the final-state gradient through
            assert torch.equal(full["d_initial_state"][n].cpu(), dfin[n])
            continue
        one = B.gdn_chunk_bwd(d["q"][a:b].contiguous(), d["k"][a:b].contiguous(),
                              d["v"][a:b].contiguous(), d["g"][a:b].contiguous(),
                              d["beta"][a:b].contiguous(), do[a:b].contiguous().cuda(),
                              x["scale"], d["initial_state"][n:n + 1].contiguous(),
                              torch.tensor([0, b - a], dtype=torch.int32, device="cuda"),
                              dfin[n:n + 1].contiguous().cuda())
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(one[key], full[key][a:b]), (n, key)
        assert torch.equal(one["d_initial_state"][0], full["d_initial_state"][n])


def test_gradients_match_finite_differences_of_the_forward():
    """The GPU backward against central differences of the GPU forward (fp32 inputs,
    loss <do, out> + <dfin, final>), for a few entries of every input."""
    x = make_inputs(8, seed=55, T=70, H=1, Hv=1, dtype="f32", with_initial_state=True)
    do, dfin = upstream(x, 11)
    d = to_dev(x)
    got = B.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do.cuda(), x["scale"],
                          d["initial_state"], d["cu_seqlens"], dfin.cuda())

    def loss(**over):
        a = dict(d)
        a.update(over)
        o, f = B.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], x["scale"],
                               a["initial_state"], a["cu_seqlens"], out_dtype=torch.float32)
        return float((o.double().cpu() * do.double()).sum() + (f.double().cpu() * dfin.double()).sum())

    rng = np.random.default_rng(0)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                      ("initial_state", "d_initial_state")):
        base = d[name]
        for _ in range(3):
            idx = tuple(int(rng.integers(0, s)) for s in base.shape)
            eps = 1e-2 * max(1.0, abs(float(base[idx])))
            plus, minus = base.clone(), base.clone()
            plus[idx] += eps
            minus[idx] -= eps
            fd = (loss(**{name: plus}) - loss(**{name: minus})) / (2 * eps)
            g = float(got[key][idx])
            assert abs(g - fd) <= 2e-2 * max(1.0, abs(fd)), (name, idx, g, fd)


@pytest.mark.parametrize("wid", [2, 8])
def test_full_size(wid):
    """T = 4096, H = 16, Hv = 32 (d = 128 and d = 64), every element against the oracle."""
    x = make_inputs(wid)
    do, dfin = upstream(x, 12)
    check(x, *run_pair(x, do, dfin))


def test_rejects_per_channel_gates_and_l2norm():
    x = make_inputs(9, seed=56, T=64, H=1, Hv=1)
    d = to_dev(x)
    do = torch.zeros(64, 1, 128, device="cuda")
    with pytest.raises(B.GdnError):
        B.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], do, x["scale"],
                        d["initial_state"], d["cu_seqlens"])
