"""Front end (causal conv + SiLU + q/k L2 norm) through the C ABI against the fp64
oracle. Outputs are compared per element within one rounding of the output type
(bf16: 2^-8 relative; fp32: 1e-5 relative, the fp32 tap sum and exp), conv states
and snapshots bit for bit (they are copies of inputs)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_conv_inputs
from oracle.conv_front import conv_front

pytestmark = pytest.mark.gpu


def run_pair(c, l2norm=False, n_snapshots=0, **kw):
    dev = {k: (c[k].cuda() if c.get(k) is not None else None) for k in ("x", "w", "state", "cu_seqlens")}
    q, k, v, s1, sn = B.gdn_conv_front(dev["x"], dev["w"], c["H"], c["Hv"], dev["state"],
                                       dev["cu_seqlens"], use_qk_l2norm=l2norm,
                                       n_snapshots=n_snapshots, **kw)
    ref = conv_front(c["x"], c["w"], c["H"], c["Hv"], conv_state=c["state"],
                     cu_seqlens=c["cu_seqlens"], l2norm=l2norm, n_snapshots=n_snapshots)
    return (q, k, v, s1, sn), ref


def close(a, ref, dtype, rows):
    a = a.double().cpu().numpy()[rows]
    ref = np.asarray(ref)[rows]
    rel = 2.0 ** -8 if dtype == "bf16" else 1e-5
    err = np.abs(a - ref) - (rel * np.abs(ref) + 1e-6)
    assert err.max() <= 0, float(np.abs(a - ref).max())


def check(c, got, ref):
    cu = c["cu_seqlens"].numpy()
    rows = np.arange(int(cu[0]), int(cu[-1]))
    for g, r in zip(got[:3], ref[:3]):
        close(g, r, c["dtype"], rows)
    if got[3] is not None:
        np.testing.assert_array_equal(got[3].cpu().numpy(), ref[3].astype(np.float32))
    if got[4] is not None:
        np.testing.assert_array_equal(got[4].cpu().numpy(), ref[4].astype(np.float32))


def test_qwen_shape_prefill():
    """T=4096, H=16, Hv=32 (C=8192), d_conv=4, bf16, one sequence with a conv state."""
    c = make_conv_inputs(seed=1, T=4096, H=16, Hv=32, d_conv=4)
    got, ref = run_pair(c)
    check(c, got, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d_conv", [1, 2, 3, 4, 5, 8])
def test_widths_and_dtypes(d_conv, dtype):
    c = make_conv_inputs(seed=10 + d_conv, T=70, H=2, Hv=4, d_conv=d_conv, dtype=dtype,
                         lengths=[1, 33, 0, 36])
    got, ref = run_pair(c, n_snapshots=3 if d_conv > 1 else 0)
    check(c, got, ref)


def test_l2norm_and_no_state():
    c = make_conv_inputs(seed=4, T=50, H=2, Hv=2, d_conv=4, with_state=False, lengths=[20, 30])
    got, ref = run_pair(c, l2norm=True)
    check(c, got, ref)


def test_rows_outside_sequences_are_untouched():
    """cu_seqlens starting at row 3 and ending before the last rows: those rows keep
    whatever the output buffers held."""
    c = make_conv_inputs(seed=6, H=1, Hv=1, d_conv=4, lengths=[9, 5], rows=20, cu_offset=3)
    T = c["T"]
    canary = torch.full((T, 1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    q, k, v = canary.clone(), canary.clone(), canary.clone()
    got, ref = run_pair(c, q=q, k=k, v=v)
    check(c, got, ref)
    for t in list(range(3)) + list(range(17, 20)):
        assert torch.all(q[t] == 7.0) and torch.all(k[t] == 7.0) and torch.all(v[t] == 7.0)


def test_state_carries_across_calls_bitwise():
    """One call over 40 rows == calls over 7 + 33 rows with the state passed along."""
    c = make_conv_inputs(seed=8, T=40, H=2, Hv=2, d_conv=4)
    d = {k: c[k].cuda() for k in ("x", "w", "state")}
    q, k, v, s_all, _ = B.gdn_conv_front(d["x"], d["w"], 2, 2, d["state"])
    q1, k1, v1, s1, _ = B.gdn_conv_front(d["x"][:7].contiguous(), d["w"], 2, 2, d["state"])
    q2, k2, v2, s2, _ = B.gdn_conv_front(d["x"][7:].contiguous(), d["w"], 2, 2, s1)
    assert torch.equal(torch.cat([q1, q2]), q) and torch.equal(torch.cat([v1, v2]), v)
    assert torch.equal(s2, s_all)


def test_state_out_may_alias_state_in():
    c = make_conv_inputs(seed=9, T=30, H=2, Hv=2, d_conv=4, lengths=[2, 28])
    d = {k: c[k].cuda() for k in ("x", "w", "state", "cu_seqlens")}
    ref = B.gdn_conv_front(d["x"], d["w"], 2, 2, d["state"].clone(), d["cu_seqlens"])
    s = d["state"].clone()
    got = B.gdn_conv_front(d["x"], d["w"], 2, 2, s, d["cu_seqlens"], conv_state_out=s)
    for a, b in zip(got[:4], ref[:4]):
        assert torch.equal(a, b)


def test_status_word_for_malformed_cu_seqlens():
    c = make_conv_inputs(seed=2, T=16, H=1, Hv=1, d_conv=3, lengths=[6, 10])
    d = {k: c[k].cuda() for k in ("x", "w", "state")}
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    *_, desc = B.gdn_conv_front(d["x"], d["w"], 1, 1, d["state"],
                                c["cu_seqlens"].cuda(), status=status, return_desc=True)
    assert B.gdn_read_status(desc) == 0
    bad = torch.tensor([0, 9, 4], dtype=torch.int32, device="cuda")
    *_, desc = B.gdn_conv_front(d["x"], d["w"], 1, 1, d["state"], bad, status=status,
                                return_desc=True)
    assert B.gdn_read_status(desc) & 1
