"""Token-serial kernel (decode / speculative verify) through the C ABI.

Against the fp64 oracle element by element, and against itself: a call over n
tokens must reproduce n one-token calls bit for bit ("Chunking Qwen3.5's gated
DeltaNet for 1.5x faster prefill on Apple Silicon", section "Does the chunked
kernel match the serial one?": verification reproduces decode's numerics).
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs

from gpu_helpers import ratio, run_oracle, to_dev

pytestmark = pytest.mark.gpu

# fp32 arithmetic throughout (inputs are exact on both sides): max|x - ref| / rms(ref).
TOL = 1e-4


def run_rec(x, out_dtype=torch.float32, status=None, **kw):
    d = to_dev(x)
    return B.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                               d.get("initial_state"), d["cu_seqlens"], out_dtype=out_dtype,
                               status=status, **kw)


def check(x, o, f, o_ref, f_ref, tol=TOL):
    cu = x["cu_seqlens"].numpy()
    rows = np.arange(int(cu[0]), int(cu[-1]))
    ro = ratio(o[rows], o_ref[rows]) if rows.size else 0.0
    rf = ratio(f, f_ref)
    assert ro <= tol and rf <= tol, (ro, rf)


@pytest.mark.parametrize("wid", [5, 6])
def test_decode_and_verify_workloads(wid):
    """64 sequences x 1 token (decode) and 8 x 8 tokens (verify), H=16 Hv=32 bf16."""
    x = make_inputs(wid)
    o, f = run_rec(x)
    o_ref, f_ref = run_oracle(x)
    check(x, o, f, o_ref, f_ref)


CASES = [
    dict(T=1), dict(T=4), dict(T=16), dict(T=100),
    dict(lengths=[1, 4, 0, 16, 3], H=2, Hv=4),
    dict(lengths=[7], H=1, Hv=3),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("init", [True, False])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_small_grid(case, init, dtype):
    kw = dict(H=2, Hv=4)
    kw.update(case)
    x = make_inputs(6, seed=91, dtype=dtype, with_initial_state=init, **kw)
    o, f = run_rec(x)
    o_ref, f_ref = run_oracle(x)
    check(x, o, f, o_ref, f_ref)


def test_l2norm_in_kernel():
    """Raw (unnormalised) q, k with the in-kernel L2 norm against the oracle's."""
    x = make_inputs(6, seed=5, H=2, Hv=4, lengths=[3, 9], normalise_qk=False)
    o, f = run_rec(x, use_qk_l2norm=True)
    o_ref, f_ref = run_oracle(x, qk_l2norm=True)
    check(x, o, f, o_ref, f_ref)


def test_verify_equals_decode_steps_bitwise():
    """n tokens in one call == n one-token calls with the state carried along."""
    n_tok = 8
    x = make_inputs(6, seed=3, H=4, Hv=8, lengths=[n_tok])
    d = to_dev(x)
    o_all, f_all = B.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                       d["initial_state"], d["cu_seqlens"],
                                       out_dtype=torch.float32)
    state = d["initial_state"].clone()
    outs = []
    for t in range(n_tok):
        sl = slice(t, t + 1)
        cu1 = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
        o1, state = B.gdn_recurrent_fwd(d["q"][sl].contiguous(), d["k"][sl].contiguous(),
                                        d["v"][sl].contiguous(), d["g"][sl].contiguous(),
                                        d["beta"][sl].contiguous(), x["scale"], state, cu1,
                                        out_dtype=torch.float32)
        outs.append(o1)
    o_steps = torch.cat(outs)
    assert torch.equal(o_all, o_steps)
    assert torch.equal(f_all, state)


def test_bf16_output_is_rounded_fp32_output():
    x = make_inputs(6, seed=8, H=2, Hv=4, lengths=[5, 2])
    o32, _ = run_rec(x, out_dtype=torch.float32)
    o16, _ = run_rec(x, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_final_state_may_alias_initial_state():
    x = make_inputs(6, seed=12, H=2, Hv=4, lengths=[4, 6])
    d = to_dev(x)
    ref_o, ref_f = run_rec(x)
    s = d["initial_state"].clone()
    o, f = B.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], s,
                               d["cu_seqlens"], out_dtype=torch.float32, final_state=s)
    assert f.data_ptr() == s.data_ptr()
    assert torch.equal(o, ref_o) and torch.equal(s, ref_f)


def test_status_word_and_malformed_cu_seqlens():
    """A clean call leaves the status word 0; a decreasing cu_seqlens pair sets
    GDN_DEV_BAD_CU_SEQLENS and that sequence is empty (its state passes through)."""
    x = make_inputs(6, seed=21, H=2, Hv=4, lengths=[3, 4])
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    o, f, desc = run_rec(x, status=status, return_desc=True)
    assert B.gdn_read_status(desc) == 0
    d = to_dev(x)
    bad = torch.tensor([0, 3, 1], dtype=torch.int32, device="cuda")
    o2, f2, desc2 = B.gdn_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                        d["initial_state"], bad, out_dtype=torch.float32,
                                        status=status, return_desc=True)
    assert B.gdn_read_status(desc2) & 1
    assert torch.equal(f2[1], d["initial_state"][1])   # empty sequence: state unchanged
    assert torch.equal(f2[0], f[0])


def test_matches_chunked_path_on_a_prompt():
    """The serial and chunked forwards agree to the bf16 bar on a 200-token prompt."""
    from gpu_helpers import run_gpu, TOL_BF16
    x = make_inputs(2, seed=4, H=2, Hv=4, T=200)
    o_c, f_c = run_gpu(x, out_dtype=torch.float32)
    o_r, f_r = run_rec(x)
    o_ref, f_ref = run_oracle(x)
    assert ratio(o_r, o_ref) <= TOL and ratio(f_r, f_ref) <= TOL
    assert ratio(o_c, o_r.double().cpu().numpy()) <= TOL_BF16
