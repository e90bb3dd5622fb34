"""Head size 64, per-channel gates and fp32 inputs (the fp32 SIMT kernels; bf16 inputs
on the tensor-core kernels, per-channel gates through their own intra kernel) through
the C ABI against the CPU oracle, element by element.

Tolerances are those of the tensor-core path: max|x - x_ref| / rms(x_ref) <= 1e-4
for fp32 inputs and <= 1e-2 for bf16 inputs (fp32 output store, fp32 state)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs

from gpu_helpers import TOL_F32, ratio, run_gpu, run_oracle, to_dev, tol_for, valid_rows

pytestmark = pytest.mark.gpu

# (head size, per-channel gates) of the SIMT path; bf16 d=128 scalar is the tensor-core path
KINDS = [(64, False), (64, True), (128, True)]


def kind_id(k):
    return f"d{k[0]}-{'channel' if k[1] else 'scalar'}"


def check(x, o, f, o_ref, f_ref, tol=None):
    tol = tol or tol_for(x)
    rows = valid_rows(x)
    ro = ratio(o[rows], o_ref[rows])
    rf = ratio(f, f_ref) if f_ref is not None else 0.0
    assert ro <= tol and rf <= tol, (ro, rf, tol)


CASES = [
    dict(T=1), dict(T=63), dict(T=65), dict(T=200),
    dict(lengths=[5, 0, 70, 33], H=2, Hv=4),
    dict(lengths=[129, 1, 64], H=1, Hv=3),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kind", KINDS, ids=kind_id)
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_small_grid(case, kind, dtype):
    d, chan = kind
    kw = dict(H=2, Hv=4)
    kw.update(case)
    x = make_inputs(9, seed=31, dtype=dtype, d=d, channel_gates=chan, **kw)
    o, f = run_gpu(x)
    check(x, o, f, *run_oracle(x))


def test_fp32_d128_scalar_gates():
    """fp32 inputs with d = 128 and scalar gates also run on these kernels."""
    x = make_inputs(0, seed=5, T=190, H=2, Hv=4, with_initial_state=True)
    o, f = run_gpu(x)
    check(x, o, f, *run_oracle(x), TOL_F32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("offsets", [(-6.0, 4.0), (-40.0, -20.0)])
@pytest.mark.parametrize("d", [64, 128])
def test_channel_gates_wide_range(d, offsets, dtype):
    """Channels whose decays differ by orders of magnitude, down to gates near -40 per
    token (exp(G) underflows inside a chunk; on the bf16 path the 16-row diagonal blocks
    then exceed the middle reference's range and are formed entry by entry): the result
    stays finite and within tolerance."""
    x = make_inputs(9, seed=41, T=150, H=1, Hv=2, dtype=dtype, d=d, channel_gates=True,
                    gate_offsets=offsets)
    o, f = run_gpu(x)
    assert torch.isfinite(o).all() and torch.isfinite(f).all()
    check(x, o, f, *run_oracle(x))


def test_uniform_channel_gates_match_scalar_gates():
    x = make_inputs(8, seed=12, T=140, H=2, Hv=4, dtype="f32")
    xc = dict(x, g=x["g"][:, :, None].expand(-1, -1, x["dk"]).contiguous())
    o1, f1 = run_gpu(x)
    o2, f2 = run_gpu(xc)
    assert ratio(o2, o1.cpu().double().numpy()) <= 1e-5
    assert ratio(f2, f1.cpu().double().numpy()) <= 1e-5


@pytest.mark.parametrize("kind", KINDS, ids=kind_id)
def test_varlen_packed_equals_each_sequence_alone_bitwise(kind):
    d, chan = kind
    x = make_inputs(9, seed=13, lengths=[70, 0, 1, 129], H=2, Hv=4, d=d, channel_gates=chan)
    o, f = run_gpu(x)
    cu = x["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if a == b:
            assert torch.equal(f[n].cpu(), x["initial_state"][n])
            continue
        sub = dict(x, q=x["q"][a:b], k=x["k"][a:b], v=x["v"][a:b], g=x["g"][a:b],
                   beta=x["beta"][a:b], initial_state=x["initial_state"][n:n + 1],
                   cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32))
        o1, f1 = run_gpu(sub)
        assert torch.equal(o1, o[a:b]) and torch.equal(f1[0], f[n])


@pytest.mark.parametrize("kind", KINDS, ids=kind_id)
def test_rows_outside_sequences_untouched(kind):
    d, chan = kind
    x = make_inputs(9, seed=14, lengths=[30, 45], T=90, H=1, Hv=2, d=d, channel_gates=chan)
    canary = torch.full((90, 2, d), 3.5, dtype=torch.float32, device="cuda")
    o, _ = run_gpu(x, out=canary)
    assert torch.all(o[75:] == 3.5)


@pytest.mark.parametrize("kind", KINDS, ids=kind_id)
def test_split_and_resume(kind):
    d, chan = kind
    x = make_inputs(9, seed=15, T=230, H=2, Hv=2, d=d, channel_gates=chan, dtype="f32")
    o, f = run_gpu(x)
    a = dict(x, cu_seqlens=torch.tensor([0, 100], dtype=torch.int32))
    _, fa = run_gpu(a)
    b = dict(x, cu_seqlens=torch.tensor([100, 230], dtype=torch.int32),
             initial_state=fa.cpu())
    ob, fb = run_gpu(b)
    assert ratio(ob[100:], o[100:].cpu().double().numpy()) <= TOL_F32
    assert ratio(fb, f.cpu().double().numpy()) <= TOL_F32


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_qk_l2norm_prologue_d64(dtype):
    x = make_inputs(8, seed=16, T=100, H=2, Hv=4, dtype=dtype, normalise_qk=False)
    o, f = run_gpu(x, use_qk_l2norm=True)
    check(x, o, f, *run_oracle(x, qk_l2norm=True))


def test_bf16_output_is_rounded_fp32_output():
    x = make_inputs(9, seed=17, T=150, H=2, Hv=4)
    o32, _ = run_gpu(x, out_dtype=torch.float32)
    o16, _ = run_gpu(x, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_cuda_graph_replay_bitwise():
    x = make_inputs(9, seed=18, lengths=[90, 40], H=2, Hv=4, d=64, channel_gates=True)
    d = to_dev(x)
    out = torch.empty(x["T"], 4, 64, dtype=torch.float32, device="cuda")
    fin = torch.empty(2, 4, 64, 64, dtype=torch.float32, device="cuda")
    desc = B.make_desc(x["T"], 2, 2, 4, torch.bfloat16, torch.float32, dk=64, dv=64,
                       flags=B.GDN_FLAG_CHANNEL_GATES)
    ws = B.alloc_workspace(desc, "cuda")

    def call():
        B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                        d["initial_state"], d["cu_seqlens"], out=out, final_state=fin,
                        workspace=ws)

    call()
    torch.cuda.synchronize()
    eager_o, eager_f = out.clone(), fin.clone()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    fin.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager_o) and torch.equal(fin, eager_f)


@pytest.mark.parametrize("wid", [8, 9])
def test_full_size_workloads(wid):
    """The two benchmark workloads at full size (T = 4096, H = 16, Hv = 32), every
    element against the oracle."""
    x = make_inputs(wid)
    o, f = run_gpu(x)
    check(x, o, f, *run_oracle(x))



@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_channel_gates_with_qk_l2norm(d, dtype):
    """Per-channel gates with the q/k L2 norm on (the row factors enter the decayed q and
    k operands of the per-channel kernels)."""
    x = make_inputs(9, seed=57, lengths=[70, 1, 58], H=2, Hv=4, d=d, dtype=dtype,
                    channel_gates=True, normalise_qk=False)
    o, f = run_gpu(x, use_qk_l2norm=True)
    check(x, o, f, *run_oracle(x, qk_l2norm=True))
