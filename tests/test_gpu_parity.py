"""CUDA path (through the C ABI) against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs
from oracle.chunk_table import build_chunk_table, nt_max_bound

from gpu_helpers import TOL_BF16, TOL_F32, ratio, run_gpu, run_oracle, to_dev, tol_for, valid_rows

pytestmark = pytest.mark.gpu


def check_parity(x, o, f, o_ref, f_ref, tol=None):
    tol = tol or tol_for(x)
    rows = valid_rows(x)
    ro = ratio(o[rows], o_ref[rows])
    rf = ratio(f, f_ref) if f_ref is not None else 0.0
    assert ro <= tol and rf <= tol, (ro, rf, tol)
    return ro, rf


def test_tiny_fp32_single_sequence():
    """T=128 (two chunks), H=Hv=2, fp32 inputs: 1e-4."""
    x = make_inputs(0)
    o, f = run_gpu(x, out_dtype=torch.float32)
    o_ref, f_ref = run_oracle(x)
    check_parity(x, o, f, o_ref, f_ref, TOL_F32)


SMALL = [
    dict(T=1), dict(T=63), dict(T=64), dict(T=65), dict(T=200),
    dict(lengths=[5, 0, 70, 33], H=2, Hv=4),
    dict(lengths=[129, 1, 64], H=1, Hv=3),
    dict(lengths=[0, 0, 3], H=2, Hv=2),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_small_grid(case, dtype):
    kw = dict(H=2, Hv=4)
    kw.update(case)
    x = make_inputs(2, seed=77, dtype=dtype, **kw)
    o, f = run_gpu(x, out_dtype=torch.float32)
    o_ref, f_ref = run_oracle(x)
    check_parity(x, o, f, o_ref, f_ref)


@pytest.mark.parametrize("wid", [1, 2, 3, 4])
def test_full_size_workloads(wid):
    """Full-size Qwen3.5-shaped workloads against the oracle (every output element)."""
    x = make_inputs(wid)
    o, f = run_gpu(x, out_dtype=torch.float32)
    o_ref, f_ref = run_oracle(x)
    if wid in (3, 4):  # per-sequence ratios
        cu = x["cu_seqlens"].numpy()
        for n in range(len(cu) - 1):
            a, b = int(cu[n]), int(cu[n + 1])
            if b > a:
                assert ratio(o[a:b], o_ref[a:b]) <= TOL_BF16, n
            if x["initial_state"] is not None or b > a:
                assert ratio(f[n], f_ref[n]) <= TOL_BF16, n
    else:
        check_parity(x, o, f, o_ref, f_ref, TOL_BF16)


def test_bf16_output_is_rounded_fp32_output():
    """The bf16 output is the RNE rounding of the fp32 output of the same kernels."""
    x = make_inputs(2, seed=5, T=300, H=2, Hv=4)
    o32, _ = run_gpu(x, out_dtype=torch.float32)
    o16, _ = run_gpu(x, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_bf16_output_is_rounded_fp32_output_full_size():
    """Same at the benchmarked shape (T=4096, H=16, Hv=32): the bf16 store the benchmark
    times is the RNE rounding of the parity-tested fp32 output, bit for bit."""
    x = make_inputs(2)
    o32, f32 = run_gpu(x, out_dtype=torch.float32)
    o16, f16 = run_gpu(x, out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(f16, f32)


def test_decreasing_cu_seqlens_run_as_their_prefix_maximum():
    """A malformed cu_seqlens is sanitized to its running maximum (clamped to [0, T]):
    [0, 100, 50, 200] runs exactly as [0, 100, 100, 200] (the middle sequence empty, no
    two sequences overlapping), with status bit 1 and no fault."""
    x = make_inputs(2, seed=3, T=256, H=2, Hv=4)
    d = to_dev(x)
    s0 = torch.randn(3, 4, 128, 128, device="cuda") * 0.02
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], s0)
    bad = torch.tensor([0, 100, 50, 200], dtype=torch.int32, device="cuda")
    good = torch.tensor([0, 100, 100, 200], dtype=torch.int32, device="cuda")
    out_b = torch.full((256, 4, 128), 7.0, device="cuda")
    out_g = out_b.clone()
    o, f, desc, _ = B.gdn_chunk_fwd(*args, bad, out=out_b, out_dtype=torch.float32,
                                    return_desc=True)
    assert B.gdn_read_status(desc) == 1
    o2, f2, desc2, _ = B.gdn_chunk_fwd(*args, good, out=out_g, out_dtype=torch.float32,
                                       return_desc=True)
    assert B.gdn_read_status(desc2) == 0
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(f, f2)
    assert torch.equal(f[1], s0[1])                     # the empty sequence passes its state
    assert bool((o[200:] == 7.0).all())                 # rows past the last sequence untouched


def test_nonfinite_status_bit_for_fp16_range():
    """Values whose decayed correction exceeds the fp16 range of the tensor-core path's state
    update (|v| ~ 1e6 here) make the state non-finite: the call completes, no fault, and the
    status word carries GDN_DEV_NONFINITE (16); the same call on in-range values is clean."""
    x = make_inputs(2, seed=9, T=200, H=2, Hv=4)
    run_gpu(x, out_dtype=torch.float32)                 # asserts a clean status word
    x["v"] = (x["v"].float() * 1e6).to(torch.bfloat16)
    d = to_dev(x)
    o, f, desc, _ = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                    d["initial_state"], d["cu_seqlens"],
                                    out_dtype=torch.float32, return_desc=True)
    assert B.gdn_read_status(desc) & 16


@pytest.mark.parametrize("wid", [3, 4])
def test_chunk_table_bit_exact(wid):
    x = make_inputs(wid)
    d = to_dev(x)
    table, offs = B.gdn_build_chunk_indices(d["cu_seqlens"], x["T"], x["nt_max"])
    ref_t, ref_o, total = build_chunk_table(x["cu_seqlens"].tolist(), x["nt_max"])
    assert table.cpu().tolist() == ref_t
    assert offs.cpu().tolist() == ref_o


def test_chunk_table_bound_tight():
    lengths = [1] * 31 + [4096 - 31]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    nt = nt_max_bound(4096, 32)
    table, offs = B.gdn_build_chunk_indices(cu.cuda(), 4096, nt)
    ref_t, ref_o, total = build_chunk_table(cu.tolist(), nt)
    assert total == nt == 95
    assert table.cpu().tolist() == ref_t and offs.cpu().tolist() == ref_o


def test_padding_rows_and_states_untouched():
    """Static-bound workload: rows past the last sequence keep their canary bits,
    zero-length padded sequences return their initial state."""
    x = make_inputs(4)
    d = to_dev(x)
    canary = torch.full((x["T"], x["Hv"], 128), float("nan"), device="cuda")
    out = canary.clone()
    o, f = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                           d["initial_state"], d["cu_seqlens"], out=out)
    torch.cuda.synchronize()
    end = int(x["cu_seqlens"][-1])
    assert torch.isnan(o[end:]).all() and not torch.isnan(o[:end]).any()
    n_real = len(x["lengths"])
    assert torch.equal(f[n_real:], d["initial_state"][n_real:])


def test_padded_vs_unpadded_cu_seqlens_bitwise():
    x = make_inputs(4)
    n_real = len(x["lengths"])
    xu = dict(x, cu_seqlens=x["cu_seqlens"][: n_real + 1].clone(),
              initial_state=x["initial_state"][:n_real].clone(), nt_max=0)
    o1, f1 = run_gpu(x)
    o2, f2 = run_gpu(xu)
    end = int(x["cu_seqlens"][-1])
    assert torch.equal(o1[:end], o2[:end]) and torch.equal(f1[:n_real], f2)


def test_varlen_packed_equals_each_sequence_alone_bitwise():
    x = make_inputs(3)
    o, f = run_gpu(x)
    cu = x["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        xs = dict(x, q=x["q"][a:b], k=x["k"][a:b], v=x["v"][a:b], g=x["g"][a:b],
                  beta=x["beta"][a:b], initial_state=x["initial_state"][n:n + 1],
                  cu_seqlens=torch.tensor([0, b - a], dtype=torch.int32))
        os_, fs = run_gpu(xs)
        assert torch.equal(os_, o[a:b]) and torch.equal(fs[0], f[n]), n


@pytest.mark.parametrize("split", [1024, 1000])
def test_split_and_resume(split):
    x = make_inputs(2, seed=3, T=2048, H=2, Hv=4)
    o, f = run_gpu(x)
    a = dict(x, cu_seqlens=torch.tensor([0, split], dtype=torch.int32))
    oa, fa = run_gpu(a)
    b = dict(x, cu_seqlens=torch.tensor([split, 2048], dtype=torch.int32), initial_state=fa.cpu())
    ob, fb = run_gpu(b)
    if split % 64 == 0:  # same chunk boundaries: the same arithmetic
        assert torch.equal(oa[:split], o[:split]) and torch.equal(ob[split:], o[split:])
        assert torch.equal(fb, f)
    else:
        o_ref, f_ref = run_oracle(x)
        assert ratio(torch.cat([oa[:split], ob[split:]]), o_ref) <= TOL_BF16
        assert ratio(fb, f_ref) <= TOL_BF16


def test_final_state_may_alias_initial_state():
    x = make_inputs(2, seed=9, T=300, H=2, Hv=4)
    o1, f1 = run_gpu(x)
    d = to_dev(x)
    st = d["initial_state"].clone()
    o2, f2 = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], st,
                             d["cu_seqlens"], out_dtype=torch.float32, final_state=st)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, st)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_qk_l2norm_prologue(dtype):
    x = make_inputs(2, seed=13, T=333, H=2, Hv=4, dtype=dtype, normalise_qk=False)
    o, f = run_gpu(x, use_qk_l2norm=True)
    o_ref, f_ref = run_oracle(x, qk_l2norm=True, eps=1e-6)
    check_parity(x, o, f, o_ref, f_ref)


def test_caller_chunk_table_read_and_build():
    x = make_inputs(3)
    d = to_dev(x)
    o1, f1 = run_gpu(x)
    ref_t, _, _ = build_chunk_table(x["cu_seqlens"].tolist(), x["nt_max"])
    table = torch.tensor(ref_t, dtype=torch.int32, device="cuda")
    o2, f2 = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                             d["initial_state"], d["cu_seqlens"], chunk_indices=table,
                             out_dtype=torch.float32)
    built = torch.full_like(table, 12345)
    o3, f3 = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                             d["initial_state"], d["cu_seqlens"], chunk_indices=built,
                             build_chunk_indices=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    assert torch.equal(o1, o3) and torch.equal(f1, f3)
    assert built.cpu().tolist() == ref_t


def test_one_sequence_tiles_requested_before_the_table():
    """One sequence whose table the call builds: the intra kernel maps slot s to chunk s
    and requests the tiles before the chunk table is written. A caller table (read, not
    built) takes the ordinary path; both give the same bits, for a start inside a chunk.
    Reversed boundaries give no rows: the status reports them, no output row is written
    and the final state is the initial one."""
    x = make_inputs(2, seed=17, T=500, H=2, Hv=4)
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], d["initial_state"])
    cu = [37, 470]
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o1, f1 = B.gdn_chunk_fwd(*args, cu_d, out_dtype=torch.float32)
    ref_t, _, _ = build_chunk_table(cu, x["nt_max"])
    table = torch.tensor(ref_t, dtype=torch.int32, device="cuda")
    o2, f2 = B.gdn_chunk_fwd(*args, cu_d, chunk_indices=table, out_dtype=torch.float32)
    built = torch.full_like(table, 12345)  # built into the caller's buffer: the early path
    o3, f3 = B.gdn_chunk_fwd(*args, cu_d, chunk_indices=built, build_chunk_indices=True,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o1[37:470], o2[37:470]) and torch.equal(f1, f2)
    assert torch.equal(o1[37:470], o3[37:470]) and torch.equal(f1, f3)
    assert built.cpu().tolist() == ref_t
    o_ref, f_ref = run_oracle(dict(x, cu_seqlens=torch.tensor(cu, dtype=torch.int32)))
    assert ratio(o1[37:470], o_ref[37:470]) <= TOL_BF16 and ratio(f1, f_ref) <= TOL_BF16
    out = torch.full((x["T"], x["Hv"], 128), 7.0, device="cuda")
    fin = torch.full_like(d["initial_state"], 3.0)
    rev = torch.tensor([300, 100], dtype=torch.int32, device="cuda")
    _, _, desc, _ = B.gdn_chunk_fwd(*args, rev, out=out, final_state=fin, return_desc=True)
    assert B.gdn_read_status(desc) & 1
    assert bool(torch.all(out == 7.0)) and torch.equal(fin, d["initial_state"])


@pytest.mark.parametrize("H,Hv,T", [(8, 16, 2600), (4, 16, 5000), (2, 16, 9800)])
def test_last_wave_split_by_value_heads(H, Hv, T):
    """Shapes whose intra grid (key heads x chunk slots, two CTAs per SM) ends in a partial
    wave, for 2, 4 and 8 value heads per key head: the slots of that wave are taken by two
    CTAs each, one per half of the value heads. Every head still matches the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x = make_inputs(2, seed=5, H=H, Hv=Hv, T=T)
    items, places = H * x["nt_max"], 2 * sms
    if not (items > places and items % places):
        pytest.skip("no partial last wave for this shape on this GPU")
    o, f = run_gpu(x, out_dtype=torch.float32)
    o_ref, f_ref = run_oracle(x)
    check_parity(x, o, f, o_ref, f_ref)


def test_status_word_reports_bad_inputs_without_fault():
    x = make_inputs(2, seed=1, T=256, H=2, Hv=2)
    d = to_dev(x)
    bad_cu = torch.tensor([0, 300], dtype=torch.int32, device="cuda")   # beyond T
    o, f, desc, ws = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                     None, bad_cu, out_dtype=torch.float32, return_desc=True)
    assert B.gdn_read_status(desc) & 1
    small = torch.tensor([0, 256], dtype=torch.int32, device="cuda")
    o, f, desc, ws = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                     None, small, nt_max=2, out_dtype=torch.float32,
                                     return_desc=True)
    assert B.gdn_read_status(desc) & 2
    o, f, desc, ws = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                     None, small, out_dtype=torch.float32, return_desc=True)
    assert B.gdn_read_status(desc) == 0


def test_overwrite_closed_form_on_gpu():
    """beta = 1, unit keys, q = k, scale = 1: o_t = v_t."""
    x = make_inputs(2, seed=21, T=200, H=2, Hv=4, dtype="f32")
    x["beta"] = torch.ones_like(x["beta"])
    x["q"] = x["k"].clone()
    x["scale"] = 1.0
    o, _ = run_gpu(x)
    assert ratio(o, x["v"].double().numpy()) <= TOL_F32


def test_cuda_graph_replay_bitwise():
    """Capture once with static buffers; replays under new cu_seqlens match eager bitwise."""
    x = make_inputs(4)
    d = to_dev(x)
    static_cu = d["cu_seqlens"].clone()
    out = torch.zeros(x["T"], x["Hv"], 128, device="cuda")
    fin = torch.zeros_like(d["initial_state"])
    desc = B.make_desc(x["T"], x["N"], x["H"], x["Hv"], torch.bfloat16, torch.float32)
    ws = B.alloc_workspace(desc, "cuda")
    call = lambda: B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                   d["initial_state"], static_cu, out=out, final_state=fin,
                                   workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    rng = np.random.default_rng(0)
    for trial in range(3):
        lengths = list(rng.integers(1, 120, size=int(rng.integers(1, 33))))
        cu = np.concatenate([[0], np.cumsum(lengths)])
        cu = np.concatenate([cu, [cu[-1]] * (33 - len(cu))]).astype(np.int32)
        static_cu.copy_(torch.from_numpy(cu))
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        o_g, f_g = out.clone(), fin.clone()
        out.zero_()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_g, out) and torch.equal(f_g, fin), trial


def test_scan_wait_timeout_is_reported_and_recoverable():
    """A bounded on-chip wait that runs out: the testing hook makes the scan wait on an event
    that never happens; the wait gives up, the call returns with GDN_DEV_TIMEOUT in the status
    word and no fault or hang (copies in flight drained); with the hook off, the next call on
    the same workspace is clean and parity-green."""
    x = make_inputs(2, seed=11, T=1024, H=4, Hv=8)
    d = to_dev(x)
    desc = B.make_desc(x["T"], x["N"], x["H"], x["Hv"], torch.bfloat16, torch.float32)
    ws = B.alloc_workspace(desc, "cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], d["initial_state"],
            d["cu_seqlens"])
    try:
        B.gdn_test_scan_timeout(64)
        _, _, desc1, _ = B.gdn_chunk_fwd(*args, workspace=ws, out_dtype=torch.float32,
                                         return_desc=True)
        torch.cuda.synchronize()
        assert B.gdn_read_status(desc1) & 8
    finally:
        B.gdn_test_scan_timeout(0)
    o, f, desc2, _ = B.gdn_chunk_fwd(*args, workspace=ws, out_dtype=torch.float32,
                                     return_desc=True)
    assert B.gdn_read_status(desc2) == 0
    o_ref, f_ref = run_oracle(x)
    check_parity(x, o, f, o_ref, f_ref, TOL_BF16)
