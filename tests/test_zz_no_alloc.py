"""gdn_chunk_fwd_noalloc, the entry point for callers that cannot allocate
device memory (it uses the library's own static scratch instead of a
caller-provided workspace), gives the same results as gdn_chunk_fwd.

This file is collected last on purpose, and it also passes when run alone.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs

from gpu_helpers import TOL_BF16, ratio, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    """Same kernels, same inputs: the results equal gdn_chunk_fwd's bit for bit, on two
    calls in a row (the second finds the first call's contents in the shared scratch),
    and the scratch's status word reads clean."""
    x = make_inputs(2, seed=31, T=1000, H=16, Hv=32)   # workspace fits in the static scratch
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], d["initial_state"],
            d["cu_seqlens"])
    ref_o, ref_f = B.gdn_chunk_fwd(*args, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for _ in range(2):
        o, f = B.gdn_chunk_fwd_noalloc(*args, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(f, ref_f)
        assert B.gdn_noalloc_read_status() == 0
    # and against the oracle, at the bf16 path's tolerance
    assert ratio(o, run_oracle(x)[0]) <= TOL_BF16


def test_noalloc_status_word_reports_bad_cu_seqlens():
    """A device-detected problem of an allocation-free call is readable: a cu_seqlens entry
    beyond T sets GDN_DEV_BAD_CU_SEQLENS in the scratch's status word; the next clean call
    clears it."""
    x = make_inputs(2, seed=33, T=256, H=2, Hv=2)
    d = to_dev(x)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], None)
    B.gdn_chunk_fwd_noalloc(*args, torch.tensor([0, 300], dtype=torch.int32, device="cuda"),
                            out_dtype=torch.float32)
    assert B.gdn_noalloc_read_status() & 1
    B.gdn_chunk_fwd_noalloc(*args, torch.tensor([0, 256], dtype=torch.int32, device="cuda"),
                            out_dtype=torch.float32)
    assert B.gdn_noalloc_read_status() == 0


def test_noalloc_rejects_problems_larger_than_its_scratch():
    x = make_inputs(2, seed=32, T=4096, H=16, Hv=32)
    desc = B.make_desc(x["T"], x["N"], x["H"], x["Hv"], torch.bfloat16, torch.float32)
    assert B.gdn_workspace_size(desc) > B.GDN_NOALLOC_SCRATCH_BYTES
    f = ctypes.c_void_p(256)   # never dereferenced: the size check comes first
    rc = B.load_library().gdn_chunk_fwd_noalloc(ctypes.byref(desc), f, f, f, f, f, 0.0, None,
                                                None, None, f, None, None)
    assert rc == -5
