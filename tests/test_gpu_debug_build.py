"""The GDN_DEBUG build (libgdn_debug.so): device-side index checks on every global copy and
store of the bf16 forward path's chunk-table, intra and scan kernels.

On valid calls the checks must stay silent and change nothing: status 0 and every output
and final state bit for bit equal to the normal library's, on the five parity workloads
and a short ragged case. On an out-of-range index they must catch it: the testing hook
aims one intra CTA's M copies one value slot past the end of the M region (still inside
the workspace), and the call must come back with GDN_DEV_DEBUG_INDEX and no fault; the
next call on the same workspace is clean again.

The debug library is built on first use (nvcc, all translation units with -DGDN_DEBUG) and
run in a child process, so that this process keeps the normal library loaded."""
import json
import os
import subprocess
import sys

import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.build import build
from gated_delta_rule_chunk_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CASES = [dict(wid=0), dict(wid=1), dict(wid=2), dict(wid=3), dict(wid=4),
         dict(wid=2, seed=7, T=65, H=1, Hv=2)]


def run_normal(x):
    d = {k: (x[k].cuda().contiguous() if x.get(k) is not None else None)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    o, f, desc, _ = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                    d["initial_state"], d["cu_seqlens"],
                                    out_dtype=torch.float32, return_desc=True)
    return o.cpu(), f.cpu(), B.gdn_read_status(desc)


def test_debug_build_checks(tmp_path):
    assert not B.gdn_debug_build()  # this process runs the normal library
    lib = build(debug=True)
    out = str(tmp_path / "debug_results.pt")
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_child.py"), lib,
                        json.dumps(CASES), out], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = torch.load(out)
    for kw, (od, fd, sd) in zip(CASES, res["cases"]):
        x = make_inputs(**kw)
        on, fn, sn = run_normal(x)
        rows = slice(int(x["cu_seqlens"][0]), int(x["cu_seqlens"][-1]))
        assert sn == 0 and sd == 0, (kw, sn, sd)
        assert torch.equal(od[rows], on[rows]) and torch.equal(fd, fn), kw
    assert res["poisoned_status"] & B.GDN_DEV_DEBUG_INDEX, res["poisoned_status"]
    x = make_inputs(2)
    oa, fa, sa = res["after"]
    on, fn, _ = run_normal(x)
    rows = slice(int(x["cu_seqlens"][0]), int(x["cu_seqlens"][-1]))
    assert sa == 0 and torch.equal(oa[rows], on[rows]) and torch.equal(fa, fn)
