"""Child process of test_gpu_debug_build.py (not a test module): loads the GDN_DEBUG
library, runs the given workloads through gdn_chunk_fwd, and saves outputs, final states
and device status words (plus those of a run with the out-of-range testing hook on and a
clean run after it) to the file named on the command line."""
import json
import os
import sys

import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs


def run(x):
    d = {k: (x[k].cuda().contiguous() if x.get(k) is not None else None)
         for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens")}
    o, f, desc, _ = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                    d["initial_state"], d["cu_seqlens"],
                                    out_dtype=torch.float32, return_desc=True)
    return o.cpu(), f.cpu(), B.gdn_read_status(desc)


def main():
    lib_path, cases_json, out_path = sys.argv[1:4]
    B.load_library(lib_path)
    assert B.gdn_debug_build(), "the child must run the GDN_DEBUG library"
    res = {"cases": []}
    for kw in json.loads(cases_json):
        res["cases"].append(run(make_inputs(**kw)))
    x = make_inputs(2)
    B.gdn_test_debug_poison(True)
    try:
        res["poisoned_status"] = run(x)[2]
    finally:
        B.gdn_test_debug_poison(False)
    res["after"] = run(x)
    torch.save(res, out_path)


if __name__ == "__main__":
    sys.path.insert(0, os.getcwd())
    main()
