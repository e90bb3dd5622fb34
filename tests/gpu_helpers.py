"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_delta_rule_chunk_gb300 import binding as B

# Tolerances on max|x - x_ref| / rms(x_ref): fp32 inputs 1e-4, bf16 inputs
# (fp32 state, fp32 output store) 1e-2.
TOL_F32 = 1e-4
TOL_BF16 = 1e-2


def tol_for(x) -> float:
    return TOL_F32 if x["dtype"] == "f32" else TOL_BF16


def to_dev(x: dict, dev="cuda") -> dict:
    out = dict(x)
    for key in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
        if x.get(key) is not None:
            out[key] = x[key].to(dev).contiguous()
    return out


def run_gpu(x: dict, out_dtype=torch.float32, expect_status=0, **kw):
    """Run the CUDA path through the C ABI; the device status word must be clean."""
    d = to_dev(x)
    o, f, desc, _ = B.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"],
                                    d.get("initial_state"), d["cu_seqlens"],
                                    out_dtype=out_dtype, return_desc=True, **kw)
    status = B.gdn_read_status(desc)
    assert status == expect_status, f"device status {status:#x}"
    return o, f


def run_oracle(x: dict, **kw):
    return oracle.recurrent_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                    x.get("initial_state"), x["cu_seqlens"], **kw)


def ratio(a, ref) -> float:
    a = a.detach().double().cpu().numpy() if hasattr(a, "detach") else np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt((ref * ref).mean()))
    return float(np.abs(a - ref).max() / max(rms, 1e-30))


def valid_rows(x: dict) -> np.ndarray:
    cu = x["cu_seqlens"].numpy()
    return np.arange(int(cu[0]), int(cu[-1]))
