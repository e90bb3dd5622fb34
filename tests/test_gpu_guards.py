"""Guard bands: the out-of-bounds check this build uses in place of a memory checker.

Every workspace region gets a 4 KiB gap after it (GDN_FLAG_WORKSPACE_GUARDS), and out
and final_state sit inside larger buffers. Everything outside what the library may
write is filled with a NaN bit pattern before the call and must read back bit for bit
afterwards; the guarded call must also give the same results, bit for bit, as the
unguarded one (only the layout differs). Run on the five workloads of the parity tests.
"""
import pytest
import torch

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.inputs import make_inputs

from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu

PAD = 4096  # guard elements (fp32) before and after out and final_state


def _guarded(shape, device="cuda"):
    n = 1
    for s in shape:
        n *= s
    flat = torch.full((n + 2 * PAD,), -1, dtype=torch.int32, device=device).view(torch.float32)
    return flat, flat[PAD:PAD + n].view(*shape)


def _intact(flat_f32, n):
    bits = flat_f32.view(torch.int32)
    return bool((bits[:PAD] == -1).all()) and bool((bits[PAD + n:] == -1).all())


@pytest.mark.parametrize("wid", [0, 1, 2, 3, 4])
def test_guard_bands_untouched(wid):
    x = make_inputs(wid)
    d = to_dev(x)
    T, N, H, Hv, D = x["T"], x["N"], x["H"], x["Hv"], x["dk"]
    desc = B.make_desc(T, N, H, Hv, d["q"].dtype, torch.float32, dk=D, dv=D,
                       flags=B.GDN_FLAG_WORKSPACE_GUARDS)
    size = B.gdn_workspace_size(desc)
    regions = B.gdn_workspace_regions(desc)
    assert regions and regions[-1][1] <= size
    ws = torch.full((size + 4096,), 0xFF, dtype=torch.uint8, device="cuda")
    out_flat, out = _guarded((T, Hv, D))
    fin_flat, fin = _guarded((N, Hv, D, D))
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], d["initial_state"],
            d["cu_seqlens"])
    _, _, gdesc, _ = B.gdn_chunk_fwd(*args, out=out, final_state=fin, workspace=ws,
                                     out_dtype=torch.float32, return_desc=True,
                                     extra_flags=B.GDN_FLAG_WORKSPACE_GUARDS)
    assert B.gdn_read_status(gdesc) == 0
    torch.cuda.synchronize()
    assert _intact(out_flat, T * Hv * D) and _intact(fin_flat, N * Hv * D * D)
    host = ws.cpu()
    gaps = [(regions[i][1], regions[i + 1][0]) for i in range(len(regions) - 1)]
    gaps.append((regions[-1][1], size + 4096))
    for a, b in gaps:
        assert b - a >= 4096
        assert bool((host[a:b] == 0xFF).all()), (wid, a, b)
    # the guards change the layout only: same results as the unguarded call
    o2, f2 = B.gdn_chunk_fwd(*args, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = slice(int(x["cu_seqlens"][0]), int(x["cu_seqlens"][-1]))
    assert torch.equal(out[rows], o2[rows]) and torch.equal(fin, f2)
