"""libgdn loads, exports every symbol include/gdn.h declares, and validates
arguments on the host (every call here fails validation before any CUDA call,
so no GPU is needed)."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_chunk_gb300 import binding as B
from gated_delta_rule_chunk_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return B.load_library()


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[\w\s\*]*?\b(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and len(names) >= 7
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.EXPORTED) <= set(names)


def desc(**kw):
    base = dict(T=4096, N=1, H=16, Hv=32, qkv_dtype=__import__("torch").bfloat16)
    base.update(kw)
    return B.make_desc(**base)


def test_check_desc(lib):
    assert B.gdn_check_desc(desc()) == 0
    assert B.gdn_check_desc(desc(Hv=24, H=16)) == -2          # Hv % H != 0
    assert B.gdn_check_desc(desc(N=0)) == -2
    assert B.gdn_check_desc(desc(T=-1)) == -2
    assert B.gdn_check_desc(desc(nt_max=-3)) == -2
    assert B.gdn_check_desc(desc(dk=64, dv=64)) == 0           # head size 64
    assert B.gdn_check_desc(desc(dk=64, dv=128)) == -3         # dk != dv: not built
    assert B.gdn_check_desc(desc(dk=96, dv=96)) == -3
    assert B.gdn_check_desc(desc(flags=B.GDN_FLAG_CHANNEL_GATES)) == 0
    d = desc()
    d.chunk_size = 32
    assert B.gdn_check_desc(d) == -3
    d = desc()
    d.qkv_dtype = 7
    assert B.gdn_check_desc(d) == -3
    assert B.gdn_check_desc(desc(flags=B.GDN_FLAG_WORKSPACE_GUARDS)) == 0
    d = desc()
    d.flags = 16
    assert B.gdn_check_desc(d) == -3
    assert lib.gdn_check_desc(None) == -1


def test_nt_max_bound(lib):
    assert B.gdn_nt_max(4096, 32) == 95
    assert B.gdn_nt_max(4096, 1) == 64
    assert B.gdn_nt_max(128, 1) == 2
    assert B.gdn_nt_max(0, 1) == 0
    assert B.gdn_nt_max(65, 3) == 4
    assert B.gdn_nt_max(-1, 1) == -1 and B.gdn_nt_max(10, 0) == -1


def test_workspace_size(lib):
    import torch
    a = B.gdn_workspace_size(desc())
    b = B.gdn_workspace_size(desc(nt_max=128))
    c = B.gdn_workspace_size(desc(qkv_dtype=torch.float32))
    e = B.gdn_workspace_size(desc(flags=1))
    assert 0 < a < b and a < c and a < e
    # the bridge dominates: about 64 slots x 32 heads x 64 rows x (2 + 4 + 4 + ...) bytes
    assert a >= 64 * 32 * 64 * (128 * 2 + 128 * 4 + 64 * 4)
    assert B.gdn_workspace_size(desc(Hv=24)) == 0
    # the SIMT path (fp32 inputs) keeps fp32 w^T, u, M^T, the decayed q and k images and
    # exp(G_L): 4 * (64 * (4 d) + 64 * 64 + d) bytes per slot
    for dd, fl in ((64, 0), (128, B.GDN_FLAG_CHANNEL_GATES)):
        n = B.gdn_workspace_size(desc(dk=dd, dv=dd, flags=fl, qkv_dtype=torch.float32))
        assert n >= 64 * 32 * 4 * (64 * 4 * dd + 64 * 64 + dd)
    # bf16 with per-channel gates: the tensor-core bridge plus a k image and the decayed
    # q's hi/lo images per value head and exp(G_L) per channel, in place of the scalar-gate
    # path's fp16 k and q images per key head and its exp(G), exp(G_L - G) (512 B per slot)
    n = B.gdn_workspace_size(desc(flags=B.GDN_FLAG_CHANNEL_GATES))
    assert n >= a + 64 * 32 * (16384 + 32768 + 512) - 2 * 64 * 16 * 16384 - 64 * 32 * 512
    # bf16 with a head of 64 runs on the tensor-core kernels zero-padded to 128
    assert B.gdn_workspace_size(desc(dk=64, dv=64)) == a


def _fwd(lib, d, q=16, k=16, v=16, g=16, beta=16, out=16, s0=None, fin=None, cu=None, ci=None):
    f = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.gdn_chunk_fwd(ctypes.byref(d), f(q), f(k), f(v), f(g), f(beta), 0.0, f(s0), f(cu),
                             f(ci), f(out), f(fin), None)


def test_fwd_rejects_before_enqueue(lib):
    d = desc()
    d.workspace = 4096
    d.workspace_bytes = B.gdn_workspace_size(d)
    assert _fwd(lib, d, q=None) == -1
    assert _fwd(lib, d, out=None) == -1
    dd = desc()
    assert _fwd(lib, dd) == -1                                   # no workspace
    assert _fwd(lib, desc(N=2, **{}), cu=None) in (-1, -2)
    d2 = desc(N=2)
    d2.workspace = 4096
    d2.workspace_bytes = 1 << 40
    assert _fwd(lib, d2, cu=None) == -2                          # N > 1 needs cu_seqlens
    assert _fwd(lib, d, q=17) == -4                              # misaligned
    assert _fwd(lib, d, s0=8) == -4
    d3 = desc()
    d3.workspace = 4096 + 128
    d3.workspace_bytes = 1 << 40
    assert _fwd(lib, d3) == -4                                   # workspace alignment
    d4 = desc()
    d4.workspace = 4096
    d4.workspace_bytes = B.gdn_workspace_size(d4) - 1
    assert _fwd(lib, d4) == -5
    bad = desc(Hv=24)
    assert _fwd(lib, bad) == -2


def test_build_chunk_indices_rejects(lib):
    f = ctypes.c_void_p
    assert lib.gdn_build_chunk_indices(f(16), 2, 100, 5, f(16), None, None, None) == -1
    assert lib.gdn_build_chunk_indices(None, 2, 100, 5, f(16), f(16), None, None) == -2
    assert lib.gdn_build_chunk_indices(f(16), 0, 100, 5, f(16), f(16), None, None) == -2
    assert lib.gdn_build_chunk_indices(f(18), 2, 100, 5, f(16), f(16), None, None) == -4


def test_status_strings(lib):
    for s in range(0, -7, -1):
        assert B.status_string(s) not in ("", "unknown status")
    assert B.status_string(-99) == "unknown status"


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle and has no CPU fallback."""
    pkg = os.path.join(ROOT, "gated_delta_rule_chunk_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "gdn_ref" not in text, fn


def _rec(lib, d, q=4096, k=4096, v=4096, g=4096, beta=4096, s0=None, cu=4096, out=4096,
         sT=None):
    return lib.gdn_recurrent_fwd(ctypes.byref(d), q, k, v, g, beta, 0.0, s0, cu, out, sT, None)


def test_recurrent_rejects_before_enqueue(lib):
    """gdn_recurrent_fwd validates everything before touching the GPU."""
    d = desc(N=1)
    assert _rec(lib, d, q=None) == -1
    assert _rec(lib, d, beta=None) == -1
    assert _rec(lib, d, out=None) == -1
    assert _rec(lib, desc(N=3), cu=None) == -2                   # N > 1 needs cu_seqlens
    assert _rec(lib, d, v=4100) == -4                            # misaligned tensor
    assert _rec(lib, d, sT=4104) == -4
    assert _rec(lib, d, cu=4098) == -4
    dw = desc(N=1)
    dw.workspace = 4096 + 64                                     # status word alignment
    assert _rec(lib, dw) == -4
    assert _rec(lib, desc(Hv=24)) == -2
    assert _rec(lib, desc(dk=64)) == -3
    assert _rec(lib, desc(dk=64, dv=64)) == -3                   # built for d = 128 only
    assert _rec(lib, desc(flags=B.GDN_FLAG_CHANNEL_GATES)) == -3


def test_conv_front_rejects_before_enqueue(lib):
    """gdn_conv_front validates everything before touching the GPU."""
    d = desc(N=1)
    f = lambda **kw: lib.gdn_conv_front(
        ctypes.byref(kw.pop("d", d)), kw.get("x", 4096), kw.get("w", 4096), kw.get("dc", 4),
        kw.get("s0", None), kw.get("cu", None), kw.get("q", 4096), kw.get("k", 4096),
        kw.get("v", 4096), kw.get("s1", None), kw.get("sn", None), kw.get("ns", 0), None)
    assert f(x=None) == -1
    assert f(w=None) == -1
    assert f(v=None) == -1
    assert f(dc=0) == -2 and f(dc=9) == -2
    assert f(ns=2) == -2                       # snapshots requested without a buffer
    assert f(sn=4096) == -2                    # a buffer without a count
    assert f(d=desc(N=2)) == -2                # N > 1 needs cu_seqlens
    assert f(q=4104) == -4 and f(x=4100) == -4
    assert f(s1=4098) == -4
    assert f(d=desc(Hv=24)) == -2
    assert f(d=desc(dk=64, dv=64)) == -3       # built for d = 128 only


def test_workspace_regions_and_guard_bands(lib):
    """The region list covers what the library may write, in order and without overlap;
    the guard flag leaves 4 KiB after every region and changes nothing else."""
    import torch
    d0 = desc()
    dg = desc(flags=B.GDN_FLAG_WORKSPACE_GUARDS)
    r0, rg = B.gdn_workspace_regions(d0), B.gdn_workspace_regions(dg)
    assert len(r0) == len(rg) >= 8
    assert r0[0] == (0, 64)                          # the status word comes first
    for (a0, b0), (ag, bg) in zip(r0, rg):
        assert b0 - a0 == bg - ag                    # same region sizes
    for i in range(len(rg) - 1):
        assert rg[i + 1][0] - rg[i][1] >= 4096       # a guard gap after every region
        assert r0[i + 1][0] >= r0[i][1]              # ordered, no overlap
    assert B.gdn_workspace_size(d0) >= r0[-1][1]
    assert B.gdn_workspace_size(dg) >= rg[-1][1] + 4096
    assert B.gdn_workspace_size(dg) == B.gdn_workspace_size(d0) + 4096 * len(rg)
