"""Seeded synthetic inputs for the chunked gated-delta-rule forward.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests. It holds no arithmetic of the method itself: it only draws
random tensors in the shapes and distributions of the workloads and packs
them for the library boundary.

Distributions (the Qwen3.5-style workloads; all draws in fp64 on a CPU
``torch.Generator`` seeded with ``1000 + workload id`` unless a seed is given):

* q, k ~ N(0, 1), then scaled to unit L2 norm per (token, head) -- the
  standard way to sample directions uniformly (the layer's own L2-norm step is
  then a no-op, so the optional prologue stays off for these workloads);
* v ~ N(0, 1);
* g = log(sigmoid(x)) with x ~ N(2, 1), per (token, value head), evaluated as
  -log1p(exp(-x)) so that it never rounds to log(1) = 0 or overflows; with
  per-channel gates the same draw is made independently per key channel,
  g [T, Hv, dk] (optionally with a per-channel offset added to x, drawn once
  from U[lo, hi], to spread the channels' decay rates);
* beta = sigmoid(y), y ~ N(0, 1);
* initial states ~ N(0, 0.02) (0.02 read as the standard deviation), fp32,
  layout [N, Hv, dv, dk];
* scale = 1 / sqrt(dk).

q, k, v are then rounded once (RNE) to the workload dtype; g, beta and the
states stay fp32. Both sides read exactly these rounded values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

CHUNK = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    H: int
    Hv: int
    dk: int
    dv: int
    dtype: str                    # "f32" or "bf16" for q/k/v
    with_initial_state: bool
    kind: str                     # "single", "varlen", "static_bound", "fixed", "conv"
    T: int = 0                    # single: sequence length
    n_seqs: int = 1               # varlen: number of sequences
    max_len: int = 0              # varlen: lengths ~ U[1, max_len]
    T_max: int = 0                # static_bound: token budget (rows of the buffers)
    N_max: int = 0                # static_bound: padded sequence count
    n_real: int = 0               # static_bound: real sequences
    real_max_len: int = 0         # static_bound: lengths ~ U[1, real_max_len]
    fixed_lens: tuple = ()        # fixed: the sequence lengths
    gate: str = "scalar"          # "scalar" (g [T, Hv]) or "channel" (g [T, Hv, dk])


WORKLOADS = {
    0: Workload(0, "tiny single sequence T=128 H=Hv=2 d=128 fp32", 2, 2, 128, 128,
                "f32", False, "single", T=128),
    1: Workload(1, "Qwen3.5-0.8B-shaped prefill T=4096 H=16 Hv=16 d=128 bf16", 16, 16,
                128, 128, "bf16", False, "single", T=4096),
    2: Workload(2, "Qwen3.5-9B-shaped GQA prefill T=4096 H=16 Hv=32 d=128 bf16", 16, 32,
                128, 128, "bf16", True, "single", T=4096),
    3: Workload(3, "varlen batch of 8 sequences, lengths U[1,2048], H=16 Hv=32 bf16", 16,
                32, 128, 128, "bf16", True, "varlen", n_seqs=8, max_len=2048),
    4: Workload(4, "static-bound T_max=4096 N_max=32, 20 sequences, H=16 Hv=32 bf16", 16,
                32, 128, 128, "bf16", True, "static_bound", T_max=4096, N_max=32,
                n_real=20, real_max_len=204),
    # token-serial (decode / speculative verify) workloads of the recurrent kernel
    5: Workload(5, "decode step: 64 sequences x 1 token, H=16 Hv=32 d=128 bf16", 16, 32,
                128, 128, "bf16", True, "fixed", fixed_lens=(1,) * 64),
    6: Workload(6, "speculative verify: 8 sequences x 8 tokens, H=16 Hv=32 d=128 bf16", 16,
                32, 128, 128, "bf16", True, "fixed", fixed_lens=(8,) * 8),
    # front end (conv + SiLU over the qkv projection output; make_conv_inputs)
    7: Workload(7, "front end: conv1d d=4 + SiLU over the qkv projection, T=4096 H=16 Hv=32 "
                "bf16", 16, 32, 128, 128, "bf16", True, "conv", T=4096),
    # head size 64 and per-channel gates (the fp32 SIMT chunk kernels)
    8: Workload(8, "head size 64 GQA prefill T=4096 H=16 Hv=32 d=64 bf16", 16, 32, 64, 64,
                "bf16", True, "single", T=4096),
    9: Workload(9, "per-channel gates GQA prefill T=4096 H=16 Hv=32 d=128 bf16", 16, 32, 128,
                128, "bf16", True, "single", T=4096, gate="channel"),
}

HEADLINE = 2


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def draw_lengths(wl: Workload, gen: torch.Generator) -> list:
    """Sequence lengths of a workload (before any zero-length padding)."""
    if wl.kind == "single":
        return [wl.T]
    if wl.kind == "fixed":
        return list(wl.fixed_lens)
    if wl.kind == "conv":
        return [wl.T]
    if wl.kind == "varlen":
        out = []
        while len(out) < wl.n_seqs:
            x = int(torch.randint(1, wl.max_len + 1, (1,), generator=gen))
            if x % CHUNK != 0:       # the workload asks for non-multiples of 64
                out.append(x)
        return out
    if wl.kind == "static_bound":
        while True:
            ls = [int(x) for x in torch.randint(1, wl.real_max_len + 1, (wl.n_real,),
                                                generator=gen)]
            if sum(ls) <= wl.T_max - 16:
                return ls
    raise ValueError(wl.kind)


def cu_from_lengths(lengths, pad_to: Optional[int] = None) -> torch.Tensor:
    """int32 prefix sums [len(lengths)+1], optionally padded with zero-length tails."""
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + int(x))
    if pad_to is not None:
        cu += [cu[-1]] * (pad_to - len(cu))
    return torch.tensor(cu, dtype=torch.int32)


def unit_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale each last-axis row to unit length (sampling directions on the sphere)."""
    return x / x.norm(dim=-1, keepdim=True)


def gates(x: torch.Tensor) -> torch.Tensor:
    """log(sigmoid(x)) without cancellation: -log1p(exp(-x))."""
    return -torch.nn.functional.softplus(-x)


def make_inputs(wid: int = HEADLINE, seed: Optional[int] = None, T: Optional[int] = None,
                H: Optional[int] = None, Hv: Optional[int] = None,
                lengths: Optional[list] = None, dtype: Optional[str] = None,
                with_initial_state: Optional[bool] = None, normalise_qk: bool = True,
                d: Optional[int] = None, channel_gates: Optional[bool] = None,
                gate_offsets: Optional[tuple] = None) -> dict:
    """Draw one workload's inputs on the CPU.

    Overrides (T, H, Hv, lengths, dtype, with_initial_state) let tests build
    smaller cases with the same distributions; d sets dk = dv, channel_gates the
    gate kind, gate_offsets (lo, hi) the per-channel offset range. Returns a dict
    of CPU tensors: q, k [T,H,dk]; v [T,Hv,dv]; g [T,Hv] or [T,Hv,dk] and beta
    [T,Hv] fp32; initial_state
    [N,Hv,dv,dk] fp32 or None; cu_seqlens int32 [N+1]; plus scalars
    scale, T, N, H, Hv, dk, dv, nt_max, n_tokens (valid rows) and lengths.
    """
    wl = WORKLOADS[wid]
    gen = _gen(1000 + wid if seed is None else seed)
    H = H or wl.H
    Hv = Hv or wl.Hv
    dk, dv = (d, d) if d is not None else (wl.dk, wl.dv)
    chan = (wl.gate == "channel") if channel_gates is None else channel_gates
    dtype = dtype or wl.dtype
    init = wl.with_initial_state if with_initial_state is None else with_initial_state
    if lengths is None:
        if T is not None and wl.kind in ("single", "fixed"):
            lengths = [T]
        else:
            lengths = draw_lengths(wl, gen)
    lengths = [int(x) for x in lengths]
    if wl.kind == "static_bound" and T is None:
        rows = wl.T_max
        cu = cu_from_lengths(lengths, pad_to=wl.N_max + 1)
    else:
        rows = T if T is not None else sum(lengths)
        cu = cu_from_lengths(lengths)
    assert rows >= int(cu[-1])
    N = cu.numel() - 1
    f64 = torch.float64
    q = torch.randn(rows, H, dk, generator=gen, dtype=f64)
    k = torch.randn(rows, H, dk, generator=gen, dtype=f64)
    if normalise_qk:
        q, k = unit_rows(q), unit_rows(k)
    v = torch.randn(rows, Hv, dv, generator=gen, dtype=f64)
    if chan:
        x = torch.randn(rows, Hv, dk, generator=gen, dtype=f64) + 2.0
        if gate_offsets is not None:
            lo, hi = gate_offsets
            x = x + (lo + (hi - lo) * torch.rand(dk, generator=gen, dtype=f64))
        g = gates(x)
    else:
        g = gates(torch.randn(rows, Hv, generator=gen, dtype=f64) + 2.0)
    beta = torch.sigmoid(torch.randn(rows, Hv, generator=gen, dtype=f64))
    s0 = (0.02 * torch.randn(N, Hv, dv, dk, generator=gen, dtype=f64)) if init else None
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    cast = lambda x: x.to(tdt).contiguous()
    nt_max = -(-rows // CHUNK) + N - 1
    return dict(
        q=cast(q), k=cast(k), v=cast(v),
        g=g.float().contiguous(), beta=beta.float().contiguous(),
        initial_state=None if s0 is None else s0.float().contiguous(),
        cu_seqlens=cu, scale=1.0 / math.sqrt(dk),
        T=rows, N=N, H=H, Hv=Hv, dk=dk, dv=dv, nt_max=nt_max, dtype=dtype,
        n_tokens=int(cu[-1]), lengths=lengths, wid=wid, channel_gates=chan,
    )


def make_conv_inputs(seed: int = 7, T: int = 64, H: int = 2, Hv: int = 4, d_conv: int = 4,
                     lengths: Optional[list] = None, dtype: str = "bf16",
                     with_state: bool = True, rows: Optional[int] = None,
                     cu_offset: int = 0) -> dict:
    """Inputs of the front end: the qkv projection output x [rows, C] ~ N(0, 1)
    (C = 2*H*128 + Hv*128, rounded once to `dtype`), conv taps [C, d_conv] ~ N(0, 0.5)
    fp32, conv states [N, C, d_conv - 1] ~ N(0, 1) fp32 (or None), cu_seqlens from
    `lengths` (default one sequence of T rows) starting at row `cu_offset`."""
    gen = _gen(seed)
    lengths = [T] if lengths is None else [int(a) for a in lengths]
    cu = [cu_offset]
    for a in lengths:
        cu.append(cu[-1] + a)
    rows = rows if rows is not None else cu[-1]
    C = 2 * H * 128 + Hv * 128
    f64 = torch.float64
    x = torch.randn(rows, C, generator=gen, dtype=f64)
    w = 0.5 * torch.randn(C, d_conv, generator=gen, dtype=f64)
    s0 = torch.randn(len(lengths), C, d_conv - 1, generator=gen, dtype=f64) if with_state else None
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    return dict(x=x.to(tdt).contiguous(), w=w.float().contiguous(),
                state=None if s0 is None else s0.float().contiguous(),
                cu_seqlens=torch.tensor(cu, dtype=torch.int32), H=H, Hv=Hv, d_conv=d_conv,
                T=rows, N=len(lengths), C=C, dtype=dtype)
