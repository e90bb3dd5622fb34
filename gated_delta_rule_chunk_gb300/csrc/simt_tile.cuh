// Register-tiled fp32 products and small helpers shared by the SIMT kernels
// (the general forward path and the backward pass).
#pragma once

#include "gdn_common.cuh"

namespace gdn {

template <typename TIn>
__device__ __forceinline__ float ld_in(const void* base, size_t idx) {
  return to_f32(reinterpret_cast<const TIn*>(base)[idx]);
}

template <int R>
__device__ __forceinline__ void ldv(const float* p, float (&v)[R]) {
  if constexpr (R == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (R == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  } else {
    v[0] = *p;
  }
}

// acc[r][c] += sum_{k0 <= k < k1} X[k * ldx + m0 + r] * Y[k * ldy + n0 + c]: both operands
// k-major in shared memory (a warp reads one row of each per step).
template <int RM, int RN>
__device__ __forceinline__ void fma_tile(float (&acc)[RM][RN], const float* X, int ldx,
                                         const float* Y, int ldy, int m0, int n0, int k0,
                                         int k1) {
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    float a[RM], b[RN];
    ldv<RM>(X + k * ldx + m0, a);
    ldv<RN>(Y + k * ldy + n0, b);
#pragma unroll
    for (int r = 0; r < RM; ++r)
#pragma unroll
      for (int c = 0; c < RN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}

// Copy n elements with every thread keeping U loads in flight: ld(i) returns element
// i, st(i, x) stores it (usually a transposing or converting store to shared memory).
// A plain one-load-per-iteration loop would pay one memory latency per iteration.
template <int U, typename Ld, typename St>
__device__ __forceinline__ void staged_copy(int n, int tid, int nthr, Ld ld, St st) {
  for (int base = tid; base < n; base += U * nthr) {
    float r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nthr;
      r[u] = i < n ? ld(i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nthr;
      if (i < n) st(i, r[u]);
    }
  }
}

template <int RM, int RN>
__device__ __forceinline__ void zero(float (&acc)[RM][RN]) {
#pragma unroll
  for (int r = 0; r < RM; ++r)
#pragma unroll
    for (int c = 0; c < RN; ++c) acc[r][c] = 0.f;
}

// Resolve the chunk of this slot; returns false (after flagging) if the CTA has nothing to do.
template <typename P>
__device__ __forceinline__ bool resolve_slot(const P& p, int slot, int& t0, int& L,
                                             int& wslot) {
  const int2 e = p.chunk_table[slot];
  if (e.x < 0) return false;  // sentinel slot: early exit
  if (e.x >= p.N) {
    set_status(p.status, GDN_DEV_BAD_CHUNK_TABLE);
    return false;
  }
  const SeqView sv = seq_view(p, e.x);
  const int nch = (sv.len + kChunk - 1) / kChunk;
  if (e.y < 0 || e.y >= nch) {
    set_status(p.status, GDN_DEV_BAD_CHUNK_TABLE);
    return false;
  }
  wslot = sv.first_slot + e.y;
  if (wslot >= p.nt_max) {
    set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    return false;
  }
  t0 = sv.start + kChunk * e.y;
  L = min(kChunk, sv.len - kChunk * e.y);
  return true;
}

}  // namespace gdn
