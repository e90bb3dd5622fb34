// K4: optional q/k L2-norm prologue.
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 7: for a small
// fixed row length (64 or 128) the whole row is loaded once, reduced, and
// scaled by 1/sqrt(sum + eps). Here one warp owns one row (D / 32 elements per
// lane, one coalesced load) and writes only the fp32 factor 1/sqrt(sum x^2 + eps). The intra- and inter-chunk kernels apply the
// factors in fp32 where q and k enter their products, so the raw inputs stay
// exact tensor-core operands and no normalised copy of q or k is written.
#include "gdn_common.cuh"

namespace gdn {

template <bool kBf16, int D>
__global__ void __launch_bounds__(256)
l2norm_kernel(const void* __restrict__ q, const void* __restrict__ k, int rows, float eps,
              float* __restrict__ qrn, float* __restrict__ krn) {
  constexpr int E = D / 32;  // elements per lane (one coalesced load of the row)
  const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= 2 * rows) return;
  const bool is_q = warp < rows;
  const int row = is_q ? warp : warp - rows;
  const void* src = is_q ? q : k;
  float x[E];
  if constexpr (kBf16) {
    const __nv_bfloat16* r = reinterpret_cast<const __nv_bfloat16*>(src) + (size_t)row * D + lane * E;
    if constexpr (E == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(r);
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
    } else {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(r));
      x[0] = fa.x; x[1] = fa.y;
    }
  } else {
    const float* r = reinterpret_cast<const float*>(src) + (size_t)row * D + lane * E;
    if constexpr (E == 4) {
      const float4 f = *reinterpret_cast<const float4*>(r);
      x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    } else {
      const float2 f = *reinterpret_cast<const float2*>(r);
      x[0] = f.x; x[1] = f.y;
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) ss += x[e] * x[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) (is_q ? qrn : krn)[row] = 1.0f / sqrtf(ss + eps);
}

void launch_l2norm(const void* q, const void* k, bool bf16, int T, int H, int D, float eps,
                   float* qrn, float* krn, cudaStream_t s) {
  const int rows = T * H;
  if (rows == 0) return;
  const int blocks = (2 * rows * 32 + 255) / 256;
  if (D == 128) {
    if (bf16) l2norm_kernel<true, 128><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
    else l2norm_kernel<false, 128><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
  } else {
    if (bf16) l2norm_kernel<true, 64><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
    else l2norm_kernel<false, 64><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
  }
}

}  // namespace gdn
