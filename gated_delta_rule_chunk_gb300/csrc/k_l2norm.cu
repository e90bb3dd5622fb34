// K4: optional q/k L2-norm prologue.
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 7: for a small
// fixed row length (128) the whole row is loaded once, reduced, and scaled by
// 1/sqrt(sum + eps). Here one warp owns one 128-element row (8 bytes of bf16 or
// 16 bytes of fp32 per lane, one coalesced load) and writes only the fp32
// factor 1/sqrt(sum x^2 + eps). The intra- and inter-chunk kernels apply the
// factors in fp32 where q and k enter their products, so the raw inputs stay
// exact tensor-core operands and no normalised copy of q or k is written.
#include "gdn_common.cuh"

namespace gdn {

template <bool kBf16>
__global__ void __launch_bounds__(256)
l2norm_kernel(const void* __restrict__ q, const void* __restrict__ k, int rows, float eps,
              float* __restrict__ qrn, float* __restrict__ krn) {
  const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= 2 * rows) return;
  const bool is_q = warp < rows;
  const int row = is_q ? warp : warp - rows;
  const void* src = is_q ? q : k;
  float ss = 0.f;
  if (kBf16) {
    const uint2 raw = reinterpret_cast<const uint2*>(src)[(size_t)row * 32 + lane];
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    ss = fa.x * fa.x + fa.y * fa.y + fb.x * fb.x + fb.y * fb.y;
  } else {
    const float4 f = reinterpret_cast<const float4*>(src)[(size_t)row * 32 + lane];
    ss = f.x * f.x + f.y * f.y + f.z * f.z + f.w * f.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) (is_q ? qrn : krn)[row] = 1.0f / sqrtf(ss + eps);
}

void launch_l2norm(const void* q, const void* k, bool bf16, int T, int H, float eps,
                   float* qrn, float* krn, cudaStream_t s) {
  const int rows = T * H;
  if (rows == 0) return;
  const int blocks = (2 * rows * 32 + 255) / 256;
  if (bf16)
    l2norm_kernel<true><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
  else
    l2norm_kernel<false><<<blocks, 256, 0, s>>>(q, k, rows, eps, qrn, krn);
}

}  // namespace gdn
