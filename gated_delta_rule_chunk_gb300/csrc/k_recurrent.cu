// Token-serial recurrent forward: decode and speculative verification.
//
// "Chunking Qwen3.5's gated DeltaNet for 1.5x faster prefill on Apple Silicon",
// section "How does decode run a sequential update on a GPU?": at a handful of
// tokens there is nothing to parallelise across time, so the kernel keeps the
// serial order and parallelises over the state. One thread owns one value
// column of one head's fp32 state (128 floats, in registers for the whole call);
// per token it applies the decay, forms the state's prediction for the key,
// writes the rank-1 correction and reads the output, and between tokens of a
// call the state never leaves the chip. Section "Does the chunked kernel match
// the serial one?": verification must reproduce what decode computes, so a call
// over n tokens runs, token by token, exactly the operations of n one-token
// calls (the tests check this bit for bit).
//
// Per token t of a sequence, column j of the state s = S[:, j] (S is dk x dv):
//   a = exp(g_t);  pred = a (s . k_t);  s <- a s + (beta_t k_t) (v_tj - pred)
//   o_tj = scale (s . q_t)
// with k_t and q_t divided by sqrt(sum x^2 + eps) first when the L2 norm is on.
// Each dot product is summed in four interleaved partial sums, combined as
// (p0 + p1) + (p2 + p3): a fixed order, the same for every call.
//
// Grid: (sequence, value head, dv / 32); one warp per CTA owns 32 columns.
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kCols = 32;

__device__ __forceinline__ float4 load4(const void* base, size_t idx, bool bf16) {
  if (bf16) {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + idx);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kCols) recurrent_kernel(RecParams p) {
  __shared__ __align__(16) float kq[2][kDk];  // k and q of the current token
  const int lane = threadIdx.x;
  const int n = blockIdx.x, hv = blockIdx.y, j = blockIdx.z * kCols + lane;
  const int h = hv / p.HG;
  int start = 0, len = p.T;
  if (p.cu) {  // clamp to [0, T]; a decreasing pair is an empty sequence (status bit)
    int a = p.cu[n], b = p.cu[n + 1];
    const int ac = min(max(a, 0), p.T), bc = min(max(b, 0), p.T);
    if (ac != a || bc != b || bc < ac) {
      if (lane == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_status(p.status, GDN_DEV_BAD_CU_SEQLENS);
    }
    start = ac;
    len = max(bc - ac, 0);
  }
  const size_t srow = (((size_t)n * p.Hv + hv) * kDv + j) * kDk;  // state row j: S[:, j]
  float s[kDk];
  if (p.s0) {
#pragma unroll
    for (int i = 0; i < kDk; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(p.s0 + srow + i);
      s[i] = x.x;
      s[i + 1] = x.y;
      s[i + 2] = x.z;
      s[i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kDk; ++i) s[i] = 0.f;
  }

  for (int t = start; t < start + len; ++t) {
    {  // k_t and q_t (4 elements per lane), optionally L2-normalised, into shared memory
      const size_t base = ((size_t)t * p.H + h) * kDk + 4 * lane;
      float4 kv = load4(p.k, base, p.bf16_in), qv = load4(p.q, base, p.bf16_in);
      if (p.l2norm) {
        const float rk = 1.f / sqrtf(warp_sum(kv.x * kv.x + kv.y * kv.y + kv.z * kv.z + kv.w * kv.w) + p.eps);
        const float rq = 1.f / sqrtf(warp_sum(qv.x * qv.x + qv.y * qv.y + qv.z * qv.z + qv.w * qv.w) + p.eps);
        kv = make_float4(kv.x * rk, kv.y * rk, kv.z * rk, kv.w * rk);
        qv = make_float4(qv.x * rq, qv.y * rq, qv.z * rq, qv.w * rq);
      }
      __syncwarp();  // the previous token's k and q have been read
      *reinterpret_cast<float4*>(&kq[0][4 * lane]) = kv;
      *reinterpret_cast<float4*>(&kq[1][4 * lane]) = qv;
      __syncwarp();
    }
    const size_t tv = (size_t)t * p.Hv + hv;
    const float a = expf(p.g[tv]);
    const float be = p.beta[tv];
    const float vj = p.bf16_in ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.v)[tv * kDv + j])
                               : static_cast<const float*>(p.v)[tv * kDv + j];
    // pred = a (s . k)
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
    for (int i = 0; i < kDk; i += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(&kq[0][i]);
      p0 = fmaf(s[i], k4.x, p0);
      p1 = fmaf(s[i + 1], k4.y, p1);
      p2 = fmaf(s[i + 2], k4.z, p2);
      p3 = fmaf(s[i + 3], k4.w, p3);
    }
    const float d = vj - a * ((p0 + p1) + (p2 + p3));
    // s <- a s + (beta k) d
#pragma unroll
    for (int i = 0; i < kDk; i += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(&kq[0][i]);
      s[i] = fmaf(a, s[i], (be * k4.x) * d);
      s[i + 1] = fmaf(a, s[i + 1], (be * k4.y) * d);
      s[i + 2] = fmaf(a, s[i + 2], (be * k4.z) * d);
      s[i + 3] = fmaf(a, s[i + 3], (be * k4.w) * d);
    }
    // o = scale (s . q)
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
    for (int i = 0; i < kDk; i += 4) {
      const float4 q4 = *reinterpret_cast<const float4*>(&kq[1][i]);
      o0 = fmaf(s[i], q4.x, o0);
      o1 = fmaf(s[i + 1], q4.y, o1);
      o2 = fmaf(s[i + 2], q4.z, o2);
      o3 = fmaf(s[i + 3], q4.w, o3);
    }
    const float o = p.scale * ((o0 + o1) + (o2 + o3));
    if (p.out_bf16)
      static_cast<__nv_bfloat16*>(p.out)[tv * kDv + j] = __float2bfloat16_rn(o);
    else
      static_cast<float*>(p.out)[tv * kDv + j] = o;
  }

  if (p.sT) {
#pragma unroll
    for (int i = 0; i < kDk; i += 4)
      *reinterpret_cast<float4*>(p.sT + srow + i) = make_float4(s[i], s[i + 1], s[i + 2], s[i + 3]);
  }
}

}  // namespace

void launch_recurrent(const RecParams& p, cudaStream_t s) {
  if (p.N <= 0) return;
  recurrent_kernel<<<dim3(p.N, p.Hv, kDv / kCols), kCols, 0, s>>>(p);
}

}  // namespace gdn
