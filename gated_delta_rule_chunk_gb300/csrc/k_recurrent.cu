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
// (p0 + p1) + (p2 + p3): a fixed order, the same for every call. (Folding the
// output into the prediction pass, o = scale (a (s . q) + beta (k . q) d), measured
// slower here: the extra accumulators spill at 255 registers.)
//
// Data movement: the CTA's 32 state columns (32 rows of the [dv][dk] state,
// 16 KB) come in and go out as TMA tiles of 32 rows x 128 bytes with the
// 128-byte swizzle, so each thread reads its own row from shared memory without
// bank conflicts; the inputs of up to 8 tokens are staged in shared memory at a
// time (cp.async), so the serial token loop waits on no global load, and the first
// block's inputs load while the state tile is in flight (one memory round trip per
// CTA instead of two: what a one-token decode step pays for).
//
// Grid: (sequence, value head, dv / 32); one warp per CTA owns 32 columns.
#include <cuda.h>

#include "gdn_common.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int kCols = 32;
constexpr int kBlk = 8;  // tokens staged per step
constexpr uint32_t kWaitIters = 1u << 22;

// buf (16 KB): the state tile ([4 quarters of 32 columns][32 rows][128 B], swizzled) on
// the way in and out; in between, the staged token inputs of a block: v (fp32 [8][32]) at
// 0, g and beta (fp32 [8] each) at 1024 and 1056, fp32 (normalised) k and q at 8192 and
// 12288. raw: the block's k and q in the input dtype (cp.async), at 0 and 4096. The first
// block's raw k and q, v, g and beta are loaded while the state tile is in flight.
struct __align__(1024) RecSmem {
  unsigned char buf[16384];
  unsigned char raw0[8192];
  float v0[kBlk * kCols];  // v, g and beta of the first block
  float g0[kBlk], b0[kBlk];
  uint64_t bar;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}

// v of this CTA's 32 columns for the block's tokens, g and beta of token `lane`.
__device__ __forceinline__ void load_vgb(const RecParams& p, int blk, int nb, int hv, int c0,
                                         int lane, bool bf16, float (&vr)[kBlk], float& gr,
                                         float& br) {
#pragma unroll
  for (int tt = 0; tt < kBlk; ++tt) {
    const size_t tv = (size_t)(blk + tt) * p.Hv + hv;
    vr[tt] = tt < nb ? (bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.v)[tv * kDv + c0 + lane])
                             : static_cast<const float*>(p.v)[tv * kDv + c0 + lane])
                     : 0.f;
  }
  gr = br = 0.f;
  if (lane < nb) {
    const size_t tv = (size_t)(blk + lane) * p.Hv + hv;
    gr = p.g[tv];
    br = p.beta[tv];
  }
}

__device__ __forceinline__ float4 raw4(const unsigned char* p, bool bf16) {
  if (bf16) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(p);
}

__global__ void __launch_bounds__(kCols)
recurrent_kernel(const __grid_constant__ RecParams p, const __grid_constant__ CUtensorMap tm_s0,
                 const __grid_constant__ CUtensorMap tm_sT) {
  __shared__ RecSmem sm;
  unsigned char* buf = sm.buf;
  const int lane = threadIdx.x;
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * kCols;
  const int h = hv / p.HG;
  const bool bf16 = p.bf16_in != 0;
  const int esz = bf16 ? 2 : 4;
  int start = 0, len = p.T;
  if (p.cu) {  // clamp to [0, T]; a decreasing pair is an empty sequence (status bit)
    const int a = p.cu[n], b = p.cu[n + 1];
    const int ac = min(max(a, 0), p.T), bc = min(max(b, 0), p.T);
    if ((ac != a || bc != b || bc < ac) && lane == 0 && blockIdx.y == 0 && blockIdx.z == 0)
      set_status(p.status, GDN_DEV_BAD_CU_SEQLENS);
    start = ac;
    len = max(bc - ac, 0);
  }
  const int row0 = (n * p.Hv + hv) * kDv + c0;  // first state row (= value column) of this CTA
  bool fail = false;

  // Inputs of a block of up to kBlk tokens: raw k and q by cp.async (lane l: elements
  // 4l..4l+3 of each token), v of this CTA's columns and g, beta into registers.
  auto issue_raw = [&](int blk, int nb, unsigned char* rk, unsigned char* rq) {
    for (int tt = 0; tt < nb; ++tt) {
      const size_t e = ((size_t)(blk + tt) * p.H + h) * kDk + 4 * lane;
      const unsigned char* kg = static_cast<const unsigned char*>(p.k) + e * esz;
      const unsigned char* qg = static_cast<const unsigned char*>(p.q) + e * esz;
      unsigned char* kd = rk + tt * kDk * esz + 4 * lane * esz;
      unsigned char* qd = rq + tt * kDk * esz + 4 * lane * esz;
      if (bf16) {
        cp_async8(kd, kg);
        cp_async8(qd, qg);
      } else {
        cp_async16(kd, kg, true);
        cp_async16(qd, qg, true);
      }
    }
    cp_async_commit();
  };


  // ---------------------------------------------------------------- state in
  float s[kDk];
  if (p.s0 && lane == 0) {
    mbar_init(&sm.bar, 1);
    mbar_init_fence();
    mbar_expect_tx(&sm.bar, 16384);
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) tma_load_2d(buf + qd * 4096, &tm_s0, 32 * qd, row0, &sm.bar);
  }
  // The first block's inputs are loaded while the state tile is in flight.
  if (len > 0) {
    const int nb0 = min(kBlk, len);
    issue_raw(start, nb0, sm.raw0, sm.raw0 + 4096);
    float vr[kBlk], gr, br;
    load_vgb(p, start, nb0, hv, c0, lane, bf16, vr, gr, br);
#pragma unroll
    for (int tt = 0; tt < kBlk; ++tt) sm.v0[tt * kCols + lane] = vr[tt];
    if (lane < kBlk) {
      sm.g0[lane] = gr;
      sm.b0[lane] = br;
    }
  }
  if (p.s0) {
    __syncwarp();
    fail = !mbar_wait(&sm.bar, 0, kWaitIters);
#pragma unroll
    for (int qd = 0; qd < 4; ++qd)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 x = *reinterpret_cast<const float4*>(
            buf + qd * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4));
        s[32 * qd + 4 * c] = x.x;
        s[32 * qd + 4 * c + 1] = x.y;
        s[32 * qd + 4 * c + 2] = x.z;
        s[32 * qd + 4 * c + 3] = x.w;
      }
  } else {
#pragma unroll
    for (int i = 0; i < kDk; ++i) s[i] = 0.f;
  }
  __syncwarp();  // the buffer now stages token inputs

  // ---------------------------------------------------------------- tokens
  const float* kf = reinterpret_cast<const float*>(buf + 8192);
  const float* qf = reinterpret_cast<const float*>(buf + 12288);
  float* vs = reinterpret_cast<float*>(buf);
  float* gs = reinterpret_cast<float*>(buf + 1024);
  float* bs = reinterpret_cast<float*>(buf + 1056);
  for (int blk = start; blk < start + len; blk += kBlk) {
    const int nb = min(kBlk, start + len - blk);
    // raw k and q of the block (the first block's were issued before the state came in)
    const bool first = blk == start;
    const unsigned char* rk = sm.raw0;
    const unsigned char* rq = sm.raw0 + 4096;
    float vr[kBlk], gr = 0.f, br = 0.f;
    if (!first) {
      issue_raw(blk, nb, sm.raw0, sm.raw0 + 4096);
      load_vgb(p, blk, nb, hv, c0, lane, bf16, vr, gr, br);
    }
    cp_async_wait<0>();
    __syncwarp();
    // fp32 (normalised) k and q
    for (int tt = 0; tt < nb; ++tt) {
      float4 kv = raw4(rk + tt * kDk * esz + 4 * lane * esz, bf16);
      float4 qv = raw4(rq + tt * kDk * esz + 4 * lane * esz, bf16);
      if (p.l2norm) {
        const float rk = 1.f / sqrtf(warp_sum(kv.x * kv.x + kv.y * kv.y + kv.z * kv.z + kv.w * kv.w) + p.eps);
        const float rq = 1.f / sqrtf(warp_sum(qv.x * qv.x + qv.y * qv.y + qv.z * qv.z + qv.w * qv.w) + p.eps);
        kv = make_float4(kv.x * rk, kv.y * rk, kv.z * rk, kv.w * rk);
        qv = make_float4(qv.x * rq, qv.y * rq, qv.z * rq, qv.w * rq);
      }
      *reinterpret_cast<float4*>(buf + 8192 + tt * 512 + 16 * lane) = kv;
      *reinterpret_cast<float4*>(buf + 12288 + tt * 512 + 16 * lane) = qv;
    }
    __syncwarp();
    if (first) {  // (staged while the state came in)
#pragma unroll
      for (int tt = 0; tt < kBlk; ++tt) vr[tt] = sm.v0[tt * kCols + lane];
      if (lane < kBlk) {
        gr = sm.g0[lane];
        br = sm.b0[lane];
      }
    }
#pragma unroll
    for (int tt = 0; tt < kBlk; ++tt) vs[tt * kCols + lane] = vr[tt];
    if (lane < kBlk) {
      gs[lane] = gr;
      bs[lane] = br;
    }
    __syncwarp();

#pragma unroll 1
    for (int tt = 0; tt < nb; ++tt) {
      const float a = expf(gs[tt]);
      const float be = bs[tt];
      const float vj = vs[tt * kCols + lane];
      const float* kt = kf + tt * kDk;
      const float* qt = qf + tt * kDk;
      // pred = a (s . k)
      float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
      for (int i = 0; i < kDk; i += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kt + i);
        p0 = fmaf(s[i], k4.x, p0);
        p1 = fmaf(s[i + 1], k4.y, p1);
        p2 = fmaf(s[i + 2], k4.z, p2);
        p3 = fmaf(s[i + 3], k4.w, p3);
      }
      const float d = vj - a * ((p0 + p1) + (p2 + p3));
      // s <- a s + (beta k) d
#pragma unroll
      for (int i = 0; i < kDk; i += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kt + i);
        s[i] = fmaf(a, s[i], (be * k4.x) * d);
        s[i + 1] = fmaf(a, s[i + 1], (be * k4.y) * d);
        s[i + 2] = fmaf(a, s[i + 2], (be * k4.z) * d);
        s[i + 3] = fmaf(a, s[i + 3], (be * k4.w) * d);
      }
      // o = scale (s . q)
      float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
      for (int i = 0; i < kDk; i += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(qt + i);
        o0 = fmaf(s[i], q4.x, o0);
        o1 = fmaf(s[i + 1], q4.y, o1);
        o2 = fmaf(s[i + 2], q4.z, o2);
        o3 = fmaf(s[i + 3], q4.w, o3);
      }
      const float o = p.scale * ((o0 + o1) + (o2 + o3));
      const size_t oi = ((size_t)(blk + tt) * p.Hv + hv) * kDv + c0 + lane;
      if (p.out_bf16)
        static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
      else
        static_cast<float*>(p.out)[oi] = o;
    }
    __syncwarp();  // the staging buffer is reused by the next block
  }

  // ---------------------------------------------------------------- state out
  if (p.sT) {
#pragma unroll
    for (int qd = 0; qd < 4; ++qd)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(buf + qd * 4096 + lane * 128 + ((c ^ (lane & 7)) << 4)) =
            make_float4(s[32 * qd + 4 * c], s[32 * qd + 4 * c + 1], s[32 * qd + 4 * c + 2],
                        s[32 * qd + 4 * c + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) tma_store_2d(&tm_sT, 32 * qd, row0, buf + qd * 4096);
      bulk_commit();
      bulk_wait_read<0>();  // the tile has left shared memory; the writes land by grid end
    }
  }
  if (fail && lane == 0) set_status(p.status, GDN_DEV_TIMEOUT);
}

}  // namespace

bool launch_recurrent(const RecParams& p, cudaStream_t s) {
  if (p.N <= 0) return true;
  CUtensorMap tm_s0{}, tm_sT{};
  const int rows = p.N * p.Hv * kDv;
  if (p.s0 && !encode_state_tmap(&tm_s0, p.s0, rows)) return false;
  if (p.sT && !encode_state_tmap(&tm_sT, p.sT, rows)) return false;
  recurrent_kernel<<<dim3(p.N, p.Hv, kDv / kCols), kCols, 0, s>>>(p, tm_s0, tm_sT);
  return true;
}

}  // namespace gdn
