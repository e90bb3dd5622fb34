// K3, bf16 inputs: fused inter-chunk scan over [sequences, value heads, dv blocks]
// on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 5: the state
// contribution, the local-attention output and the state update are fused per
// sequence and value head, walking the chunks in order with the fp32 state
// updated in place ([sequences, Hv] chosen over [sequences, H] for
// parallelism). "Chunking Qwen3.5's gated DeltaNet ... on Apple Silicon"
// (section "How do you parallelize a recurrence for prefill?"): the value
// dimension of the state is blocked so that the tile stays on chip. A CTA owns
// 32 value columns of one (sequence, value head); thread d (0..127) holds row d
// (key dimension) of that 128x32 fp32 state in registers for the whole sequence.
//
// Per chunk (S = chunk-start state; x_hi + x_lo is a bf16 hi/lo split of fp32 x):
//   group 1 (TMEM D1, D2):  [Q; w] S_hi,  [Q; w] S_lo          (M = 128, N = 32, K = 128)
//     rows 64..127 of D1:   X = w S_hi;  v_new = u - X;  vh = exp(G_L - G) v_new
//     rows 0..63 of D1+D2:  Q S
//   group 2 (TMEM D3, D4):  K^T (vh_hi + vh_lo)                  (M = 128, N = 32, K = 64)
//                           [M_hi; M_lo] (vn_hi + vn_lo)        (M = 128, N = 32, K = 64)
//   S <- exp(G_L) S + D3;   o = scale (diag(exp(G)) Q S + D4[0:64] + D4[64:128])
// One thread issues the MMAs; tcgen05.commit arrives on an mbarrier per result,
// and every wait on those barriers is bounded (GDN_DEV_TIMEOUT on expiry). The
// next chunk's operands are prefetched with cp.async into a second stage.
// Shared-memory operands use the no-swizzle canonical layouts (umma.cuh).
#include "gdn_common.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int BV = 32;
constexpr uint32_t kWaitIters = 1u << 22;

// One prefetch stage (bytes).
constexpr uint32_t kAQ = 0;          // [Q; w]: 128 x 128 bf16, K-major (LBO 128, SBO 2048)
constexpr uint32_t kKT = 32768;      // K^T:   128 (dk) x 64 (tokens), MN-major (LBO 2048, SBO 128)
constexpr uint32_t kAM = 49152;      // [M_hi; M_lo]: 128 x 64, K-major (LBO 128, SBO 1024)
constexpr uint32_t kU = 65536;       // u block: fp32 [64][32]
constexpr uint32_t kG = 73728;       // G [64]
constexpr uint32_t kQR = 73984;      // 1/||q|| [64] (1 when the L2 norm is off)
constexpr uint32_t kKR = 74240;      // 1/||k|| [64]
constexpr uint32_t kStage = 74752;
// Operands written by the threads (B, MN-major, N = 32: LBO = 512, SBO = 128).
constexpr uint32_t kSBh = 2 * kStage;    // S_hi: K = dk (128)
constexpr uint32_t kSBl = kSBh + 8192;   // S_lo
constexpr uint32_t kVHh = kSBl + 8192;   // vh_hi: K = tokens (64)
constexpr uint32_t kVHl = kVHh + 4096;
constexpr uint32_t kVNh = kVHl + 4096;   // vn_hi
constexpr uint32_t kVNl = kVNh + 4096;
constexpr uint32_t kX4 = kVNl + 4096;    // fp32 [64][32]: rows 64..127 of D4 handed to warps 0-1
constexpr uint32_t kBar = kX4 + 8192;    // 4 mbarriers
constexpr uint32_t kMisc = kBar + 32;    // TMEM base address, abort flag
constexpr uint32_t kSmemBytes = kMisc + 16;

__device__ __forceinline__ uint32_t off_k(int r, int k, int kext) {  // K-major
  return kmajor_offset(r, k, 128u, (uint32_t)kext * 16u);
}
__device__ __forceinline__ uint32_t off_mn(int r, int k, int rext) {  // MN-major
  return mnmajor_offset(r, k, (uint32_t)rext * 16u, 128u);
}

// 8 bf16 -> 16 bytes
__device__ __forceinline__ uint4 pack8(const float* x) {
  uint4 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  u.z = pack_bf16(x[4], x[5]);
  u.w = pack_bf16(x[6], x[7]);
  return u;
}

// Write 32 fp32 values of row r (r along N = 32, MN-major B operand with K
// index k) as a bf16 hi/lo pair: 4 x 16-byte stores each.
__device__ __forceinline__ void store_row_split(unsigned char* sm, uint32_t hi_off,
                                                uint32_t lo_off, int k, const float (&x)[32]) {
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __nv_bfloat16 hb = __float2bfloat16_rn(x[8 * a + e]);
      h[e] = __bfloat162float(hb);
      l[e] = x[8 * a + e] - h[e];
    }
    const uint32_t o = off_mn(8 * a, k, BV);
    *reinterpret_cast<uint4*>(sm + hi_off + o) = pack8(h);
    *reinterpret_cast<uint4*>(sm + lo_off + o) = pack8(l);
  }
}

__device__ __forceinline__ void load_stage(unsigned char* st, const Params& p, int slot, int hv,
                                           int h, int c0, int t0, int L, int tid) {
  const size_t sl = (size_t)slot * p.Hv + hv;
  const __nv_bfloat16* wg = static_cast<const __nv_bfloat16*>(p.w) + sl * 64 * kDk;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* mg = static_cast<const __nv_bfloat16*>(p.M) + sl * 2 * 64 * 64;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int idx = tid + it * 128;  // 1024 16-byte chunks per 64 x 128 tile
    const int i = idx >> 4, c = idx & 15;
    const bool ok = i < L;
    const size_t row = ((size_t)(ok ? t0 + i : t0) * p.H + h) * kDk + 8 * c;
    cp_async16(st + kAQ + off_k(i, 8 * c, 128), qg + row, ok);             // Q rows 0..63
    cp_async16(st + kAQ + off_k(64 + i, 8 * c, 128), wg + i * kDk + 8 * c, true);  // w rows
    cp_async16(st + kKT + off_mn(8 * c, i, 128), kg + row, ok);            // K^T
    const int mi = idx >> 3, mc = idx & 7;                                 // 128 rows x 8 chunks
    cp_async16(st + kAM + off_k(mi, 8 * mc, 64), mg + mi * 64 + 8 * mc, true);
  }
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int idx = tid + it * 128;  // 512 chunks: 64 rows x 8
    const int i = idx >> 3, c = idx & 7;
    cp_async16(st + kU + (i * 32 + 4 * c) * 4, p.u + (sl * 64 + i) * kDv + c0 + 4 * c, true);
  }
  if (tid < 16) cp_async16(st + kG + 16 * tid, p.G + sl * 64 + 4 * tid, true);
  if (tid >= 64) {
    const int i = tid - 64;
    const bool ok = i < L && p.qrn;
    reinterpret_cast<float*>(st + kQR)[i] = ok ? p.qrn[(size_t)(t0 + i) * p.H + h] : 1.f;
    reinterpret_cast<float*>(st + kKR)[i] = ok ? p.krn[(size_t)(t0 + i) * p.H + h] : 1.f;
  }
}

__device__ __forceinline__ void sync_all() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__global__ void __launch_bounds__(128, 1) tc_inter_kernel(Params p) {
  extern __shared__ __align__(1024) unsigned char sm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * BV;
  const int h = hv / p.HG;
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }
  const size_t state_base = ((size_t)n * p.Hv + hv) * kDv * kDk;

  // Thread d = tid owns state row d (key dimension), 32 value columns.
  float S[32];
#pragma unroll
  for (int j = 0; j < 32; ++j)
    S[j] = p.s0 ? p.s0[state_base + (size_t)(c0 + j) * kDk + tid] : 0.f;
  store_row_split(sm, kSBh, kSBl, tid, S);

  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 4; ++b) mbar_init(&bars[b], 1);
    mbar_init_fence();
    *abort_flag = 0;
  }
  if (nch > 0) load_stage(sm, p, sv.first_slot, hv, h, c0, sv.start, min(kChunk, sv.len), tid);
  cp_async_commit();
  sync_all();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const uint32_t D1 = tmem, D2 = tmem + 32, D3 = tmem + 64, D4 = tmem + 96;
  const uint32_t id_g1 = idesc_bf16_f32(128, BV, false, true);
  const uint32_t id_s = idesc_bf16_f32(128, BV, true, true);
  const uint32_t sbase = smem_addr(sm);
  float* X4 = reinterpret_cast<float*>(sm + kX4);

  for (int ci = 0; ci < nch; ++ci) {
    const uint32_t ph = ci & 1;
    unsigned char* st = sm + (ci & 1) * kStage;
    const uint32_t st_a = sbase + (ci & 1) * kStage;
    const int t0 = sv.start + kChunk * ci;
    const int L = min(kChunk, sv.len - kChunk * ci);
    if (ci + 1 < nch)
      load_stage(sm + ((ci + 1) & 1) * kStage, p, sv.first_slot + ci + 1, hv, h, c0,
                 t0 + kChunk, min(kChunk, sv.len - kChunk * (ci + 1)), tid);
    cp_async_commit();
    cp_async_wait<1>();
    fence_async_smem();
    sync_all();  // stage ci and the S split are visible to the tensor cores
    if (*abort_flag) break;

    if (tid == 0) {  // group 1: D1 = [Q; w] S_hi, D2 = [Q; w] S_lo
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(D1, sdesc(st_a + kAQ + 256 * ks, 128, 2048), sdesc(sbase + kSBh + 1024 * ks, 512, 128),
                  id_g1, ks > 0);
      umma_commit(&bars[0]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(D2, sdesc(st_a + kAQ + 256 * ks, 128, 2048), sdesc(sbase + kSBl + 1024 * ks, 512, 128),
                  id_g1, ks > 0);
      umma_commit(&bars[1]);
    }
    const float* G = reinterpret_cast<const float*>(st + kG);
    const float gl = G[63];
    float qs[32];
    if (warp >= 2) {  // chain: token row i = tid - 64
      const int i = tid - 64;
      if (!mbar_wait(&bars[0], ph, kWaitIters)) *abort_flag = 1;
      tc_fence_after();
      float x[32];
      tmem_ld32(D1 + lane_base, x);
      tmem_ld_wait();
      const float* U = reinterpret_cast<const float*>(st + kU) + i * 32;
      const float fac = expf(gl - G[i]) * reinterpret_cast<const float*>(st + kKR)[i];
      float vh[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = U[j] - x[j];  // v_new
        vh[j] = fac * x[j];
      }
      store_row_split(sm, kVNh, kVNl, i, x);
      store_row_split(sm, kVHh, kVHl, i, vh);
    } else {  // output rows i = tid: Q S = D1 + D2
      if (!mbar_wait(&bars[1], ph, kWaitIters)) *abort_flag = 1;
      tc_fence_after();
      float a[32];
      tmem_ld32(D1 + lane_base, qs);
      tmem_ld32(D2 + lane_base, a);
      tmem_ld_wait();
      const float e = expf(G[tid]) * reinterpret_cast<const float*>(st + kQR)[tid];
#pragma unroll
      for (int j = 0; j < 32; ++j) qs[j] = (qs[j] + a[j]) * e;
    }
    fence_async_smem();
    sync_all();  // v_new / vh tiles visible to the tensor cores

    if (tid == 0) {  // group 2: D3 = K^T (vh_hi + vh_lo), D4 = [M_hi; M_lo] (vn_hi + vn_lo)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D3, sdesc(st_a + kKT + 4096 * ks, 2048, 128), sdesc(sbase + kVHh + 1024 * ks, 512, 128),
                  id_s, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D3, sdesc(st_a + kKT + 4096 * ks, 2048, 128), sdesc(sbase + kVHl + 1024 * ks, 512, 128),
                  id_s, 1);
      umma_commit(&bars[2]);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D4, sdesc(st_a + kAM + 256 * ks, 128, 1024), sdesc(sbase + kVNh + 1024 * ks, 512, 128),
                  id_g1, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D4, sdesc(st_a + kAM + 256 * ks, 128, 1024), sdesc(sbase + kVNl + 1024 * ks, 512, 128),
                  id_g1, 1);
      umma_commit(&bars[3]);
    }
    // S <- exp(G_L) S + K^T vh (row tid), then its split for the next chunk
    {
      if (!mbar_wait(&bars[2], ph, kWaitIters)) *abort_flag = 1;
      tc_fence_after();
      float inc[32];
      tmem_ld32(D3 + lane_base, inc);
      tmem_ld_wait();
      const float gam = expf(gl);
#pragma unroll
      for (int j = 0; j < 32; ++j) S[j] = fmaf(gam, S[j], inc[j]);
      store_row_split(sm, kSBh, kSBl, tid, S);
    }
    float mh[32];
    if (!mbar_wait(&bars[3], ph, kWaitIters)) *abort_flag = 1;
    tc_fence_after();
    tmem_ld32(D4 + lane_base, mh);
    tmem_ld_wait();
    if (warp >= 2) {
      float4* dst = reinterpret_cast<float4*>(X4 + (tid - 64) * 32);
#pragma unroll
      for (int a = 0; a < 8; ++a) dst[a] = make_float4(mh[4 * a], mh[4 * a + 1], mh[4 * a + 2], mh[4 * a + 3]);
    }
    fence_async_smem();
    sync_all();  // rows 64..127 of D4 visible to warps 0-1; all MMAs of this chunk done
    if (warp < 2 && tid < L) {
      const float4* lo = reinterpret_cast<const float4*>(X4 + tid * 32);
      float o[32];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float4 l4 = lo[a];
        o[4 * a] = p.scale * (qs[4 * a] + mh[4 * a] + l4.x);
        o[4 * a + 1] = p.scale * (qs[4 * a + 1] + mh[4 * a + 1] + l4.y);
        o[4 * a + 2] = p.scale * (qs[4 * a + 2] + mh[4 * a + 2] + l4.z);
        o[4 * a + 3] = p.scale * (qs[4 * a + 3] + mh[4 * a + 3] + l4.w);
      }
      const size_t oi = ((size_t)(t0 + tid) * p.Hv + hv) * kDv + c0;
      if (p.out_bf16) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + oi);
#pragma unroll
        for (int a = 0; a < 4; ++a) dst[a] = pack8(o + 8 * a);
      } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi);
#pragma unroll
        for (int a = 0; a < 8; ++a) dst[a] = make_float4(o[4 * a], o[4 * a + 1], o[4 * a + 2], o[4 * a + 3]);
      }
    }
  }
  cp_async_wait<0>();
  if (tid == 0 && *abort_flag) set_status(p.status, GDN_DEV_TIMEOUT);
  sync_all();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (p.sT) {
#pragma unroll
    for (int j = 0; j < 32; ++j) p.sT[state_base + (size_t)(c0 + j) * kDk + tid] = S[j];
  }
}

}  // namespace

void launch_tc_inter(const Params& p, cudaStream_t s) {
  ensure_smem_limit((const void*)tc_inter_kernel, (int)kSmemBytes);
  tc_inter_kernel<<<dim3(p.N, p.Hv, kDv / BV), 128, kSmemBytes, s>>>(p);
}

}  // namespace gdn
