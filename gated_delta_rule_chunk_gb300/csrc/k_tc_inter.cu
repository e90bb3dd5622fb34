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
// and every wait on those barriers is bounded (GDN_DEV_TIMEOUT on expiry).
// Data movement is TMA only: q and k tiles by tensor-map loads with the 128-byte
// swizzle, and w, M, u, G as contiguous bulk copies of images the intra kernel
// wrote in exactly this kernel's shared-memory layout. One thread issues the
// next chunk's copies into the other stage while this chunk is computed.
#include <cuda.h>

#include "gdn_common.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int BV = 32;
constexpr uint32_t kWaitIters = 1u << 22;

// One prefetch stage (bytes; 128-byte-swizzled tiles are 1024-byte aligned).
constexpr uint32_t kAQ = 0;          // [Q; w]: two dk halves of [128 rows][128 B], K-major, swizzled
constexpr uint32_t kKT = 32768;      // K^T: two dk halves of [64 tokens][128 B], MN-major, swizzled
constexpr uint32_t kAM = 49152;      // [M_hi; M_lo]: [128 rows][128 B], K-major, swizzled
constexpr uint32_t kU = 65536;       // u block: fp32 [64][32], 16-byte chunks swizzled by row
constexpr uint32_t kG = 73728;       // G [64]
constexpr uint32_t kQR = 73984;      // 1/||q|| [64] (1 when the L2 norm is off)
constexpr uint32_t kKR = 74240;      // 1/||k|| [64]
constexpr uint32_t kStage = 74752;   // 73 x 1024
// Bytes the copies of one stage deliver: q and k tiles (2 x 2 x 8 KB), w (2 x 8 KB),
// M (16 KB), u (8 KB), G (256 B).
constexpr uint32_t kStageTx = 6 * 8192 + 16384 + 8192 + 256;
// Operands written by the threads (B, MN-major, N = 32: LBO = 512, SBO = 128).
constexpr uint32_t kSBh = 2 * kStage;    // S_hi: K = dk (128)
constexpr uint32_t kSBl = kSBh + 8192;   // S_lo
constexpr uint32_t kVHh = kSBl + 8192;   // vh_hi: K = tokens (64)
constexpr uint32_t kVHl = kVHh + 4096;
constexpr uint32_t kVNh = kVHl + 4096;   // vn_hi
constexpr uint32_t kVNl = kVNh + 4096;
constexpr uint32_t kX4 = kVNl + 4096;    // fp32 [64][32]: rows 64..127 of D4 handed to warps 0-1
constexpr uint32_t kBar = kX4 + 8192;    // 4 MMA mbarriers + 2 stage mbarriers
constexpr uint32_t kMisc = kBar + 48;    // TMEM base address, abort flag
constexpr uint32_t kSmemBytes = kMisc + 16 + 1024;  // + room to align the base to 1024

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

// Swizzled position of fp32 element (r, j) of a [64][32] tile (16-byte chunk c -> c ^ (r % 8)).
__device__ __forceinline__ uint32_t u_off(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)((j >> 2) ^ (r & 7)) << 4) + (uint32_t)(j & 3) * 4u;
}

// Issued by one thread: every copy of chunk `slot` into stage `st`, counted on *full.
__device__ __forceinline__ void issue_stage(unsigned char* st, uint64_t* full, const Params& p,
                                            const CUtensorMap* tmq, const CUtensorMap* tmk,
                                            int slot, int hv, int h, int jb, int t0) {
  const size_t sl = (size_t)slot * p.Hv + hv;
  const unsigned char* wimg = static_cast<const unsigned char*>(p.w) + sl * 64 * kDk * 2;
  const unsigned char* mimg = static_cast<const unsigned char*>(p.M) + sl * 2 * 64 * 64 * 2;
  const unsigned char* uimg = reinterpret_cast<const unsigned char*>(p.u + sl * 64 * kDv);
  mbar_expect_tx(full, kStageTx);
  tma_load_3d(st + kAQ, tmq, 0, h, t0, full);
  tma_load_3d(st + kAQ + 16384, tmq, 64, h, t0, full);
  bulk_load(st + kAQ + 8192, wimg, 8192, full);
  bulk_load(st + kAQ + 16384 + 8192, wimg + 8192, 8192, full);
  tma_load_3d(st + kKT, tmk, 0, h, t0, full);
  tma_load_3d(st + kKT + 8192, tmk, 64, h, t0, full);
  bulk_load(st + kAM, mimg, 16384, full);
  bulk_load(st + kU, uimg + jb * 8192, 8192, full);
  bulk_load(st + kG, p.G + sl * 64, 256, full);
}

// Plain loads of the optional L2-norm factors of a chunk (1 when the norm is off).
__device__ __forceinline__ void load_norms(unsigned char* st, const Params& p, int h, int t0, int L,
                                           int tid) {
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

__global__ void __launch_bounds__(128, 1)
tc_inter_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
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
    for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
    mbar_init_fence();
    *abort_flag = 0;
  }
  sync_all();
  int issued = 0, waited = 0;  // stage loads issued / waited for (chunk k uses stage k & 1)
  if (nch > 0) {
    issued = 1;
    if (tid == 0) issue_stage(sm, &bars[4], p, &tmq, &tmk, sv.first_slot, hv, h, blockIdx.z, sv.start);
    load_norms(sm, p, h, sv.start, min(kChunk, sv.len), tid);
  }
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
    if (ci + 1 < nch) {  // the other stage was released at the end of chunk ci - 1
      unsigned char* nst = sm + ((ci + 1) & 1) * kStage;
      ++issued;
      if (tid == 0)
        issue_stage(nst, &bars[4 + ((ci + 1) & 1)], p, &tmq, &tmk, sv.first_slot + ci + 1, hv, h,
                    blockIdx.z, t0 + kChunk);
      load_norms(nst, p, h, t0 + kChunk, min(kChunk, sv.len - kChunk * (ci + 1)), tid);
    }
    if (!mbar_wait(&bars[4 + (ci & 1)], (ci >> 1) & 1, kWaitIters)) *abort_flag = 1;
    ++waited;
    if (L < kChunk) {  // rows past the sequence end: K^T rows are zeroed (q rows only feed unstored output)
      for (int idx = tid; idx < 2 * (kChunk - L) * 8; idx += 128) {
        const int half = idx / ((kChunk - L) * 8), rem = idx % ((kChunk - L) * 8);
        const int t = L + rem / 8, c = rem % 8;
        *reinterpret_cast<uint4*>(st + kKT + half * 8192 + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    fence_async_smem();
    sync_all();  // stage ci and the S split are visible to the tensor cores
    if (*abort_flag) break;

    if (tid == 0) {  // group 1: D1 = [Q; w] S_hi, D2 = [Q; w] S_lo
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(D1, sdesc_sw128(st_a + kAQ + (ks >> 2) * 16384 + 32 * (ks & 3), 16, 1024),
                  sdesc(sbase + kSBh + 1024 * ks, 512, 128), id_g1, ks > 0);
      umma_commit(&bars[0]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(D2, sdesc_sw128(st_a + kAQ + (ks >> 2) * 16384 + 32 * (ks & 3), 16, 1024),
                  sdesc(sbase + kSBl + 1024 * ks, 512, 128), id_g1, ks > 0);
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
      const float fac = expf(gl - G[i]) * reinterpret_cast<const float*>(st + kKR)[i];
      float vh[32];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float4 u4 = *reinterpret_cast<const float4*>(st + kU + u_off(i, 4 * a));
        x[4 * a] = u4.x - x[4 * a];  // v_new
        x[4 * a + 1] = u4.y - x[4 * a + 1];
        x[4 * a + 2] = u4.z - x[4 * a + 2];
        x[4 * a + 3] = u4.w - x[4 * a + 3];
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) vh[j] = fac * x[j];
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
        umma_bf16(D3, sdesc_sw128(st_a + kKT + 2048 * ks, 8192, 1024),
                  sdesc(sbase + kVHh + 1024 * ks, 512, 128), id_s, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D3, sdesc_sw128(st_a + kKT + 2048 * ks, 8192, 1024),
                  sdesc(sbase + kVHl + 1024 * ks, 512, 128), id_s, 1);
      umma_commit(&bars[2]);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D4, sdesc_sw128(st_a + kAM + 32 * ks, 16, 1024),
                  sdesc(sbase + kVNh + 1024 * ks, 512, 128), id_g1, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(D4, sdesc_sw128(st_a + kAM + 32 * ks, 16, 1024),
                  sdesc(sbase + kVNl + 1024 * ks, 512, 128), id_g1, 1);
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
      unsigned char* x4 = reinterpret_cast<unsigned char*>(X4);
#pragma unroll
      for (int a = 0; a < 8; ++a)
        *reinterpret_cast<float4*>(x4 + u_off(tid - 64, 4 * a)) =
            make_float4(mh[4 * a], mh[4 * a + 1], mh[4 * a + 2], mh[4 * a + 3]);
    }
    fence_async_smem();
    sync_all();  // rows 64..127 of D4 visible to warps 0-1; all MMAs of this chunk done
    if (warp < 2 && tid < L) {
      const unsigned char* x4 = reinterpret_cast<const unsigned char*>(X4);
      float o[32];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float4 l4 = *reinterpret_cast<const float4*>(x4 + u_off(tid, 4 * a));
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
  // After an early exit, give copies still in flight a bounded chance to land
  // before this CTA's shared memory is released.
  for (int k = waited; k < issued; ++k) mbar_wait(&bars[4 + (k & 1)], (k >> 1) & 1, kWaitIters);
  if (tid == 0 && *abort_flag) set_status(p.status, GDN_DEV_TIMEOUT);
  sync_all();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (p.sT) {
#pragma unroll
    for (int j = 0; j < 32; ++j) p.sT[state_base + (size_t)(c0 + j) * kDk + tid] = S[j];
  }
}

}  // namespace

bool launch_tc_inter(const Params& p, cudaStream_t s) {
  CUtensorMap tmq, tmk;
  const int rows = p.T > 0 ? p.T : 1;  // with T = 0 no tile is ever loaded
  if (!encode_rows_tmap(&tmq, p.q, rows, p.H) || !encode_rows_tmap(&tmk, p.k, rows, p.H))
    return false;
  ensure_smem_limit((const void*)tc_inter_kernel, (int)kSmemBytes);
  tc_inter_kernel<<<dim3(p.N, p.Hv, kDv / BV), 128, kSmemBytes, s>>>(p, tmq, tmk);
  return true;
}

}  // namespace gdn
