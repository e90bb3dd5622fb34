// K3, bf16 inputs: fused inter-chunk scan over [sequences, value heads, dv blocks].
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 5: the state
// contribution, the local-attention output and the state update are fused per
// sequence and value head, walking the chunks in order with the fp32 state
// updated in place ([sequences, Hv] chosen over [sequences, H] for
// parallelism). "Chunking Qwen3.5's gated DeltaNet ... on Apple Silicon"
// (section "How do you parallelize a recurrence for prefill?"): the value
// dimension of the state is blocked so that the tile stays on chip. A CTA owns
// 32 value columns of one (sequence, value head) for the whole sequence.
//
// Per chunk (S = chunk-start state; x_hi + x_lo is a bf16 hi/lo split of fp32 x):
//   chain (serial):   X = w S_hi;  v_new = u - X;  vh = exp(G_L - G) v_new
//                     S <- exp(G_L) S + K^T vh
//   output (off the chain):
//                     o = scale (diag(exp(G)) Q (S_hi + S_lo) + (M_hi + M_lo)(vn_hi + vn_lo))
//
// Warp roles (15 warps):
//   * 8 chain warps run the serial recurrence on warp-level MMAs (lowest latency
//     per dependent step); the state lives in their registers as fp32 MMA
//     accumulators (warp w owns key rows 16w..16w+15). The state-update product
//     uses fp16 operands (k as written by the intra kernel, vh rounded once), which
//     keeps about 11 significant bits where bf16 would keep 8.
//   * 1 load warp issues every TMA copy (the q tile by tensor map with the 128-byte
//     swizzle; w, M, u, G and the fp16 k tile as bulk copies of images the intra
//     kernel wrote in this kernel's layout).
//   * 2 MMA warps (one thread each) issue the output MMAs on the 5th-generation
//     tensor cores: D_QS = Q [S_hi | S_lo] and D_M = M_hi [vn_hi | vn_lo] +
//     M_lo [vn_hi | vn_lo] (M = 64, N = 64, fp32 accumulators in TMEM, double-buffered
//     per chunk; the two column halves are summed when the output is formed). What
//     the chain reads (w, fp16 k, u, G) streams through a 3-slot ring so that each
//     chunk's copies are issued two chunks ahead; q (double-buffered) and M (one
//     buffer, refilled once the previous chunk's D_M is complete) feed only the
//     output MMAs.
//   * 4 output warps (one per TMEM lane quarter; rows 16q..16q+15 of an M = 64
//     result sit in lanes 32q..32q+15) finish chunk c's output while the chain
//     works on chunk c + 1.
//
// Per-channel gates (template parameter CH): the state's key row d decays by
// exp(G_L) of channel d; the state update's k operand is the value head's
// exp(G_L - G) * k image (so v_new needs no row factor); the output operand is
// exp(G) * q as a bf16 hi/lo pair written by the per-channel intra kernel (D_QS gains
// a q_lo [S_hi | S_lo] pass and the output needs no row factor); to make room for the
// hi/lo q buffers the ring has two slots instead of three.
// Hand-offs use mbarriers; every wait is bounded (GDN_DEV_TIMEOUT on expiry).
#include <cuda.h>

#include "gdn_common.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int BV = 32;
constexpr uint32_t kWaitIters = 1u << 22;
constexpr int kChainWarps = 8;
constexpr int kOutWarps = 4;
constexpr int kLoadWarp = kChainWarps + kOutWarps;
constexpr int kQsWarp = kLoadWarp + 1;  // issues D_QS; owns the TMEM allocation
constexpr int kMWarp = kQsWarp + 1;     // issues D_M
constexpr int kThreads = (kMWarp + 1) * 32;
constexpr int kChainThreads = kChainWarps * 32;

// Ring slot of the chain's operands (bytes; 128-byte-swizzled tiles are 1024-byte aligned).
constexpr uint32_t kW = 0;           // w: two dk halves of [64 rows][128 B], K-major, swizzled
constexpr uint32_t kK = 16384;       // k (fp16 image): two dk halves of [64 tokens][128 B], swizzled
constexpr uint32_t kU = 32768;       // u block: fp32 [64][32], 16-byte chunks swizzled by row
constexpr uint32_t kG = 40960;       // G [64] (per-channel mode: exp(G_L) [128])
constexpr uint32_t kSlot = 41984;    // 41 x 1024
constexpr uint32_t kSBsz = 16384;
constexpr uint32_t kVNsz = 8192;

// The rest of the layout depends on the gate kind. Per-channel gates: the q operand is
// the decayed q as a bf16 hi/lo pair (two 16 KB images per buffer), which the ring's
// third slot makes room for.
template <bool CH>
struct Lay {
  static constexpr int kRing = CH ? 2 : 3;
  static constexpr uint32_t kTxRing = 2 * 8192 + 16384 + 8192 + (CH ? 512 : 256);  // w, k, u, G
  // q (two buffers of two swizzled [64 rows][128 B] key-dim halves; hi then lo with
  // per-channel gates) and [M_hi; M_lo] ([128 rows][128 B], swizzled) for the output MMAs.
  static constexpr uint32_t kQ = kRing * kSlot;
  static constexpr uint32_t kQsz = CH ? 32768 : 16384;
  static constexpr uint32_t kM = kQ + 2 * kQsz;
  // Operands written by the threads (no-swizzle MN-major core matrices: the K
  // group stride is the descriptor's lbo, sbo = 128 along N).
  static constexpr uint32_t kSB = kM + 16384;       // 2 x [S_hi | S_lo]: N = 64, K = 128
  static constexpr uint32_t kVN = kSB + 2 * kSBsz;  // 2 x [vn_hi | vn_lo]: N = 64, K = 64
  static constexpr uint32_t kVH = kVN + 2 * kVNsz;  // vh (fp16): N = 32, K = 64 (tokens)
  static constexpr uint32_t kBar = kVH + 4096;      // 19 mbarriers
  static constexpr uint32_t kMisc = kBar + 256;     // TMEM base address, abort flag
  static constexpr uint32_t kSmemBytes = kMisc + 16 + 1024;  // + room to align the base
};
static_assert(Lay<true>::kSmemBytes <= 232448 && Lay<false>::kSmemBytes <= 232448,
              "shared memory over the per-CTA limit");

// mbarrier indices. Ring barriers: chunk c uses slot c % 3 with parity (c / 3) & 1;
// double-buffered barriers: index + (c & 1) with parity (c >> 1) & 1; B_MF: one
// completion per chunk, parity c & 1.
constexpr int B_FULL = 0;   // ring slot of chunk c landed (transaction count)
constexpr int B_CD = 3;     // chain warps done reading the ring slot of chunk c (per chain warp)
constexpr int B_QF = 6;     // q of chunk c landed
constexpr int B_MF = 8;     // M of chunk c landed
constexpr int B_XD = 9;     // chain warps finished X of chunk c (one arrival per chain warp);
                            // each had written the S split of chunk c before
constexpr int B_QSD = 11;   // D_QS of chunk c complete (tcgen05.commit)
constexpr int B_MD = 13;    // D_M of chunk c complete (tcgen05.commit)
constexpr int B_OD = 15;    // output warps done with the TMEM buffer of chunk c (per output warp)
constexpr int kNumBars = 17;
constexpr uint32_t kTmemCols = 256;

// Byte offset of (n, k) in a no-swizzle MN-major tile with `kgrp` bytes per 8-deep K group.
__device__ __forceinline__ uint32_t mn_off(int n, int k, uint32_t kgrp) {
  return (uint32_t)(n >> 3) * 128u + (uint32_t)(k >> 3) * kgrp + (uint32_t)(k & 7) * 16u +
         (uint32_t)(n & 7) * 2u;
}
// Byte offset of the 16-byte chunk holding element (row, col) of a [rows][128 B] swizzled tile.
__device__ __forceinline__ uint32_t sw_chunk(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)((col >> 3) ^ (row & 7)) << 4);
}
// Swizzled position of fp32 element (r, j) of a [64][32] tile (16-byte chunk c -> c ^ (r % 8)).
__device__ __forceinline__ uint32_t u_off(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)((j >> 2) ^ (r & 7)) << 4) + (uint32_t)(j & 3) * 4u;
}

__device__ __forceinline__ uint4 pack8_bf16(const float* x) {
  uint4 u;
  u.x = pack_bf16(x[0], x[1]);
  u.y = pack_bf16(x[2], x[3]);
  u.z = pack_bf16(x[4], x[5]);
  u.w = pack_bf16(x[6], x[7]);
  return u;
}

// Wait for chunk c's phase of double-buffered barrier `base`. Gives up after a
// bounded number of polls (raising the abort flag), and at once when the flag is
// already raised, so that after a failure every role runs through its remaining
// iterations without waiting and the CTA's barriers stay consistent.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity,
                                           volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitIters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ bool wait_chunk(uint64_t* bars, int base, int c,
                                           volatile int* abort_flag) {
  return wait_phase(&bars[base + (c & 1)], (uint32_t)((c >> 1) & 1), abort_flag);
}
template <int kRing>
__device__ __forceinline__ bool wait_ring(uint64_t* bars, int base, int c,
                                          volatile int* abort_flag) {
  return wait_phase(&bars[base + c % kRing], (uint32_t)((c / kRing) & 1), abort_flag);
}

// Issued by one thread: the chain's copies of chunk `slot` into ring slot `st`. The k
// image is per key head with a scalar gate and per value head with per-channel gates
// (the decay is inside it); G is the in-chunk gate sum, or exp(G_L) per channel.
template <bool CH>
__device__ __forceinline__ void issue_ring(unsigned char* st, uint64_t* full, const Params& p,
                                           int slot, int hv, int h, int jb) {
  const size_t sl = (size_t)slot * p.Hv + hv;
  const unsigned char* wimg = static_cast<const unsigned char*>(p.w) + sl * 64 * kDk * 2;
  const unsigned char* uimg = reinterpret_cast<const unsigned char*>(p.u + sl * 64 * kDv);
  const unsigned char* kimg = static_cast<const unsigned char*>(p.k16) +
                              (CH ? sl : (size_t)slot * p.H + h) * 64 * kDk * 2;
  mbar_expect_tx(full, Lay<CH>::kTxRing);
  bulk_load(st + kW, wimg, 16384, full);
  bulk_load(st + kK, kimg, 16384, full);
  bulk_load(st + kU, uimg + jb * 8192, 8192, full);
  if (CH)
    bulk_load(st + kG, p.gam + sl * 128, 512, full);
  else
    bulk_load(st + kG, p.G + sl * 64, 256, full);
}

// Issued by one thread: chunk c's q operand. Scalar gate: the two key-dim halves of the
// q tile (rows t0..t0+63) by tensor map; per-channel gates: the decayed q's hi and lo
// images the intra kernel wrote for (slot, value head).
template <bool CH>
__device__ __forceinline__ void issue_q(unsigned char* dst, uint64_t* full, const CUtensorMap* tmq,
                                        const Params& p, int h, int t0, int slot, int hv) {
  if (CH) {
    mbar_expect_tx(full, 32768);
    bulk_load(dst, static_cast<const unsigned char*>(p.qimg) + ((size_t)slot * p.Hv + hv) * 32768,
              32768, full);
  } else {
    mbar_expect_tx(full, 2 * 8192);
    tma_load_3d(dst, tmq, 0, h, t0, full);
    tma_load_3d(dst + 8192, tmq, 64, h, t0, full);
  }
}
// Issued by one thread: the [M_hi; M_lo] image of chunk `slot`.
__device__ __forceinline__ void issue_m(unsigned char* dst, uint64_t* full, const Params& p,
                                        int slot, int hv) {
  const size_t sl = (size_t)slot * p.Hv + hv;
  mbar_expect_tx(full, 16384);
  bulk_load(dst, static_cast<const unsigned char*>(p.M) + sl * 2 * 64 * 64 * 2, 16384, full);
}

template <bool CH>
__global__ void __launch_bounds__(kThreads, 1)
tc_inter_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmq) {
  using LY = Lay<CH>;
  constexpr int kRing = LY::kRing;
  constexpr uint32_t kQ = LY::kQ, kQsz = LY::kQsz, kM = LY::kM, kSB = LY::kSB, kVN = LY::kVN,
                     kVH = LY::kVH, kBar = LY::kBar, kMisc = LY::kMisc;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x, hv = blockIdx.y, jb = blockIdx.z, c0 = jb * BV;
  const int h = hv / p.HG;
  const size_t state_base = ((size_t)n * p.Hv + hv) * p.D * p.D;  // key rows >= D are padding
  const uint32_t sbase = smem_addr(sm);
  const int g = lane >> 2, c2 = 2 * (lane & 3);

  if (warp == kQsWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) {
      const bool per_chain = (b >= B_CD && b < B_QF) || (b >= B_XD && b < B_QSD);  // CD, XD
      mbar_init(&bars[b], per_chain ? kChainWarps : (b >= B_OD ? kOutWarps : 1));
    }
    mbar_init_fence();
    *abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // everything below reads what the chunk-table and intra kernels wrote
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }

  if (warp < kChainWarps) {
    // ------------------------------------------------------------------ chain
    // State rows 16*warp + g (+8), columns 8*nt + c2 (+1), as MMA accumulators.
    float S[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
        S[nt][e] = (p.s0 && d < p.D) ? p.s0[state_base + (size_t)(c0 + j) * p.D + d] : 0.f;
      }
    const int mt = warp & 3, np = warp >> 2;  // X tile: token rows 16mt.., columns 16np..
    auto store_split_state = [&](int buf) {
      unsigned char* sb = sm + kSB + buf * kSBsz;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int d = 16 * warp + g + 8 * hh, j = 8 * nt + c2;
          const float x0 = S[nt][2 * hh], x1 = S[nt][2 * hh + 1];
          const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
          const float2 hf = __bfloat1622float2(hi);
          *reinterpret_cast<__nv_bfloat162*>(sb + mn_off(j, d, 1024)) = hi;
          *reinterpret_cast<uint32_t*>(sb + mn_off(32 + j, d, 1024)) =
              pack_bf16(x0 - hf.x, x1 - hf.y);
        }
      fence_async_smem();
      __syncwarp();
    };
    if (nch > 0) store_split_state(0);
    named_sync(1, kChainThreads);
    for (int c = 0; c < nch; ++c) {
      const int b = c & 1;
      unsigned char* st = sm + (c % kRing) * kSlot;
      const uint32_t st_a = sbase + (c % kRing) * kSlot;
      wait_ring<kRing>(bars, B_FULL, c, abort_flag);
      // Row factors of this chunk, formed before X so that their latency hides under its
      // MMAs: exp(G_L - G_i) of this thread's two v_new rows (per-channel gates: inside the
      // k image) and the state decay of its two key rows (exp(G_L), or per channel).
      float fac[2], gam0, gam1;
      {
        const float* gst = reinterpret_cast<const float*>(st + kG);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          fac[hh] = CH ? 1.f : expf(gst[63] - gst[16 * (warp & 3) + g + 8 * hh]);
        gam0 = CH ? gst[16 * warp + g] : expf(gst[63]);
        gam1 = CH ? gst[16 * warp + g + 8] : gam0;
      }
      if (p.hs) {  // chunk-start state, [dv][dk] rows of the slot (the backward's recompute)
        float* hs = p.hs + ((size_t)(sv.first_slot + c) * p.Hv + hv) * p.D * p.D;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
            if (d < p.D) hs[(size_t)(c0 + j) * p.D + d] = S[nt][e];
          }
      }

      // X = w S_hi: token rows 16mt.., columns 16np..16np+15
      float xa[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) xa[q][e] = 0.f;
      const uint32_t sbb = sbase + kSB + b * kSBsz;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4], bb[4];
        const int i = lane >> 3;
        {
          const int row = 16 * mt + (lane & 7) + (i & 1) * 8;
          const int col = (16 * ks + (i >> 1) * 8) & 63;
          ldsm_x4_addr(a, st_a + kW + (ks >> 2) * 8192 + sw_chunk(row, col));
        }
        {
          const int nn = 16 * np + (i >> 1) * 8, kk = 16 * ks + (i & 1) * 8;
          ldsm_x4_t_addr(bb, sbb + (uint32_t)(nn >> 3) * 128u + (uint32_t)(kk >> 3) * 1024u +
                                 (uint32_t)(lane & 7) * 16u);
        }
        mma_bf16(xa[0], a, bb[0], bb[1]);
        mma_bf16(xa[1], a, bb[2], bb[3]);
      }
      // The output MMAs share the tensor datapath with the warp MMAs: D_QS of chunk c is
      // issued now and runs while the chain forms v_new (no MMAs there).
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_XD + b]);
      // v_new = u - X; vn (bf16 hi|lo) for the output MMA; vh (fp16) for the state update.
      if (c >= 2) wait_chunk(bars, B_MD, c - 2, abort_flag);  // vn buffer b no longer read
      {
        unsigned char* vn = sm + kVN + b * kVNsz;
        unsigned char* vhb = sm + kVH;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 16 * mt + g + 8 * hh;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int j = 16 * np + 8 * q + c2;
            const float2 u2 = *reinterpret_cast<const float2*>(st + kU + u_off(i, j));
            const float v0 = u2.x - xa[q][2 * hh], v1 = u2.y - xa[q][2 * hh + 1];
            if (p.vn_out)  // v_new of the chunk (the backward's recompute)
              *reinterpret_cast<float2*>(
                  p.vn_out + (((size_t)(sv.first_slot + c) * p.Hv + hv) * 64 + i) * p.D + c0 + j) =
                  make_float2(v0, v1);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v0, v1);
            const float2 hf = __bfloat1622float2(hi);
            *reinterpret_cast<__nv_bfloat162*>(vn + mn_off(j, i, 1024)) = hi;
            *reinterpret_cast<uint32_t*>(vn + mn_off(32 + j, i, 1024)) =
                pack_bf16(v0 - hf.x, v1 - hf.y);
            *reinterpret_cast<uint32_t*>(vhb + mn_off(j, i, 512)) = pack_f16(fac[hh] * v0, fac[hh] * v1);
          }
        }
      }
      fence_async_smem();  // vn visible to the tensor cores once this warp arrives on B_CD
      named_sync(1, kChainThreads);  // vh visible to every chain warp

      // S <- exp(G_L) S + K^T vh   (key rows 16*warp.., all 32 columns; fp16 operands)
      {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[nt][e] *= (e >> 1) ? gam1 : gam0;
        const uint32_t kt = st_a + kK + (warp >> 2) * 8192;
        const uint32_t vhb = sbase + kVH;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4];
          const int i = lane >> 3;
          {
            const int t = 16 * ks + (i >> 1) * 8 + (lane & 7);
            const int col = 16 * (warp & 3) + (i & 1) * 8;
            ldsm_x4_t_addr(a, kt + sw_chunk(t, col));
          }
#pragma unroll
          for (int p2 = 0; p2 < 2; ++p2) {
            uint32_t bb[4];
            const int nn = 16 * p2 + (i >> 1) * 8, kk = 16 * ks + (i & 1) * 8;
            ldsm_x4_t_addr(bb, vhb + (uint32_t)(nn >> 3) * 128u + (uint32_t)(kk >> 3) * 512u +
                                   (uint32_t)(lane & 7) * 16u);
            mma_f16(S[2 * p2], a, bb[0], bb[1]);
            mma_f16(S[2 * p2 + 1], a, bb[2], bb[3]);
          }
        }
      }
      // Ring slot of chunk c released; vn of chunk c complete. D_M of chunk c runs while
      // the chain stores the split of the next state (no MMAs there).
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_CD + c % kRing]);
      // split of S_{c+1} for the next chunk (its buffer was last read by D_QS of chunk c - 1)
      if (c + 1 < nch) {
        if (c >= 1) wait_chunk(bars, B_QSD, c - 1, abort_flag);
        store_split_state((c + 1) & 1);
      }
      named_sync(1, kChainThreads);  // new split visible; vh may be rewritten
    }
    if (p.sT) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
          if (d < p.D) p.sT[state_base + (size_t)(c0 + j) * p.D + d] = S[nt][e];
        }
    }
  } else if (warp < kLoadWarp) {
    // ------------------------------------------------------------------ output
    const int qd = warp - kChainWarps;  // TMEM lane quarter
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const int i = 16 * qd + (lane & 15);  // token row of this lane (lanes 16..31 idle)
    for (int c = 0; c < nch; ++c) {
      const int b = c & 1;
      const int t0 = sv.start + kChunk * c;
      const int L = min(kChunk, sv.len - kChunk * c);
      // row factor exp(G_i) / ||q_i|| straight from global memory (off the critical path)
      const size_t sl = (size_t)(sv.first_slot + c) * p.Hv + hv;
      // exp(G_i) / ||q_i|| (per-channel gates: both are inside the q operand)
      const float grow = CH ? 0.f : p.G[sl * 64 + i];
      const float qrow = (!CH && p.qrn && i < L) ? p.qrn[(size_t)(t0 + i) * p.H + h] : 1.f;
      wait_chunk(bars, B_QSD, c, abort_flag);
      wait_chunk(bars, B_MD, c, abort_flag);
      tc_fence_after();
      const uint32_t dq = tmem + b * 128 + lane_base, dm = dq + 64;
      float m[32], qs[32], t[32];
      tmem_ld32(dm, m);
      tmem_ld32(dm + 32, t);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) m[j] += t[j];  // M (vn_hi + vn_lo)
      tmem_ld32(dq, qs);
      tmem_ld32(dq + 32, t);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) qs[j] += t[j];  // Q (S_hi + S_lo)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_OD + b]);
      if (p.out && lane < 16 && i < L) {  // (no output when only the states are wanted)
        const float e = expf(grow) * qrow;
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = p.scale * (e * qs[j] + m[j]);
        const size_t oi = ((size_t)(t0 + i) * p.Hv + hv) * p.D + c0;
        if (p.out_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + oi);
#pragma unroll
          for (int a = 0; a < 4; ++a) dst[a] = pack8_bf16(o + 8 * a);
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi);
#pragma unroll
          for (int a = 0; a < 8; ++a)
            dst[a] = make_float4(o[4 * a], o[4 * a + 1], o[4 * a + 2], o[4 * a + 3]);
        }
      }
    }
  } else if (warp == kLoadWarp && lane == 0) {
    // ------------------------------------------------------------------ loads
    // ring chunks issued, q tiles issued, M tiles issued
    int issued = 0, q_issued = 0, m_issued = 0;
    for (int k = 0; k < min(nch, kRing - 1); ++k) {
      issue_ring<CH>(sm + k * kSlot, &bars[B_FULL + k], p, sv.first_slot + k, hv, h, jb);
      issued = k + 1;
    }
    for (int k = 0; k < min(nch, 2); ++k) {
      issue_q<CH>(sm + kQ + k * kQsz, &bars[B_QF + k], &tmq, p, h, sv.start + kChunk * k,
                  sv.first_slot + k, hv);
      q_issued = k + 1;
    }
    if (nch > 0) {
      issue_m(sm + kM, &bars[B_MF], p, sv.first_slot, hv);
      m_issued = 1;
    }
    for (int c = 0; c < nch; ++c) {
      if (*abort_flag) break;
      if (c + kRing - 1 < nch) {  // ring slot of chunk c - 1 is free once the chain released it
        if (c >= 1 && !wait_ring<kRing>(bars, B_CD, c - 1, abort_flag)) break;
        const int cn = c + kRing - 1;
        issue_ring<CH>(sm + (cn % kRing) * kSlot, &bars[B_FULL + cn % kRing], p,
                       sv.first_slot + cn, hv, h, jb);
        issued = cn + 1;
      }
      // q buffer of chunk c - 1 is free once its D_QS completed
      if (c >= 1 && c + 1 < nch) {
        if (!wait_chunk(bars, B_QSD, c - 1, abort_flag)) break;
        issue_q<CH>(sm + kQ + ((c + 1) & 1) * kQsz, &bars[B_QF + ((c + 1) & 1)], &tmq, p, h,
                    sv.start + kChunk * (c + 1), sv.first_slot + c + 1, hv);
        q_issued = c + 2;
      }
      // M is free once chunk c's D_M completed
      if (c + 1 < nch) {
        if (!wait_chunk(bars, B_MD, c, abort_flag)) break;
        issue_m(sm + kM, &bars[B_MF], p, sv.first_slot + c + 1, hv);
        m_issued = c + 2;
      }
    }
    // Before the CTA retires: every copy this thread issued has landed (bounded waits).
    for (int k = max(0, issued - kRing); k < issued; ++k)
      mbar_wait(&bars[B_FULL + k % kRing], (uint32_t)((k / kRing) & 1), kWaitIters);
    for (int k = max(0, q_issued - 2); k < q_issued; ++k)
      mbar_wait(&bars[B_QF + (k & 1)], (uint32_t)((k >> 1) & 1), kWaitIters);
    if (m_issued > 0) mbar_wait(&bars[B_MF], (uint32_t)((m_issued - 1) & 1), kWaitIters);
  } else if (warp == kQsWarp && lane == 0) {
    // ------------------------------------------------------------------ D_QS
    // D_QS of chunk c = Q [S_hi | S_lo]; issued once the chain finished X of chunk c,
    // so that it runs while the chain forms v_new (the output MMAs share the tensor
    // datapath with the warp MMAs of the chain).
    const uint32_t id_o = idesc_bf16_f32(64, 64, false, true);
    int committed = 0;
    for (int c = 0; c < nch; ++c) {
      const int b = c & 1;
      if (*abort_flag) break;
      wait_chunk(bars, B_QF, c, abort_flag);
      wait_chunk(bars, B_XD, c, abort_flag);
      if (c >= 2) wait_chunk(bars, B_OD, c - 2, abort_flag);
      tc_fence_after();
      const uint32_t q_a = sbase + kQ + b * kQsz;
      const uint32_t sbb = sbase + kSB + b * kSBsz;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tmem + b * 128, sdesc_sw128(q_a + (ks >> 2) * 8192 + 32 * (ks & 3), 16, 1024),
                  sdesc(sbb + 2048 * ks, 1024, 128), id_o, ks > 0);
      if (CH) {  // + q_lo [S_hi | S_lo]: the decayed q is a hi/lo pair
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tmem + b * 128,
                    sdesc_sw128(q_a + 16384 + (ks >> 2) * 8192 + 32 * (ks & 3), 16, 1024),
                    sdesc(sbb + 2048 * ks, 1024, 128), id_o, true);
      }
      umma_commit(&bars[B_QSD + b]);
      committed = c + 1;
    }
    // Before the CTA retires: every MMA this thread issued has completed (bounded wait).
    if (committed > 0)
      mbar_wait(&bars[B_QSD + ((committed - 1) & 1)], (uint32_t)(((committed - 1) >> 1) & 1),
                kWaitIters);
  } else if (warp == kMWarp && lane == 0) {
    // ------------------------------------------------------------------ D_M
    // D_M of chunk c = M_hi [vn_hi | vn_lo] + M_lo [vn_hi | vn_lo]; issued once the
    // chain finished the state update of chunk c, so that it runs while the chain
    // stores the split of the next state.
    const uint32_t id_o = idesc_bf16_f32(64, 64, false, true);
    const uint32_t m_a = sbase + kM;
    int committed = 0;
    for (int c = 0; c < nch; ++c) {
      const int b = c & 1;
      if (*abort_flag) break;
      wait_phase(&bars[B_MF], (uint32_t)(c & 1), abort_flag);
      wait_ring<kRing>(bars, B_CD, c, abort_flag);
      if (c >= 2) wait_chunk(bars, B_OD, c - 2, abort_flag);
      tc_fence_after();
      const uint32_t vnb = sbase + kVN + b * kVNsz;
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tmem + b * 128 + 64, sdesc_sw128(m_a + 8192 * part + 32 * ks, 16, 1024),
                    sdesc(vnb + 2048 * ks, 1024, 128), id_o, part > 0 || ks > 0);
      umma_commit(&bars[B_MD + b]);
      committed = c + 1;
    }
    if (committed > 0)
      mbar_wait(&bars[B_MD + ((committed - 1) & 1)], (uint32_t)(((committed - 1) >> 1) & 1),
                kWaitIters);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && *abort_flag) set_status(p.status, GDN_DEV_TIMEOUT);
  if (warp == kQsWarp) tmem_dealloc(tmem, kTmemCols);
}

template <bool CH>
bool launch_tc_inter_t(const Params& p, cudaStream_t s) {
  CUtensorMap tmq;
  const int rows = p.T > 0 ? p.T : 1;  // with T = 0 no tile is ever loaded
  if (!encode_rows_tmap(&tmq, p.q, rows, p.H, p.D)) return false;
  constexpr uint32_t smem = Lay<CH>::kSmemBytes;
  ensure_smem_limit((const void*)tc_inter_kernel<CH>, (int)smem);
  return launch_pdl(tc_inter_kernel<CH>, dim3(p.N, p.Hv, p.D / BV), dim3(kThreads), smem, s, p,
                    tmq) == cudaSuccess;
}

}  // namespace

bool launch_tc_inter(const Params& p, bool channel_gates, cudaStream_t s) {
  return channel_gates ? launch_tc_inter_t<true>(p, s) : launch_scan(p, s);
}

}  // namespace gdn
