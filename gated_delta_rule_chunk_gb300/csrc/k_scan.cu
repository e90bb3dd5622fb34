// K3, bf16 inputs with scalar gates: fused inter-chunk scan over [sequences, value heads,
// dv blocks of 32].
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 5: the state contribution,
// the local-attention output and the state update are fused per sequence and value
// head, walking the chunks in order with the fp32 state updated in place. "Chunking
// Qwen3.5's gated DeltaNet ... on Apple Silicon" (section "How do you parallelize a
// recurrence for prefill?"): the value dimension of the state is blocked so that the
// tile stays on chip. A CTA owns 32 value columns of one (sequence, value head).
//
// Per chunk, with S the chunk-start state ([dk][dv], held transposed as S^T [dv][dk]),
// G the in-chunk gate sum and L the last row:
//   chain (serial):   X^T = S^T w^T;  v_new^T = u^T - X^T
//                     S^T <- exp(G_L) S^T + (v_new^T diag(exp(G_L - G))) K
//   output (lags the chain by one chunk):
//                     o = scale (diag(exp(G) / ||q||) Q S + M v_new)
//
// Warp roles (8 warps; warp w runs on SM sub-partition w % 4):
//   * warps 0, 1 (chain): warp r owns the 16 value columns 16r..16r+15 of the block with
//     all 128 key rows, as fp32 MMA accumulators of S^T. Because S^T sits in the
//     accumulator layout of m16n8 tiles, pairs of its n-tiles are directly the A
//     fragments of the next product (as are those of X^T), so the chain never moves the
//     state through shared memory: two dependent warp-MMA groups per chunk (64 m16n8k16
//     each), with w (bf16) and the fp16 k image as the shared-memory operands.
//   * warps 2, 3, 6, 7 (output): each takes one 16-token row tile of the chunk for all 32
//     columns (warps 2 and 6, which share a sub-partition, tiles 0 and 3; warps 3 and 7
//     tiles 1 and 2, which balances the triangular M product between the two):
//     Q S with fp16 operands (the intra kernel's fp16 q image, the chain's fp16 copy of
//     S) and M v_new as two fp16 products (the intra kernel's fp16 hi/lo pair of M, the
//     chain's fp16 v_new: M_hi v + M_lo v).
//     They run on the two sub-partitions the chain leaves free, so the two roles do not
//     share a tensor unit (no tcgen05 anywhere in this kernel).
//   * warp 4 (loads): one thread issues every copy: a 3-slot ring of what the chain
//     reads (w, k, the u block, G; bulk copies of images the intra kernel wrote in this
//     kernel's layout) and a double buffer of what the output warps read (the fp16 q
//     image and the [M_hi; M_lo] image).
// The chain hands each chunk's fp16 S and fp16 v_new to the output warps through a
// double-buffered shared tile (stmatrix). Precision (CPU emulation against the fp64
// oracle at the headline distributions, two seeds): w S with bf16 operands, the state
// update with fp16 operands, Q S with fp16 operands and M v_new with M an fp16 hi/lo pair
// and v_new one fp16 rounding keep the output within 2.9-3.4e-3 of its rms (bf16 hi/lo
// pairs for both, three products: 2.3-2.4e-3; one fp16 rounding of M as well: 5.6-6.4e-3).
// M in fp16 asks |M_ij| <= 65504 (|q.k| exp(G_i - G_j), at most |q||k|); a value out of
// range makes the output non-finite, which sets GDN_DEV_NONFINITE.
//
// Hand-offs use mbarriers; every wait is bounded (GDN_DEV_TIMEOUT on expiry, after which
// every role runs through without waiting; the load thread still waits, at the full
// bound, for each copy it issued before the CTA retires). A testing hook makes the chain
// wait on an event that never happens, to exercise that path. A non-finite state or output (an fp16
// operand out of range, or non-finite inputs) sets GDN_DEV_NONFINITE.
#include <cuda.h>

#include "gdn_common.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int BV = 32;
constexpr uint32_t kWaitIters = 1u << 22;
constexpr int kLoadWarp = 4;
constexpr int kThreads = 256;
constexpr int kOutWarps = 4;  // warps 2, 3, 6, 7; warp 5 has no role
constexpr int kMT = 4 / kOutWarps;  // 16-row tiles of a chunk per output warp
constexpr int kRing = 3;

// Ring slot (bytes; 128-byte-swizzled tiles are 1024-byte aligned).
constexpr uint32_t rW = 0;        // w, bf16: two dk halves of [64 tokens][128 B], 128-B swizzle
constexpr uint32_t rK = 16384;    // k, fp16: same layout
constexpr uint32_t rU = 32768;    // u block, fp32 [32 columns][64 tokens], 32-B groups swizzled
constexpr uint32_t rE = 40960;    // exp(G) [64], exp(G_L - G) [64]
constexpr uint32_t kSlot = 41984;
constexpr uint32_t kTxRing = 16384 + 16384 + 8192 + 512;
// Output operands, double-buffered: q (two dk halves of [64][128 B], swizzled, by tensor
// map) and [M_hi; M_lo] ([128 rows][128 B], swizzled).
constexpr uint32_t kQM = kRing * kSlot;
constexpr uint32_t qQ = 0;
constexpr uint32_t qM = 16384;
constexpr uint32_t kQMsz = 32768;
// Chain -> output hand-off, double-buffered: S fp16 [32 columns][256 B] and v_new fp16
// [32 columns][128 B] (16-byte chunk c of row r stored at chunk c ^ (r % 8)), and the
// chunk's G [64].
constexpr uint32_t kSV = kQM + 2 * kQMsz;
constexpr uint32_t vS = 0;
constexpr uint32_t vV = 8192;
constexpr uint32_t vG = 12288;
constexpr uint32_t kSVsz = 12288 + 1024;
// Output staging: per output warp two [16 tokens][64 B] bf16 tiles (16-byte chunk c of
// row r at c ^ ((r / 2) % 4)), stored by stmatrix and read back as 16-byte rows.
constexpr uint32_t kOST = kSV + 2 * kSVsz;
constexpr uint32_t kOSTsz = 1024 * kMT;
constexpr uint32_t kBar = kOST + kOutWarps * kOSTsz;
constexpr uint32_t kMisc = kBar + 128;
constexpr uint32_t kSmemBytes = kMisc + 16 + 1024;  // + room to align the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

// mbarriers. Ring: chunk c uses slot c % 3, parity (c / 3) & 1. Double buffers: index
// c & 1, parity (c >> 1) & 1.
constexpr int B_FULL = 0;   // ring slot landed (transaction bytes)
constexpr int B_EMPTY = 3;  // both chain warps done with the ring slot
constexpr int B_QF = 6;     // q and M of chunk c landed
constexpr int B_QE = 8;     // every output warp done with q and M of chunk c
constexpr int B_SF = 10;    // both chain warps wrote S and v_new of chunk c
constexpr int B_SE = 12;    // every output warp done with the hand-off buffer of chunk c
constexpr int B_STALL = 14; // never completes (the testing hook's wait)
constexpr int kNumBars = 15;

// Byte offset of the 16-byte chunk holding column-chunk ch of row r in a tile of
// `rowb`-byte rows whose chunks are swizzled by row (c ^ (r % 8)).
__device__ __forceinline__ uint32_t swz(int r, int ch, uint32_t rowb) {
  return (uint32_t)r * rowb + ((uint32_t)(ch ^ (r & 7)) << 4);
}
// Chunk ch (0..15) of row r of a two-half K-major image ([64 rows][128 B] per 64 columns).
__device__ __forceinline__ uint32_t half_img(int r, int ch) {
  return (uint32_t)(ch >> 3) * 8192u + swz(r, ch & 7, 128);
}
// fp32 element (column j, token i) of a u block: [32][64], 32-byte groups swizzled by row.
__device__ __forceinline__ uint32_t u_blk(int j, int i) {
  return (uint32_t)j * 256u + ((uint32_t)((i >> 3) ^ (j & 7)) << 5) + (uint32_t)(i & 7) * 4u;
}

__device__ __forceinline__ void stsm_x4(uint32_t saddr, uint32_t r0, uint32_t r1, uint32_t r2,
                                        uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(saddr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// Bounded wait for the phase of `bar` with parity `parity`. Gives up after a bounded
// number of polls (raising the abort flag), and at once when the flag is already raised.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         volatile int* abort_flag, uint32_t limit = kWaitIters) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// Same, with a short sleep between polls: for the load thread, which shares its SM
// sub-partition with a chain warp and is never on the critical path.
__device__ __forceinline__ bool wait_bar_sleep(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitIters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    __nanosleep(128);
  }
  *abort_flag = 1;
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
scan_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Grid (see launch_scan): one sequence: x = value head, y = value block; several: x =
  // (value block, value head), value block fastest, so that the CTAs that share a head's
  // images (then a sequence's) start together and meet in L2, and y + 65535 z = the
  // sequence's rank in the longest-first order (or its index), so that long sequences
  // start first.
  const int nvb = p.D / BV;
  const bool one = p.N == 1;
  const int vb = one ? (int)blockIdx.y : (int)blockIdx.x % nvb;
  const int hv = one ? (int)blockIdx.x : (int)blockIdx.x / nvb;
  const int rank = one ? 0 : (int)(blockIdx.z * 65535 + blockIdx.y);
  if (rank >= p.N) return;  // (uniform over the CTA)
  const int c0 = vb * BV;
  const int h = hv / p.HG;
  const int g = lane >> 2, c2 = 2 * (lane & 3);
  const bool has_out = p.out != nullptr;

  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b)
      mbar_init(&bars[b], (b < B_EMPTY || (b >= B_QF && b < B_QE))
                              ? 1
                              : ((b >= B_QE && b < B_SF) || b >= B_SE) ? kOutWarps : 2);
    mbar_init_fence();
    *abort_flag = 0;
  }
  __syncthreads();
  pdl_wait();  // everything below reads what the chunk-table and intra kernels wrote
  const int n = p.seq_order ? p.seq_order[rank] : rank;
  const size_t state_base = ((size_t)n * p.Hv + hv) * p.D * p.D;
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }

  if (warp < 2) {
    // ---------------------------------------------------------------- chain
    // S^T accumulators: S[nt][e] = S^T[column 16r + g + 8(e >> 1)][key 8nt + c2 + (e & 1)].
    const int r = warp, rb = 16 * r;
    float S[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int col = c0 + rb + g + 8 * hh, key = 8 * nt + c2;
        float2 x = make_float2(0.f, 0.f);
        if (p.s0 && key < p.D)
          x = *reinterpret_cast<const float2*>(p.s0 + state_base + (size_t)col * p.D + key);
        S[nt][2 * hh] = x.x;
        S[nt][2 * hh + 1] = x.y;
      }
    // fp16 S^T to the hand-off buffer of chunk cc (its 16 x 16 blocks by stmatrix)
    auto store_s16 = [&](int cc) {
      const uint32_t dst = sbase + kSV + (cc & 1) * kSVsz + vS;
      const int row = rb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        stsm_x4(dst + swz(row, 2 * ks + (lane >> 4), 256), pack_f16(S[2 * ks][0], S[2 * ks][1]),
                pack_f16(S[2 * ks][2], S[2 * ks][3]), pack_f16(S[2 * ks + 1][0], S[2 * ks + 1][1]),
                pack_f16(S[2 * ks + 1][2], S[2 * ks + 1][3]));
    };
    if (nch > 0 && has_out) store_s16(0);
    // testing hook: a bounded wait for an event that never happens (nothing arrives on
    // B_STALL), so that the call takes the timeout path below
    if (p.stall_polls && nch > 0) wait_bar(&bars[B_STALL], 0, abort_flag, p.stall_polls);
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kRing, b = c & 1;
      const unsigned char* st = sm + slot * kSlot;
      const uint32_t st_a = sbase + slot * kSlot;
      wait_bar(&bars[B_FULL + slot], (uint32_t)((c / kRing) & 1), abort_flag);
      // row factors exp(G_L - G_i) of this thread's 16 tokens and the state decay, formed
      // first so that their latency hides under the X product
      const float* E = reinterpret_cast<const float*>(st + rE);
      float fac[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 ff = *reinterpret_cast<const float2*>(&E[64 + 8 * nt + c2]);
        fac[nt][0] = ff.x;
        fac[nt][1] = ff.y;
      }
      const float gam = E[63];
      const size_t slot_hv = (size_t)(sv.first_slot + c) * p.Hv + hv;
      // chunk-start state [dv][dk] (the backward's recompute)
      if (p.hs && dbg_ok(slot_hv < (size_t)p.nt_max * p.Hv, p.status)) {
        float* hs = p.hs + slot_hv * p.D * p.D;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int col = c0 + rb + g + 8 * hh, key = 8 * nt + c2;
            if (key < p.D)
              *reinterpret_cast<float2*>(hs + (size_t)col * p.D + key) =
                  make_float2(S[nt][2 * hh], S[nt][2 * hh + 1]);
          }
      }

      // this thread's u values, loaded before the X product so their latency hides
      float2 uu[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          uu[nt][hh] = *reinterpret_cast<const float2*>(st + rU + u_blk(rb + g + 8 * hh, 8 * nt + c2));
      // X^T = S^T w^T: columns 16r.., tokens 0..63 (8 n-tiles), keys in 8 steps of 16
      float X[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) X[nt][e] = 0.f;
      {
        const int m = lane >> 3;
        const int brow = (m >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          // bf16 A fragment of S^T for keys 16ks..16ks+15: n-tiles 2ks and 2ks + 1
          const uint32_t sa[4] = {pack_bf16(S[2 * ks][0], S[2 * ks][1]),
                                  pack_bf16(S[2 * ks][2], S[2 * ks][3]),
                                  pack_bf16(S[2 * ks + 1][0], S[2 * ks + 1][1]),
                                  pack_bf16(S[2 * ks + 1][2], S[2 * ks + 1][3])};
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            uint32_t bb[4];
            ldsm_x4_addr(bb, st_a + rW + half_img(16 * np + brow, 2 * ks + (m & 1)));
            mma_bf16(X[2 * np], sa, bb[0], bb[1]);
            mma_bf16(X[2 * np + 1], sa, bb[2], bb[3]);
          }
        }
      }
      // v_new^T = u^T - X^T (in place in X)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float2 u2 = uu[nt][hh];
          X[nt][2 * hh] = u2.x - X[nt][2 * hh];
          X[nt][2 * hh + 1] = u2.y - X[nt][2 * hh + 1];
        }
      // v_new [64 tokens][dv] of the chunk (the backward's recompute)
      if (p.vn_out && dbg_ok(slot_hv < (size_t)p.nt_max * p.Hv, p.status)) {
        float* vo = p.vn_out + slot_hv * 64 * p.D + c0 + rb;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            vo[(size_t)(8 * nt + c2 + (e & 1)) * p.D + g + 8 * (e >> 1)] = X[nt][e];
      }
      if (has_out) {  // v_new in fp16 for the output's M v_new
        const uint32_t dst = sbase + kSV + b * kSVsz;
        const int row = rb + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt)
          stsm_x4(dst + vV + swz(row, 2 * kt + (lane >> 4), 128),
                  pack_f16(X[2 * kt][0], X[2 * kt][1]), pack_f16(X[2 * kt][2], X[2 * kt][3]),
                  pack_f16(X[2 * kt + 1][0], X[2 * kt + 1][1]),
                  pack_f16(X[2 * kt + 1][2], X[2 * kt + 1][3]));
        if (r == 0)  // the chunk's G for the output's row factors
          *reinterpret_cast<float2*>(sm + kSV + b * kSVsz + vG + 8 * lane) =
              *reinterpret_cast<const float2*>(&E[2 * lane]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_SF + b]);
      }
      // fp16 A fragments of v_new^T diag(exp(G_L - G)) (tokens in 4 k-steps of 16)
      uint32_t va[4][4];
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        va[kt][0] = pack_f16(fac[2 * kt][0] * X[2 * kt][0], fac[2 * kt][1] * X[2 * kt][1]);
        va[kt][1] = pack_f16(fac[2 * kt][0] * X[2 * kt][2], fac[2 * kt][1] * X[2 * kt][3]);
        va[kt][2] = pack_f16(fac[2 * kt + 1][0] * X[2 * kt + 1][0],
                             fac[2 * kt + 1][1] * X[2 * kt + 1][1]);
        va[kt][3] = pack_f16(fac[2 * kt + 1][0] * X[2 * kt + 1][2],
                             fac[2 * kt + 1][1] * X[2 * kt + 1][3]);
      }
      // S^T <- exp(G_L) S^T + va K  (keys in 16 n-tiles; the k image read transposed)
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) S[nt][e] *= gam;
      {
        const int m = lane >> 3;
        const int krow = (m & 1) * 8 + (lane & 7);
#pragma unroll
        for (int kt = 0; kt < 4; ++kt)
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            uint32_t bb[4];
            ldsm_x4_t_addr(bb, st_a + rK + half_img(16 * kt + krow, 2 * np + (m >> 1)));
            mma_f16(S[2 * np], va[kt], bb[0], bb[1]);
            mma_f16(S[2 * np + 1], va[kt], bb[2], bb[3]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_EMPTY + slot]);  // ring slot released
      if (c + 1 < nch) {
        if (has_out) {
          // the hand-off buffer of chunk c + 1 was last read by the output of chunk c - 1
          if (c >= 1) wait_bar(&bars[B_SE + ((c + 1) & 1)], (uint32_t)(((c - 1) >> 1) & 1),
                               abort_flag);
          store_s16(c + 1);
        }
      }
    }
    bool finite = true;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) finite = finite && isfinite(S[nt][e]);
    if (!__all_sync(0xffffffffu, finite) && lane == 0) set_status(p.status, GDN_DEV_NONFINITE);
    if (p.sT) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int col = c0 + rb + g + 8 * hh, key = 8 * nt + c2;
          if (key < p.D)
            *reinterpret_cast<float2*>(p.sT + state_base + (size_t)col * p.D + key) =
                make_float2(S[nt][2 * hh], S[nt][2 * hh + 1]);
        }
    }
  } else if ((warp & 3) >= 2) {
    // ---------------------------------------------------------------- output
    // Row tiles by warp: 2 -> 0, 3 -> 1, 6 -> 3, 7 -> 2, so that each SM sub-partition's
    // pair has the same M steps (1 + 4 = 2 + 3).
    const int ow = (warp & 1) + ((warp >> 2) << 1);
    const int mts[kMT] = {ow < 2 ? ow : 5 - ow};
    float chk = 0.f;  // stays 0 unless an output is non-finite (x * 0 is NaN for inf, NaN)
    const uint32_t ost = sbase + kOST + ow * kOSTsz;
    // (no output wanted: the backward's recompute keeps only states and v_new, and the
    // chain then makes no hand-off)
    for (int c = 0; has_out && c < nch; ++c) {
      const int b = c & 1;
      const int t0 = sv.start + kChunk * c;
      const int L = min(kChunk, sv.len - kChunk * c);
      wait_bar(&bars[B_QF + b], (uint32_t)((c >> 1) & 1), abort_flag);
      wait_bar(&bars[B_SF + b], (uint32_t)((c >> 1) & 1), abort_flag);
      const uint32_t qa = sbase + kQM + b * kQMsz, sva = sbase + kSV + b * kSVsz;
      // row factors scale exp(G_i) of this thread's rows (1/||q_i|| is inside the q image)
      float f[kMT][2];
      {
        const float* Gs = reinterpret_cast<const float*>(sm + kSV + b * kSVsz + vG);
#pragma unroll
        for (int mi = 0; mi < kMT; ++mi)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            f[mi][hh] = p.scale * Gs[16 * mts[mi] + g + 8 * hh];
      }
      const int m = lane >> 3;
      const int arow = (lane & 7) + (m & 1) * 8;   // A fragment row inside a 16-row tile
      const int brow = (m >> 1) * 8 + (lane & 7);  // B fragment row (column of o) in 16
      float qs[kMT][4][4], mv[kMT][4][4];
#pragma unroll
      for (int mi = 0; mi < kMT; ++mi)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qs[mi][nt][e] = 0.f;
            mv[mi][nt][e] = 0.f;
          }
      // Q S (fp16): A = the fp16 q image's rows, B = the chain's fp16 S^T rows. The
      // output warps' loops stay compact: run once per chunk, unrolled code does not stay
      // in the instruction cache.
#pragma unroll 2
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t bs[2][4];
#pragma unroll
        for (int np = 0; np < 2; ++np)
          ldsm_x4_addr(bs[np], sva + vS + swz(16 * np + brow, 2 * ks + (m & 1), 256));
#pragma unroll
        for (int mi = 0; mi < kMT; ++mi) {
          uint32_t a[4];
          ldsm_x4_addr(a, qa + qQ + half_img(16 * mts[mi] + arow, 2 * ks + (m >> 1)));
          mma_f16(qs[mi][0], a, bs[0][0], bs[0][1]);
          mma_f16(qs[mi][1], a, bs[0][2], bs[0][3]);
          mma_f16(qs[mi][2], a, bs[1][0], bs[1][1]);
          mma_f16(qs[mi][3], a, bs[1][2], bs[1][3]);
        }
      }
      // M v_new: M lower triangular, so row tile mt needs token steps 0..mt only
#pragma unroll
      for (int mi = 0; mi < kMT; ++mi) {
        const int mt = mts[mi];
        for (int ks = 0; ks <= mt; ++ks) {
          uint32_t ah[4], al[4], bv[2][4];
          const uint32_t aoff = swz(16 * mt + arow, 2 * ks + (m >> 1), 128);
          ldsm_x4_addr(ah, qa + qM + aoff);
          ldsm_x4_addr(al, qa + qM + 8192 + aoff);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            const uint32_t boff = swz(16 * np + brow, 2 * ks + (m & 1), 128);
            ldsm_x4_addr(bv[np], sva + vV + boff);
          }
#pragma unroll
          for (int np = 0; np < 2; ++np)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float(&acc)[4] = mv[mi][2 * np + q];
              mma_f16(acc, ah, bv[np][2 * q], bv[np][2 * q + 1]);
              mma_f16(acc, al, bv[np][2 * q], bv[np][2 * q + 1]);
            }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[B_QE + b]);
        mbar_arrive(&bars[B_SE + b]);
      }
      // o = f qs + scale mv; rows past the sequence end are not stored. bf16: each 16-row
      // tile goes through a staging tile (stmatrix) and leaves as 16-byte rows.
#pragma unroll
      for (int mi = 0; mi < kMT; ++mi) {
        const int mt = mts[mi];
        uint32_t pk[4][2];
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const float a = f[mi][hh] * qs[mi][nt][2 * hh] + p.scale * mv[mi][nt][2 * hh];
            const float b2 = f[mi][hh] * qs[mi][nt][2 * hh + 1] + p.scale * mv[mi][nt][2 * hh + 1];
            rs[hh] += a + b2;
            if (p.out_bf16) {
              pk[nt][hh] = pack_bf16(a, b2);
            } else if (16 * mt + g + 8 * hh < L &&
                       dbg_ok(t0 + 16 * mt + g + 8 * hh < p.T, p.status)) {
              *reinterpret_cast<float2*>(static_cast<float*>(p.out) +
                                         ((size_t)(t0 + 16 * mt + g + 8 * hh) * p.Hv + hv) * p.D +
                                         c0 + 8 * nt + c2) = make_float2(a, b2);
            }
          }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) chk += (16 * mt + g + 8 * hh < L) ? rs[hh] * 0.f : 0.f;
        if (p.out_bf16) {
          const uint32_t st = ost + mi * 1024;
          const int srow = (lane & 7) + (m & 1) * 8;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            stsm_x4(st + srow * 64 + ((uint32_t)((2 * hf + (m >> 1)) ^ ((srow >> 1) & 3)) << 4),
                    pk[2 * hf][0], pk[2 * hf][1], pk[2 * hf + 1][0], pk[2 * hf + 1][1]);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int row = (lane >> 2) + 8 * j, ch = lane & 3;
            uint4 v;
            asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "r"(st + row * 64 + ((uint32_t)(ch ^ ((row >> 1) & 3)) << 4)));
            if (16 * mt + row < L && dbg_ok(t0 + 16 * mt + row < p.T, p.status))
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                        ((size_t)(t0 + 16 * mt + row) * p.Hv + hv) * p.D + c0 +
                                        8 * ch) = v;
          }
        }
      }
    }
    if (__any_sync(0xffffffffu, chk != 0.f) && lane == 0) set_status(p.status, GDN_DEV_NONFINITE);
  } else if (warp == kLoadWarp && lane == 0) {
    // ---------------------------------------------------------------- loads
    auto issue_ring = [&](int cc) {
      const int slot = cc % kRing;
      unsigned char* st = sm + slot * kSlot;
      uint64_t* full = &bars[B_FULL + slot];
      size_t wslot = (size_t)sv.first_slot + cc;
      if (!dbg_ok(wslot < (size_t)p.nt_max, p.status)) wslot = 0;  // (keeps the tx count)
      const size_t sl = wslot * p.Hv + hv;
      mbar_expect_tx(full, kTxRing);
      bulk_load(st + rW, static_cast<const unsigned char*>(p.w) + sl * 16384, 16384, full);
      bulk_load(st + rK, static_cast<const unsigned char*>(p.k16) + (wslot * p.H + h) * 16384,
                16384, full);
      bulk_load(st + rU, reinterpret_cast<const unsigned char*>(p.u) + sl * 32768 +
                             vb * 8192, 8192, full);
      bulk_load(st + rE, p.EF + sl * 128, 512, full);
    };
    auto issue_qm = [&](int cc) {
      unsigned char* dst = sm + kQM + (cc & 1) * kQMsz;
      uint64_t* full = &bars[B_QF + (cc & 1)];
      size_t wslot = (size_t)sv.first_slot + cc;
      if (!dbg_ok(wslot < (size_t)p.nt_max, p.status)) wslot = 0;  // (keeps the tx count)
      const size_t sl = wslot * p.Hv + hv;
      mbar_expect_tx(full, kQMsz);
      bulk_load(dst + qQ, static_cast<const unsigned char*>(p.q16) + (wslot * p.H + h) * 16384,
                16384, full);
      bulk_load(dst + qM, static_cast<const unsigned char*>(p.M) + sl * 16384, 16384, full);
    };
    int issued = 0, qm_issued = 0;
    for (int k = 0; k < min(nch, kRing); ++k) issue_ring(k);
    issued = min(nch, kRing);
    if (has_out) {
      for (int k = 0; k < min(nch, 2); ++k) issue_qm(k);
      qm_issued = min(nch, 2);
    }
    for (int c = 0; c < nch; ++c) {
      if (*abort_flag) break;
      if (c + kRing < nch) {  // ring slot of chunk c is free once both chain warps released it
        if (!wait_bar_sleep(&bars[B_EMPTY + c % kRing], (uint32_t)((c / kRing) & 1), abort_flag))
          break;
        issue_ring(c + kRing);
        issued = c + kRing + 1;
      }
      if (has_out && c + 2 < nch) {  // q / M buffer of chunk c is free once the output read it
        if (!wait_bar_sleep(&bars[B_QE + (c & 1)], (uint32_t)((c >> 1) & 1), abort_flag)) break;
        issue_qm(c + 2);
        qm_issued = c + 3;
      }
    }
    // Before the CTA retires: every copy this thread issued has landed (bounded waits).
    for (int k = max(0, issued - kRing); k < issued; ++k)
      mbar_wait(&bars[B_FULL + k % kRing], (uint32_t)((k / kRing) & 1), kWaitIters);
    for (int k = max(0, qm_issued - 2); k < qm_issued; ++k)
      mbar_wait(&bars[B_QF + (k & 1)], (uint32_t)((k >> 1) & 1), kWaitIters);
  }

  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(p.status, GDN_DEV_TIMEOUT);
}

}  // namespace

bool launch_scan(const Params& p, cudaStream_t s) {
  ensure_smem_limit((const void*)scan_kernel, (int)kSmemBytes);
  const int nvb = p.D / BV;
  const dim3 grid = p.N == 1 ? dim3(p.Hv, nvb, 1)
                             : dim3(p.Hv * nvb, p.N < 65535 ? p.N : 65535, (p.N + 65534) / 65535);
  return launch_pdl(scan_kernel, grid, dim3(kThreads), kSmemBytes, s, p) == cudaSuccess;
}

}  // namespace gdn
