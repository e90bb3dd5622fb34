// K2, bf16 inputs: fused intra-chunk kernel over [chunk slots, key heads].
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 4: K K^T is
// computed once per (chunk, key head) and reused by the value heads of the
// group; per value head the decay/beta-scaled A, its triangular inverse and
// the products that need it are formed without writing A to global memory.
// Section 8: the triangular solve stays triangular.
//
// Per (chunk, key head h), with rows past the end of the sequence masked
// (k = q = v = 0, beta = 0, g = 0):
//   [P; R] = [K; Q] K^T          (one M = 128 tcgen05 MMA group, fp32 in TMEM:
//                                 P = K K^T in TMEM lanes 0..63, R = Q K^T in 64..127)
//   per value head hv of the group:
//     G = inclusive in-chunk cumsum of g (fp32, left to right)
//     A_ij = beta_i exp(G_i - G_j) P_ij (j < i);  T = (I + A)^-1 in place (fp32 diagonal
//            blocks, off-diagonal blocks on warp MMAs with split operands)
//     w    = (T diag(beta exp(G))) K   (bf16 T operand; tcgen05, M = 64, N = 128)
//     u    = (T diag(beta)) V          (formed transposed, u^T = V^T (T diag(beta))^T, M = 128
//                                       value columns, N = 64 tokens; the T operand split
//                                       into bf16 hi + lo, two MMA groups into one
//                                       accumulator)
//     M_ij = exp(G_i - G_j) R_ij (j <= i)   (stored as a hi/lo pair: fp16 halves for the
//                                           forward's scan, bf16 halves for the backward)
// (1/||k|| and 1/||q|| enter as fp32 row factors when the L2 norm is on.) The hi/lo
// split keeps about 22 (fp16) or 16 (bf16) significant bits where one bf16 rounding
// would cost ~1e-2 of the output's rms.
//
// The bridge is written as the exact shared-memory images the inter-chunk
// kernel reads, so that kernel moves each with one bulk copy:
//   w: two 64-column halves, each [64 rows][128 B] with the 128-byte swizzle
//      (16-byte chunk c of row r stored at chunk c ^ (r % 8));
//   M: [128 rows: hi then lo][128 B], same swizzle;
//   u: [dv/32 blocks][32 columns][64 tokens] fp32 (each block stored column-major, the
//      scan's chain reads two tokens of one column at a time), 32-byte group c of column j
//      at c ^ (j % 8);
//   k and q (once per key head): fp16, scaled by 1/||k|| and 1/||q|| when the L2 norm is
//      on, zero past the sequence end, two 64-column halves of [64 rows][128 B] with the
//      128-byte swizzle.
// Each image is assembled in shared memory and written with bulk copies (TMA), so
// the warps never wait on scattered global stores; tiles come in by TMA tensor maps
// (128-byte swizzle), which are also the tensor-core operand layouts.
//
// One CTA of 8 warps per (key head, chunk); ~113 KB of shared memory and 256 TMEM
// columns, so two CTAs share an SM and hide each other's latency. Warps w and w + 4
// read the same TMEM lane quarter and split its columns. The chunk slots of the grid's
// last, partial wave can be split (split_slots): two CTAs per slot, one per half of the
// group's value heads, so that the wave ends sooner.
#include <cuda.h>

#include "gdn_common.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int LDT = 68;  // fp32 stride of the A/T tile (16-byte rows)
constexpr uint32_t kWaitIters = 1u << 22;
constexpr uint32_t kTmemCols = 256;
constexpr int kMStoreThread = kThreads - 32;  // issues the M image copies (warp 7, lane 0)

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t kKQ = 0;       // [K_h0 | Q_h0 | K_h1 | Q_h1], each [64 rows][128 B], swizzled;
                                  // the Q halves later hold the M image and the u operands
constexpr uint32_t kV = 32768;    // two buffers of [V_h0 | V_h1]
constexpr uint32_t kAT = 65536;   // fp32 [64][LDT]: A, then T; staging of the w image
constexpr int LDX = 36;  // fp32 stride of the inverse's scratch (32 rows)
constexpr uint32_t kX = kAT + 64 * LDT * 4;  // fp32 [32][LDX]: scratch of the inverse
constexpr uint32_t kTW = 88064;   // bf16 [64][128 B], swizzled: T diag(beta exp(G)) (w operand)
constexpr uint32_t kVec = kTW + 8192;        // 6 x fp32 [64] row vectors
constexpr uint32_t kBar = kVec + 6 * 256;    // 6 mbarriers
constexpr uint32_t kMisc = kBar + 64;        // TMEM base address, failure flag
constexpr uint32_t kST = kMisc + 16;         // 16 KB staging: the k image, then u blocks 2, 3
constexpr uint32_t kSmemBytes = kST + 16384 + 1024;  // + room to align the base to 1024
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs no longer share an SM");
static_assert(kX + 32 * LDX * 4 <= kTW, "shared-memory layout overlaps");
static_assert(kWarps == 8, "the triangular inverse is written for eight warps");

// Byte offset of 16-byte chunk ch of row r in a [rows][128 B] tile with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4);
}
__device__ __forceinline__ bool resolve(const Params& p, int slot, int& t0, int& L, int& wslot) {
  const int2 e = p.chunk_table[slot];
  if (e.x < 0) return false;  // sentinel: early exit
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

// Bounded wait; on expiry the CTA's failure flag is raised (reported as GDN_DEV_TIMEOUT).
__device__ __forceinline__ void wait_or_flag(uint64_t* bar, uint32_t parity, volatile int* fail) {
  if (!mbar_wait(bar, parity, kWaitIters)) *fail = 1;
}

// Rows L..63 of a [64 rows][128 B] tile read as zero (the tile holds the rows that
// follow the sequence, or padding, there).
__device__ __forceinline__ void zero_tail(unsigned char* tile, int L, int tid) {
  for (int idx = tid; idx < (64 - L) * 8; idx += kThreads)
    *reinterpret_cast<uint4*>(tile + (uint32_t)(L + (idx >> 3)) * 128u + (idx & 7) * 16u) =
        make_uint4(0u, 0u, 0u, 0u);
}

// Value-head tile of group member r (rows t0..t0+63) into V buffer r & 1.
__device__ __forceinline__ void issue_v(unsigned char* sm, uint64_t* bars, const CUtensorMap* tmv,
                                        int hv, int t0, int r) {
  uint64_t* bar = &bars[1 + (r & 1)];
  unsigned char* dst = sm + kV + (r & 1) * 16384;
  mbar_expect_tx(bar, 16384);
  tma_load_3d(dst, tmv, 0, hv, t0, bar);
  tma_load_3d(dst + 8192, tmv, 64, hv, t0, bar);
}

__global__ void __launch_bounds__(kThreads, 2)
tc_intra_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  float* AT = reinterpret_cast<float*>(sm + kAT);
  float* X = reinterpret_cast<float*>(sm + kX);
  float* G = reinterpret_cast<float*>(sm + kVec);
  float* Bt = G + 64;   // beta
  float* KR = G + 128;  // 1/||k|| (1 when the norm is off)
  float* FW = G + 192;  // beta exp(G) / ||k||: column factor of the w operand
  float* QR = G + 256;  // 1/||q|| (1 when the norm is off)
  // mbarriers: 0 k/q landed, 1-2 v buffers landed, 3 [P; R] done, 4 w done, 5 u done (one
  // completion per value head for 4 and 5)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* fail = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Key head fastest in the grid: CTAs resident together read all heads of the same
  // tokens (contiguous rows of q, k and v) rather than one head of many chunks.
  const int h = blockIdx.x;
  // Chunk slot and the value heads of the group this CTA takes: all of them, or for the
  // last split_slots slots one half (two CTAs per slot, adjacent in the grid).
  int slot = (int)blockIdx.y, r_begin = 0, nr = p.HG;
  if (slot >= p.nt_max - p.split_slots) {
    const int j = slot - (p.nt_max - p.split_slots);
    slot = p.nt_max - p.split_slots + (j >> 1);
    nr = p.HG >> 1;
    r_begin = (j & 1) * nr;
  }
  const bool writes_img = r_begin == 0;  // the k and q images: once per (slot, key head)
  int t0 = 0, L = 0, wslot = 0;
  // One sequence whose table this call builds: slot s is chunk s of the sequence, whose
  // bounds are sanitized here exactly as the chunk-table kernel does, so the tiles (the
  // caller's inputs) are requested while that kernel still runs. Other slots are sentinels.
  bool early = false;
  int seq_s0 = 0, seq_nch = 0;  // (the one sequence's start and chunk count)
  if (p.early_one) {
    const int s0 = p.cu ? min(max(p.cu[0], 0), p.T) : 0;
    const int e0 = p.cu ? max(min(max(p.cu[1], 0), p.T), s0) : p.T;
    const int nch = (e0 - s0 + kChunk - 1) / kChunk;
    if (slot >= nch) {  // (the table holds a sentinel there)
      pdl_wait();  // no CTA of this grid ends before the chunk-table kernel: the scan reads
      return;      // what that kernel wrote once this grid is done
    }
    early = true;
    seq_s0 = s0;
    seq_nch = nch;
    t0 = s0 + kChunk * slot;
    L = min(kChunk, e0 - t0);
    wslot = slot;
  } else {
    pdl_wait();     // the chunk table (and the L2-norm factors) are written
    pdl_release();  // the inter kernel may take SMs as this grid drains
    if (!resolve(p, slot, t0, L, wslot)) return;  // uniform over the CTA
  }
  // The q image is staged in the second V buffer, whose tile is loaded once the image has
  // been read out.
  const bool v1_late = writes_img && p.q16 != nullptr && nr > 1;
  const size_t n_vslots = (size_t)p.nt_max * p.Hv;  // value slots of the bridge regions

  // g and beta of group member r (warp 0, 2 rows per lane), loaded one member ahead of
  // their use; the first member's loads are in flight during the setup below.
  float gn0 = 0.f, gn1 = 0.f, bn0 = 0.f, bn1 = 0.f;
  auto load_gates = [&](int r) {
    const int hv = h * p.HG + r;
    const size_t b0 = (size_t)(t0 + lane) * p.Hv + hv, b1 = (size_t)(t0 + lane + 32) * p.Hv + hv;
    gn0 = lane < L ? p.g[b0] : 0.f;
    gn1 = lane + 32 < L ? p.g[b1] : 0.f;
    bn0 = lane < L ? p.beta[b0] : 0.f;
    bn1 = lane + 32 < L ? p.beta[b1] : 0.f;
  };
  if (warp == 0) {
    load_gates(r_begin);
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 6; ++b) mbar_init(&bars[b], 1);
    mbar_init_fence();
    *fail = 0;
    mbar_expect_tx(&bars[0], 32768);
    tma_load_3d(sm + kKQ, &tmk, 0, h, t0, &bars[0]);
    tma_load_3d(sm + kKQ + 16384, &tmk, 64, h, t0, &bars[0]);
    tma_load_3d(sm + kKQ + 8192, &tmq, 0, h, t0, &bars[0]);
    tma_load_3d(sm + kKQ + 24576, &tmq, 64, h, t0, &bars[0]);
    for (int rl = 0; rl < min(nr, v1_late ? 1 : 2); ++rl)
      issue_v(sm, bars, &tmv, h * p.HG + r_begin + rl, t0, rl);
  }
  if (tid < 64) KR[tid] = (tid < L && p.krn) ? p.krn[(size_t)(t0 + tid) * p.H + h] : 1.f;
  else if (tid < 128)
    QR[tid - 64] = (tid - 64 < L && p.qrn) ? p.qrn[(size_t)(t0 + tid - 64) * p.H + h] : 1.f;
  // 1/||q|| of the row this thread forms M for (warps 2, 3, 6 and 7 own rows 0..63 of R)
  const int qrow = 32 * (warp & 1) + lane;
  const float qr = ((warp & 3) >= 2 && p.qrn && qrow < L) ? p.qrn[(size_t)(t0 + qrow) * p.H + h] : 1.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto prefetch_next_wave = [&]() {
    if (tid != kMStoreThread || p.pf_ahead <= 0) return;
    // L2 prefetch of the tiles of the slot about one wave ahead, which the CTA that next
    // takes this SM is likely to hold, so that its loads hit L2
    const int s1 = slot + p.pf_ahead;
    int t1 = -1;
    if (early) {  // (slot s1 is chunk s1 of the one sequence)
      if (s1 < seq_nch) t1 = seq_s0 + kChunk * s1;
    } else if (s1 < p.nt_max) {
      const int2 e = p.chunk_table[s1];
      if (e.x >= 0 && e.x < p.N) {
        const SeqView sv1 = seq_view(p, e.x);
        if (e.y >= 0 && kChunk * e.y < sv1.len) t1 = sv1.start + kChunk * e.y;
      }
    }
    if (t1 >= 0) {
#pragma unroll 1
      for (int x = 0; x < p.D; x += 64) {  // (a head of 64 has one half)
        tma_prefetch_3d(&tmk, x, h, t1);
        tma_prefetch_3d(&tmq, x, h, t1);
#pragma unroll 1
        for (int r = 0; r < p.HG; ++r) tma_prefetch_3d(&tmv, x, h * p.HG + r, t1);
      }
      const int rows = min(kChunk, p.T - t1);
      const uint32_t gb = (uint32_t)(rows * p.Hv * 4) & ~15u;
      const size_t go = (size_t)t1 * p.Hv;
      if (h == 0 && gb > 0 && ((go * 4) & 15) == 0) {  // every head's gates of those rows
        bulk_prefetch_l2(p.g + go, gb);
        bulk_prefetch_l2(p.beta + go, gb);
      }
    }
  };
  if (!early) prefetch_next_wave();
  // Gates of group member r and their in-chunk inclusive cumsum (warp 0, 2 rows per lane).
  auto gates = [&](int r) {
    const size_t sl = (size_t)wslot * p.Hv + h * p.HG + r;
    float g0 = gn0, g1 = gn1;
    const float be0 = bn0, be1 = bn1;
    if (r + 1 < r_begin + nr) load_gates(r + 1);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_up_sync(0xffffffffu, g0, o);
      const float y1 = __shfl_up_sync(0xffffffffu, g1, o);
      if (lane >= o) {
        g0 += y0;
        g1 += y1;
      }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
    G[lane] = g0;
    G[lane + 32] = g1;
    Bt[lane] = be0;
    Bt[lane + 32] = be1;
    const float e0 = expf(g0), e1 = expf(g1);
    FW[lane] = be0 * e0 * KR[lane];
    FW[lane + 32] = be1 * e1 * KR[lane + 32];
    if (!dbg_ok(sl < n_vslots, p.status)) return;
    p.G[sl * 64 + lane] = g0;
    p.G[sl * 64 + lane + 32] = g1;
    if (p.EF) {  // exp(G) and exp(G_L - G) for the scan (G is flat past the last row)
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      float* ef = p.EF + sl * 128;
      ef[lane] = e0;
      ef[lane + 32] = e1;
      ef[64 + lane] = expf(gl - g0);
      ef[96 + lane] = expf(gl - g1);
    }
  };
  wait_or_flag(&bars[0], 0, fail);
  if (L < kChunk) {  // (a full chunk needs no barrier: thread 0 waited for the tiles itself)
    zero_tail(sm + kKQ, L, tid);
    zero_tail(sm + kKQ + 8192, L, tid);
    zero_tail(sm + kKQ + 16384, L, tid);
    zero_tail(sm + kKQ + 24576, L, tid);
    fence_async_smem();
    __syncthreads();
  }
  if (tid == 0) {  // [P; R] = [K; Q] K^T
    tc_fence_after();
    const uint32_t id = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a = sbase + kKQ + (ks >> 2) * 16384 + 32 * (ks & 3);
      umma_bf16(tmem, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024), id, ks > 0);
    }
    umma_commit(&bars[3]);
  }

  // fp16 images of the (normalised) k and q tiles, assembled in the A/T region and the
  // second V buffer, each two halves of [64 rows][128 B] with the 128-byte swizzle; the
  // scan reads them with one bulk copy each.
  auto f16_image = [&](const unsigned char* src, unsigned char* img, const float* rowf) {
#pragma unroll
    for (int it = 0; it < 1024 / kThreads; ++it) {
      const int idx = tid + it * kThreads;  // 1024 chunks of 8 elements
      const int half = idx >> 9, t = (idx >> 3) & 63, ch = idx & 7;
      const uint32_t off = (uint32_t)half * 16384u + sw_off(t, ch);
      const uint4 raw = *reinterpret_cast<const uint4*>(src + off);
      const uint32_t* rw = reinterpret_cast<const uint32_t*>(&raw);
      uint4 v;
      uint32_t* o = reinterpret_cast<uint32_t*>(&v);
      const float sc = rowf[t];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rw[e]));
        o[e] = pack_f16(f.x * sc, f.y * sc);
      }
      *reinterpret_cast<uint4*>(img + (uint32_t)half * 8192u + sw_off(t, ch)) = v;
    }
  };
  unsigned char* const qstage = sm + kV + 16384;
  if (writes_img) f16_image(sm + kKQ, sm + kST, KR);
  if (writes_img && p.q16) f16_image(sm + kKQ + 8192, qstage, QR);
  fence_async_smem();
  __syncthreads();
  if (early) {
    // Nothing up to the end of this CTA reads what the chunk-table kernel writes, and only
    // the status word is written by both: it is written here only after the wait at the
    // end (the debug build's index checks may write it anywhere, so that build waits here).
#ifdef GDN_DEBUG
    pdl_wait();
#endif
    pdl_release();
    prefetch_next_wave();
  }


  if (tid == 0) {
    const size_t img = ((size_t)wslot * p.H + h) * 64 * kDk * 2;
    if (writes_img && dbg_ok(wslot < p.nt_max && h < p.H, p.status)) {
      bulk_store(static_cast<unsigned char*>(p.k16) + img, sm + kST, 16384);
      if (p.q16) bulk_store(static_cast<unsigned char*>(p.q16) + img, qstage, 16384);
    }
    bulk_commit();
  }

  for (int rl = 0; rl < nr; ++rl) {
    const int r = r_begin + rl;  // (rl picks the V buffer and the barrier parities)
    const int hv = h * p.HG + r;
    const size_t sl = (size_t)wslot * p.Hv + hv;
    const uint32_t par = (uint32_t)(rl & 1);  // parity of this member's MMA barriers
    if (warp == 0) gates(r);  // (member 0's g and beta were loaded during the setup)
    // the previous member's w image read out of A/T (its u copies may still be reading)
    if (tid == 0 && rl > 0) bulk_wait_read<1>();
    __syncthreads();
    if (rl == 0) wait_or_flag(&bars[3], 0, fail);
    tc_fence_after();

    // A (TMEM lane quarters 0-1, rows of P) into A/T; M hi/lo image (quarters 2-3, rows of
    // R) into the Q halves; warps w and w + 4 share a lane quarter and take columns 0..31
    // and 32..63. Branch-free: every decay factor is formed and the mask is a select (exp
    // of a positive exponent above the diagonal may be inf; it is never used). Eight
    // columns per step, not unrolled, to keep the kernel's code small.
    {
      const int i = 32 * (warp & 1) + lane;
      const bool rows_p = (warp & 3) < 2;
      const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      const float gi = G[i];
      const float rowf = rows_p ? Bt[i] * KR[i] : qr;
      const int ch0 = 4 * (warp >> 2);
#pragma unroll 2
      for (int ch = ch0; ch < ch0 + 4; ++ch) {
        const int j = 8 * ch;
        float v[8];
        tmem_ld8(trow + j, v);
        const float4 ga = *reinterpret_cast<const float4*>(&G[j]);
        const float4 gb = *reinterpret_cast<const float4*>(&G[j + 4]);
        const float4 ka = *reinterpret_cast<const float4*>(&KR[j]);
        const float4 kb = *reinterpret_cast<const float4*>(&KR[j + 4]);
        const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
        const float kk[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
        float d[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) d[e] = __expf(gi - gg[e]) * rowf * kk[e];
        tmem_ld_wait();
        if (rows_p) {  // strictly lower
#pragma unroll
          for (int e = 0; e < 8; ++e) d[e] = (j + e < i) ? d[e] * v[e] : 0.f;
          *reinterpret_cast<float4*>(&AT[i * LDT + j]) = make_float4(d[0], d[1], d[2], d[3]);
          *reinterpret_cast<float4*>(&AT[i * LDT + j + 4]) = make_float4(d[4], d[5], d[6], d[7]);
        } else {  // lower, diagonal included
#pragma unroll
          for (int e = 0; e < 8; ++e) d[e] = (j + e <= i) ? d[e] * v[e] : 0.f;
          uint32_t hi[4], lo[4];
          if (p.m_f16) {
#pragma unroll
            for (int e = 0; e < 4; ++e) split_pack2_f16(d[2 * e], d[2 * e + 1], hi[e], lo[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) split_pack2(d[2 * e], d[2 * e + 1], hi[e], lo[e]);
          }
          const uint32_t off = sw_off(i, ch);
          *reinterpret_cast<uint4*>(sm + kKQ + 8192 + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm + kKQ + 24576 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == kMStoreThread) {  // (thread 0 leads the inverse's first step)
      size_t slm = sl;
#ifdef GDN_DEBUG
      // testing hook: one past the end of the M region (the next region follows it)
      if (p.dbg_poison && blockIdx.x == 0 && blockIdx.y == 0) slm = n_vslots;
#endif
      if (dbg_ok(slm < n_vslots, p.status)) {
        unsigned char* mimg = static_cast<unsigned char*>(p.M) + slm * 2 * 64 * 64 * 2;
        bulk_store(mimg, sm + kKQ + 8192, 8192);
        bulk_store(mimg + 8192, sm + kKQ + 24576, 8192);
      }
      bulk_commit();
    }
    tri_inverse_64_rd(AT, LDT, X, LDX, tid);  // ends with the CTA synchronized

    // This member's V tile (rows past the end zeroed) and the M image read out of the Q halves.
    wait_or_flag(&bars[1 + (rl & 1)], (uint32_t)((rl >> 1) & 1), fail);
    unsigned char* vt = sm + kV + (rl & 1) * 16384;
    if (L < kChunk) {
      zero_tail(vt, L, tid);
      zero_tail(vt + 8192, L, tid);
    }
    if (tid == kMStoreThread) bulk_wait_read<0>();  // the M image read out of the Q halves
    if (tid == 0) {
      // the k image (member 0) or the previous member's u blocks read out of the staging
      // region, and the q image out of the second V buffer
      bulk_wait_read<0>();
      if (rl == 0 && v1_late) issue_v(sm, bars, &tmv, hv + 1, t0, 1);  // into the q staging
    }
    __syncthreads();
    // T operand images: T diag(beta exp(G) / ||k||) (bf16) and T diag(beta) as a bf16
    // hi/lo pair (hi into the first Q half, lo into the second).
#pragma unroll 1
    for (int idx = tid; idx < 512; idx += kThreads) {
      const int i = idx >> 3, ch = idx & 7, j0 = 8 * ch;
      const float4 x0 = *reinterpret_cast<const float4*>(&AT[i * LDT + j0]);
      const float4 x1 = *reinterpret_cast<const float4*>(&AT[i * LDT + j0 + 4]);
      const float4 fa = *reinterpret_cast<const float4*>(&FW[j0]);
      const float4 fb = *reinterpret_cast<const float4*>(&FW[j0 + 4]);
      const float4 ba = *reinterpret_cast<const float4*>(&Bt[j0]);
      const float4 bb = *reinterpret_cast<const float4*>(&Bt[j0 + 4]);
      uint32_t th[4], tl[4];
      split_pack2(x0.x * ba.x, x0.y * ba.y, th[0], tl[0]);
      split_pack2(x0.z * ba.z, x0.w * ba.w, th[1], tl[1]);
      split_pack2(x1.x * bb.x, x1.y * bb.y, th[2], tl[2]);
      split_pack2(x1.z * bb.z, x1.w * bb.w, th[3], tl[3]);
      const uint4 tw = make_uint4(pack_bf16(x0.x * fa.x, x0.y * fa.y), pack_bf16(x0.z * fa.z, x0.w * fa.w),
                                  pack_bf16(x1.x * fb.x, x1.y * fb.y), pack_bf16(x1.z * fb.z, x1.w * fb.w));
      const uint32_t off = sw_off(i, ch);
      *reinterpret_cast<uint4*>(sm + kTW + off) = tw;
      *reinterpret_cast<uint4*>(sm + kKQ + 8192 + off) = make_uint4(th[0], th[1], th[2], th[3]);
      *reinterpret_cast<uint4*>(sm + kKQ + 24576 + off) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
    }
    fence_async_smem();
    __syncthreads();
    // TMEM: [P; R] in columns 0..63 (lanes 0..127), u^T in 64..127 (lanes 0..127), w in
    // 128..255 (lanes 32 q .. 32 q + 15 for rows 16 q .. 16 q + 15).
    const uint32_t dw = tmem + 128, du = tmem + 64;
    const uint32_t vb = sbase + kV + (rl & 1) * 16384;
    const uint32_t id_w = idesc_bf16_f32(64, 128, false, true);
    // u^T = V^T T_hi^T + V^T T_lo^T: A is the v tile read MN-major (M = the 128 value
    // columns, K = tokens), B the T_hi and T_lo images (K-major, N = 64 tokens). Row j of
    // D (TMEM lane j) is value column j, so a thread's TMEM row is one column of the
    // column-major u image.
    const uint32_t id_u = idesc_bf16_f32(128, 64, true, false);
    if (tid == 0) {
      tc_fence_after();
      // w = TW K: B is the k tile read MN-major (N = key dim, K = tokens)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(dw, sdesc_sw128(sbase + kTW + 32 * ks, 16, 1024),
                  sdesc_sw128(sbase + kKQ + 2048 * ks, 16384, 1024), id_w, ks > 0);
      umma_commit(&bars[4]);
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(du, sdesc_sw128(vb + 2048 * ks, 8192, 1024),
                    sdesc_sw128(sbase + kKQ + 8192 + 16384 * part + 32 * ks, 16, 1024), id_u,
                    part > 0 || ks > 0);
      umma_commit(&bars[5]);
    }
    wait_or_flag(&bars[4], par, fail);
    tc_fence_after();
    const bool bridge_ok = dbg_ok(sl < n_vslots, p.status);
    {  // w rows 16 q .. 16 q + 15 (TMEM lanes 32 q .., q = warp % 4), bf16, into the A/T
       // region; warps w and w + 4 take column blocks 0-1 and 2-3
      const int i = 16 * (warp & 3) + (lane & 15);
      unsigned char* img = sm + kAT;
#pragma unroll
      for (int cb = 2 * (warp >> 2); cb < 2 * (warp >> 2) + 2; ++cb) {
        float v[32];
        tmem_ld32(dw + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * cb, v);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = 32 * cb + 8 * q;
            const uint4 pk = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]),
                                        pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                        pack_bf16(v[8 * q + 4], v[8 * q + 5]),
                                        pack_bf16(v[8 * q + 6], v[8 * q + 7]));
            *reinterpret_cast<uint4*>(img + (col >> 6) * 8192 + sw_off(i, (col & 63) >> 3)) = pk;
          }
        }
      }
    }
    // the w image leaves while the u^T rows are read out (its own bulk group: the next
    // member's A overwrites the A/T region once it has been read)
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      if (bridge_ok)
        bulk_store(static_cast<unsigned char*>(p.w) + sl * 64 * kDk * 2, sm + kAT, 16384);
      bulk_commit();
    }
    // u^T: value column 32 q + lane (TMEM lane quarter q = warp % 4), tokens 32 th ..
    // 32 th + 31 (th = warp / 4), into block q of the u image: blocks 0, 1 staged in this
    // member's V buffer (the u MMAs have read the tile), 2, 3 in the staging region
    wait_or_flag(&bars[5], par, fail);
    tc_fence_after();
    auto u_stage = [&](int b) {
      return b < 2 ? vt + 8192 * b : sm + kST + 8192 * (b - 2);
    };
    {
      const int q = warp & 3, th = warp >> 2, j = lane;
      float v[32];
      tmem_ld32(du + ((uint32_t)(32 * q) << 16) + 32 * th, v);
      tmem_ld_wait();
      unsigned char* blk = u_stage(q);
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {  // 8-token group 4 th + gi: 32 bytes, swizzled by j
        const uint32_t off = (uint32_t)j * 256u + ((uint32_t)((4 * th + gi) ^ (j & 7)) << 5);
        *reinterpret_cast<float4*>(blk + off) =
            make_float4(v[8 * gi], v[8 * gi + 1], v[8 * gi + 2], v[8 * gi + 3]);
        *reinterpret_cast<float4*>(blk + off + 16) =
            make_float4(v[8 * gi + 4], v[8 * gi + 5], v[8 * gi + 6], v[8 * gi + 7]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      if (bridge_ok) {
        unsigned char* uimg = reinterpret_cast<unsigned char*>(p.u + sl * 64 * kDv);
#pragma unroll
        for (int b = 0; b < 4; ++b) bulk_store(uimg + b * 8192, u_stage(b), 8192);
      }
      bulk_commit();
    }
    if (tid == 0 && rl + 2 < nr) {  // this V buffer serves member r + 2 once the copies read it
      bulk_wait_read<0>();
      issue_v(sm, bars, &tmv, hv + 2, t0, rl + 2);
    }
  }

  if (early) {
#ifndef GDN_DEBUG
    pdl_wait();  // the status word is cleared and the table written from here on
#endif
    if (tid == 0) {  // cross-check: the table maps slot s to chunk s of sequence 0
      const int2 e = p.chunk_table[slot];
      if (e.x != 0 || e.y != slot) set_status(p.status, GDN_DEV_BAD_CHUNK_TABLE);
    }
  }
  if (tid == 0) {
    bulk_wait_read<0>();  // every image read out (the grid's end completes the writes)
    for (int rl = max(0, nr - 2); rl < nr; ++rl)  // (all V loads were consumed; bounded)
      mbar_wait(&bars[1 + (rl & 1)], (uint32_t)((rl >> 1) & 1), kWaitIters);
    if (*fail) set_status(p.status, GDN_DEV_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool launch_tc_intra(const Params& p, cudaStream_t s) {
  CUtensorMap tmk, tmq, tmv;
  const int rows = p.T > 0 ? p.T : 1;  // with T = 0 every slot is a sentinel
  if (!encode_rows_tmap(&tmk, p.k, rows, p.H, p.D) ||
      !encode_rows_tmap(&tmq, p.q, rows, p.H, p.D) ||
      !encode_rows_tmap(&tmv, p.v, rows, p.Hv, p.D))
    return false;
  ensure_smem_limit((const void*)tc_intra_kernel, (int)kSmemBytes);
  return launch_pdl(tc_intra_kernel, dim3(p.H, p.nt_max + p.split_slots), dim3(kThreads),
                    kSmemBytes, s, p, tmk,
                    tmq, tmv) == cudaSuccess;
}

}  // namespace gdn
