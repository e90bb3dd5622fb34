// Reverse scan of the backward pass on warp-level tensor-core MMAs (bf16 inputs, head
// size 128, or 64 zero-padded to 128; scalar gates): the state-gradient recurrence of the chunked gated delta
// rule, walking the chunks of each (sequence, value head, 32-column value block) from
// last to first.
//
// The stage is the state-gradient scan of the backward kernels listed in the FLA
// graph-capture RFC ("What needs to change", GDN bwd). With the forward's chunk
// quantities (w, M = Gamma * (Q K^T), the in-chunk gate sums G) and dS the gradient
// of the next chunk-start state, each chunk computes
//   dv_new = exp(G_L - G) * (K dS) + scale M^T dO
//   dS    <- exp(G_L) dS + scale Q^T (exp(G) * dO) - w^T dv_new
// and stores the incoming dS and dv_new for the per-chunk gradient kernels. The two
// products that read dS or dv_new are the serial chain; M^T dO and Q^T (exp(G) dO)
// only read the chunk's inputs.
//
// Layout, as in the forward scan: 8 compute warps hold dS (128 key rows x 32 value
// columns, fp32) as MMA accumulators, warp w owning key rows 16w..16w+15; one load warp
// brings each chunk's k and q tiles (TMA, 128-byte swizzle), the w and [M_hi; M_lo]
// images of the forward's bridge and G into a two-slot ring one chunk ahead. The
// operands the warps produce (dS, dv_new, dO and exp(G) dO) are written to shared memory
// as bf16 hi/lo pairs (about 16 significant bits each; a bf16 dO is exact), so every
// product takes the hi and lo terms of its fp32 operand against an exact bf16 input
// (k, q) or a bridge image (w, M). Rows past the end of a sequence: dO is read as zero
// (which also cancels the q rows there) and dv_new is zero (the k rows there belong to
// the next sequence and are masked). Every wait is bounded (GDN_DEV_TIMEOUT on expiry).
#include <cuda.h>

#include "gdn_common.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int kD = 128;  // key rows of the computed state (a head size of 64 is zero-padded)
constexpr int BV = 32;
constexpr int kCompWarps = 8;
constexpr int kLoadWarp = kCompWarps;
constexpr int kThreads = (kCompWarps + 1) * 32;
constexpr int kCompThreads = kCompWarps * 32;
constexpr uint32_t kWaitIters = 1u << 22;

// Ring slot (bytes from a 1024-aligned base): k and q tiles (two swizzled [64 rows][128 B]
// key-dim halves each), the w image (same layout), [M_hi; M_lo] ([128 rows][128 B],
// swizzled) and G [64].
constexpr uint32_t sK = 0, sQ = 16384, sW = 32768, sM = 49152, sG = 65536;
constexpr uint32_t kSlot = 66560;
constexpr uint32_t kTx = 4 * 16384 + 256;
constexpr int kRing = 2;
// Operands written by the warps: no-swizzle MN-major core matrices (n-block stride 128 B,
// stride 1024 B between 8-deep K groups); hi in columns 0..31, lo in 32..63.
constexpr uint32_t oDS = kRing * kSlot;  // dS split, K = 128 key rows
constexpr uint32_t oVN = oDS + 16384;    // dv_new split, K = 64 tokens
constexpr uint32_t oFQ = oVN + 8192;     // exp(G) dO split
constexpr uint32_t oDO = oFQ + 8192;     // dO split
constexpr uint32_t oBar = oDO + 8192;    // full[2], empty[2]
constexpr uint32_t oMisc = oBar + 64;    // abort flag
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

__device__ __forceinline__ uint32_t mn_off(int n, int k) {
  return (uint32_t)(n >> 3) * 128u + (uint32_t)(k >> 3) * 1024u + (uint32_t)(k & 7) * 16u +
         (uint32_t)(n & 7) * 2u;
}
__device__ __forceinline__ uint32_t sw_chunk(int row, int col) {
  return (uint32_t)row * 128u + ((uint32_t)((col >> 3) ^ (row & 7)) << 4);
}
// Lane address of ldmatrix.x4.trans for the B fragments of two n-tiles (n0.., n0 + 8..)
// over k0..k0 + 15 of an MN-major operand.
__device__ __forceinline__ uint32_t b_lane(int n0, int k0, int lane) {
  const int i = lane >> 3;
  const int nn = n0 + (i >> 1) * 8, kk = k0 + (i & 1) * 8;
  return (uint32_t)(nn >> 3) * 128u + (uint32_t)(kk >> 3) * 1024u + (uint32_t)(lane & 7) * 16u;
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitIters; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_scan_tc_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmq) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);  // 0-1 slot landed, 2-3 slot consumed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + oMisc);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * BV, h = hv / p.HG;
  const size_t state_base = ((size_t)n * p.Hv + hv) * D * D;  // [dv][dk] with head size D

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], kCompWarps);
    mbar_init(&bars[3], kCompWarps);
    mbar_init_fence();
    *abort_flag = 0;
  }
  __syncthreads();
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }

  if (warp == kLoadWarp) {
    if (lane == 0) {
      int issued = 0;
      for (int m = 0; m < nch; ++m) {
        const int c = nch - 1 - m, s = m & 1;
        if (m >= kRing && !wait_phase(&bars[2 + s], (uint32_t)(((m - kRing) >> 1) & 1), abort_flag))
          break;
        const size_t sl = (size_t)(sv.first_slot + c) * p.Hv + hv;
        const int t0 = sv.start + kChunk * c;
        unsigned char* st = sm + s * kSlot;
        uint64_t* full = &bars[s];
        mbar_expect_tx(full, kTx);
        tma_load_3d(st + sK, &tmk, 0, h, t0, full);
        tma_load_3d(st + sK + 8192, &tmk, 64, h, t0, full);
        tma_load_3d(st + sQ, &tmq, 0, h, t0, full);
        tma_load_3d(st + sQ + 8192, &tmq, 64, h, t0, full);
        bulk_load(st + sW, static_cast<const unsigned char*>(p.wimg) + sl * 16384, 16384, full);
        bulk_load(st + sM, static_cast<const unsigned char*>(p.mimg) + sl * 16384, 16384, full);
        bulk_load(st + sG, p.G + sl * 64, 256, full);
        issued = m + 1;
      }
      // Before the CTA retires, the copies it issued have landed (bounded).
      for (int m = max(0, issued - kRing); m < issued; ++m)
        mbar_wait(&bars[m & 1], (uint32_t)((m >> 1) & 1), kWaitIters);
    }
  } else {
    const int g = lane >> 2, c2 = 2 * (lane & 3), i8 = lane >> 3;
    const int mt = warp & 3, np = warp >> 2;  // dv_new tile: token rows 16mt.., columns 16np..
    // With a head size of 64 the upper key half is zero (the k tile reads the TMA fill there):
    // K dS contracts over D key rows only, and the warps whose dS rows lie past D (never
    // stored, never read) skip their products. They still take every barrier.
    constexpr int nks = D / 16;
    const bool live = 16 * warp < D;  // always at D = 128
    // dS: key rows 16 warp + g (+8), value columns 8 nt + c2 (+1)
    float dS[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
        dS[nt][e] = (p.dfin && d < D) ? p.dfin[state_base + (size_t)(c0 + j) * D + d] : 0.f;
      }
    auto store_ds_split = [&]() {
      unsigned char* b = sm + oDS;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int d = 16 * warp + g + 8 * hh, j = 8 * nt + c2;
          uint32_t hi, lo;
          split_pack2(dS[nt][2 * hh], dS[nt][2 * hh + 1], hi, lo);
          *reinterpret_cast<uint32_t*>(b + mn_off(j, d)) = hi;
          *reinterpret_cast<uint32_t*>(b + mn_off(32 + j, d)) = lo;
        }
    };
    // dO of a chunk: thread t holds row t / 4, columns 8 (t % 4) .. + 7 of this block,
    // loaded one chunk ahead; rows past the sequence end are zero.
    const int pr = tid >> 2, pq = 8 * (tid & 3);
    float od[8];
    auto load_do = [&](int c) {
      const int t0 = sv.start + kChunk * c, L = min(kChunk, sv.len - kChunk * c);
      if (pr < L) {
        const size_t idx = ((size_t)(t0 + pr) * p.Hv + hv) * D + c0 + pq;
        if (p.dout_bf16) {
          const uint4 r = *reinterpret_cast<const uint4*>(
              reinterpret_cast<const __nv_bfloat16*>(p.dout) + idx);
          const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
            od[2 * e] = f.x;
            od[2 * e + 1] = f.y;
          }
        } else {
          const float* src = reinterpret_cast<const float*>(p.dout) + idx;
          const float4 a = *reinterpret_cast<const float4*>(src);
          const float4 b = *reinterpret_cast<const float4*>(src + 4);
          od[0] = a.x; od[1] = a.y; od[2] = a.z; od[3] = a.w;
          od[4] = b.x; od[5] = b.y; od[6] = b.z; od[7] = b.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) od[e] = 0.f;
      }
    };
    if (nch > 0) {
      store_ds_split();
      load_do(nch - 1);
    }

    for (int m = 0; m < nch; ++m) {
      const int c = nch - 1 - m, s = m & 1;
      const size_t sl = (size_t)(sv.first_slot + c) * p.Hv + hv;
      const int L = min(kChunk, sv.len - kChunk * c);
      unsigned char* st = sm + s * kSlot;
      const uint32_t st_a = sbase + s * kSlot;
      {  // the incoming gradient is this chunk's dS_next: kept for the chunk kernels
        float* dh = p.dhs + sl * D * D;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
            if (d < D) dh[(size_t)(c0 + j) * D + d] = dS[nt][e];
          }
      }
      wait_phase(&bars[s], (uint32_t)((m >> 1) & 1), abort_flag);
      const float* G = reinterpret_cast<const float*>(st + sG);
      {  // dO and exp(G) dO operands (bf16 hi/lo)
        const float fq = expf(G[pr]);
        uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          split_pack2(od[2 * e], od[2 * e + 1], h1[e], l1[e]);
          split_pack2(fq * od[2 * e], fq * od[2 * e + 1], h2[e], l2[e]);
        }
        const uint32_t ohi = mn_off(pq, pr), olo = mn_off(32 + pq, pr);
        *reinterpret_cast<uint4*>(sm + oDO + ohi) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        *reinterpret_cast<uint4*>(sm + oDO + olo) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
        *reinterpret_cast<uint4*>(sm + oFQ + ohi) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
        *reinterpret_cast<uint4*>(sm + oFQ + olo) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
      }
      if (m + 1 < nch) load_do(c - 1);  // in flight while this chunk is processed
      named_sync(1, kCompThreads);       // dO operands and the dS split visible

      // K dS (chain) and M^T dO: token rows 16mt.., columns 16np..16np+15
      float x1[2][4], x2[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) x1[q][e] = x2[q][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        if (ks >= nks) break;
        uint32_t a[4], bh[4], bl[4];
        const int row = 16 * mt + (lane & 7) + (i8 & 1) * 8;
        const int col = (16 * ks + (i8 >> 1) * 8) & 63;
        ldsm_x4_addr(a, st_a + sK + (ks >> 2) * 8192 + sw_chunk(row, col));
        const uint32_t bo = sbase + oDS + b_lane(16 * np, 16 * ks, lane);
        ldsm_x4_t_addr(bh, bo);
        ldsm_x4_t_addr(bl, bo + 512);
        mma_bf16(x1[0], a, bh[0], bh[1]);
        mma_bf16(x1[1], a, bh[2], bh[3]);
        mma_bf16(x1[0], a, bl[0], bl[1]);
        mma_bf16(x1[1], a, bl[2], bl[3]);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // A = M^T: image rows are the contraction index
        uint32_t ah[4], al[4], bh[4];
        const int t = 16 * ks + (i8 >> 1) * 8 + (lane & 7);
        const int col = 16 * mt + (i8 & 1) * 8;
        ldsm_x4_t_addr(ah, st_a + sM + sw_chunk(t, col));
        ldsm_x4_t_addr(al, st_a + sM + sw_chunk(64 + t, col));
        const uint32_t bo = sbase + oDO + b_lane(16 * np, 16 * ks, lane);
        ldsm_x4_t_addr(bh, bo);
        mma_bf16(x2[0], ah, bh[0], bh[1]);
        mma_bf16(x2[1], ah, bh[2], bh[3]);
        mma_bf16(x2[0], al, bh[0], bh[1]);
        mma_bf16(x2[1], al, bh[2], bh[3]);
        if (!p.dout_bf16) {  // an fp32 dO carries a lo half
          uint32_t bl[4];
          ldsm_x4_t_addr(bl, bo + 512);
          mma_bf16(x2[0], ah, bl[0], bl[1]);
          mma_bf16(x2[1], ah, bl[2], bl[3]);
        }
      }
      // Q^T (exp(G) dO): key rows 16 warp.., all 32 columns (no dS in it)
      float y1[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) y1[nt][e] = 0.f;
      const int arow = 16 * (warp & 3) + (i8 & 1) * 8;  // this warp's key rows in its half
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (!live) break;
        uint32_t a[4];
        const int t = 16 * ks + (i8 >> 1) * 8 + (lane & 7);
        ldsm_x4_t_addr(a, st_a + sQ + (warp >> 2) * 8192 + sw_chunk(t, arow));
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          uint32_t bh[4], bl[4];
          const uint32_t bo = sbase + oFQ + b_lane(16 * p2, 16 * ks, lane);
          ldsm_x4_t_addr(bh, bo);
          ldsm_x4_t_addr(bl, bo + 512);
          mma_bf16(y1[2 * p2], a, bh[0], bh[1]);
          mma_bf16(y1[2 * p2 + 1], a, bh[2], bh[3]);
          mma_bf16(y1[2 * p2], a, bl[0], bl[1]);
          mma_bf16(y1[2 * p2 + 1], a, bl[2], bl[3]);
        }
      }
      // dv_new = exp(G_L - G) (K dS) + scale M^T dO; rows past the sequence end are zero
      {
        unsigned char* vn = sm + oVN;
        const float gl = G[63];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 16 * mt + g + 8 * hh;
          const float fk = i < L ? expf(gl - G[i]) : 0.f;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int j = 16 * np + 8 * q + c2;
            const float v0 = fmaf(fk, x1[q][2 * hh], p.scale * x2[q][2 * hh]);
            const float v1 = fmaf(fk, x1[q][2 * hh + 1], p.scale * x2[q][2 * hh + 1]);
            *reinterpret_cast<float2*>(p.dvn + (sl * 64 + i) * D + c0 + j) = make_float2(v0, v1);
            uint32_t hi, lo;
            split_pack2(v0, v1, hi, lo);
            *reinterpret_cast<uint32_t*>(vn + mn_off(j, i)) = hi;
            *reinterpret_cast<uint32_t*>(vn + mn_off(32 + j, i)) = lo;
          }
        }
      }
      named_sync(1, kCompThreads);  // dv_new visible to every warp

      // dS <- exp(G_L) dS + scale Q^T (exp(G) dO) - w^T dv_new
      if (live) {
        float y2[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) y2[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4];
          const int t = 16 * ks + (i8 >> 1) * 8 + (lane & 7);
          ldsm_x4_t_addr(a, st_a + sW + (warp >> 2) * 8192 + sw_chunk(t, arow));
#pragma unroll
          for (int p2 = 0; p2 < 2; ++p2) {
            uint32_t bh[4], bl[4];
            const uint32_t bo = sbase + oVN + b_lane(16 * p2, 16 * ks, lane);
            ldsm_x4_t_addr(bh, bo);
            ldsm_x4_t_addr(bl, bo + 512);
            mma_bf16(y2[2 * p2], a, bh[0], bh[1]);
            mma_bf16(y2[2 * p2 + 1], a, bh[2], bh[3]);
            mma_bf16(y2[2 * p2], a, bl[0], bl[1]);
            mma_bf16(y2[2 * p2 + 1], a, bl[2], bl[3]);
          }
        }
        const float gam = expf(G[63]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dS[nt][e] = fmaf(gam, dS[nt][e], fmaf(p.scale, y1[nt][e], -y2[nt][e]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[2 + s]);  // this warp is done with the ring slot
      // split of the updated dS for the next chunk (every warp has passed this chunk's
      // K dS, so the buffer is free; the next chunk's first barrier publishes it)
      if (m + 1 < nch && live) store_ds_split();
    }
    if (p.dh0) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = 16 * warp + g + (e >> 1) * 8, j = 8 * nt + c2 + (e & 1);
          if (d < D) p.dh0[state_base + (size_t)(c0 + j) * D + d] = dS[nt][e];
        }
    }
  }
  __syncthreads();
  if (tid == 0 && *abort_flag) set_status(p.status, GDN_DEV_TIMEOUT);
}

}  // namespace

bool launch_bwd_scan_tc(const BwdParams& p, int D, cudaStream_t s) {
  if (D != 64 && D != kD) return false;
  CUtensorMap tmk, tmq;
  const int rows = p.T > 0 ? p.T : 1;  // with T = 0 no tile is ever loaded
  // With D = 64 the second key-dim half of every k and q tile lies outside the tensor and
  // is filled with zeros, and so are the bridge's w columns 64..127: the padded rows of
  // dS stay zero.
  if (!encode_rows_tmap(&tmk, p.k, rows, p.H, D) || !encode_rows_tmap(&tmq, p.q, rows, p.H, D))
    return false;
  if (D == kD) {
    ensure_smem_limit((const void*)bwd_scan_tc_kernel<kD>, (int)kSmemBytes);
    bwd_scan_tc_kernel<kD><<<dim3(p.N, p.Hv, D / BV), kThreads, kSmemBytes, s>>>(p, tmk, tmq);
  } else {
    ensure_smem_limit((const void*)bwd_scan_tc_kernel<64>, (int)kSmemBytes);
    bwd_scan_tc_kernel<64><<<dim3(p.N, p.Hv, D / BV), kThreads, kSmemBytes, s>>>(p, tmk, tmq);
  }
  return cudaPeekAtLastError() == cudaSuccess;
}

}  // namespace gdn
