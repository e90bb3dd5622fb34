// Intra-chunk kernel for per-channel gates (bf16 inputs) on warp-level tensor-core
// MMAs: one CTA of 16 warps per (chunk, value head). It writes the bridge the tensor-core
// scan reads in its per-channel mode.
//
// With G the in-chunk cumulative log-decay of each key channel d (gates g <= 0, so G is
// non-increasing along the chunk):
//   A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd)   (j < i)        T = (I + A)^-1
//   M_ij =        sum_d q_id k_jd exp(G_id - G_jd)   (j <= i)
//   w    = T diag(beta) (exp(G) * k),   u = T diag(beta) v
// (the chunked form of the per-channel delta rule, "Optimizing GDN Chunk Prefill on Intel
// AMX CPU", sections 4-5, with the scalar decay replaced by one per key channel).
//
// A and M as tensor-core products. The 64 rows are cut into 16-row blocks. For two
// blocks bi > bj the entries are products of k_i exp(G_i - G_r) and k_j exp(G_r - G_j)
// with the reference row r = 16 bi: both factors are <= 1. Inside a diagonal block the
// reference is the block's middle row m = 16 b + 8, so the factors are bounded by
// exp(R / 2) with R the block's largest gate range over its 16 rows; for R <= 80 every
// factor stays inside fp32 and bf16 range, and a block with a larger range is formed
// entry by entry instead (exp(G_i - G_j) <= 1). The factors are split into bf16 hi + lo
// (about 16 significant bits) and multiplied as hi*hi + hi*lo + lo*hi with fp32
// accumulation, 32 channels at a time.
//
// Outputs per (chunk, value head), in the layouts of the scalar-gate path's bridge:
//   w (bf16, two 64-column halves of [64][128 B], 128-byte swizzle), u (fp32, [4 blocks
//   of 32 columns][64][32], 16-byte chunks swizzled), M (bf16 hi then lo, [128][128 B],
//   swizzled), and for the scan's per-channel mode: exp(G_L - G) * k (fp16, the state
//   update's operand), exp(G) * q as a bf16 hi/lo pair (the output's operand; one bf16
//   rounding of it would cost about 1e-2 of the output's rms) and exp(G_L) per channel.
#include <cuda.h>

#include "gdn_common.cuh"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int kThr = 512;
constexpr int kWarps = kThr / 32;
constexpr int LDT = 68;     // fp32 stride of the A / T tile
constexpr int LI = 40;      // bf16 stride of image rows (80 B: ldmatrix rows conflict-free)
constexpr int LTW = 72;     // bf16 stride of the T operand rows (144 B)
constexpr int LKG = 136;    // bf16 stride of the exp(G) k rows (272 B)
constexpr float kDiagRange = 80.f;
constexpr uint32_t kWaitIters = 1u << 22;

// Image rows (each stored hi, then lo): E side of the A / M products with the
// off-diagonal reference (k, q), with the diagonal reference (k, q); F side with the
// diagonal reference (k); F side of the six off-diagonal pairs (k).
constexpr int R_EK = 0, R_EQ = 64, R_DK = 128, R_DQ = 192, R_FD = 256, R_FO = 320, R_IMG = 416;

// Shared memory (bytes from a 1024-aligned base)
constexpr uint32_t sK = 0;                         // k, q, v tiles (TMA, 128-byte swizzle)
constexpr uint32_t sQ = 16384;
constexpr uint32_t sV = 32768;
// The gates' row stride: 132 floats, so that the rows a warp reads in one step fall in
// different shared-memory banks (with 128 every row starts in bank 0).
constexpr int GS = 132;
constexpr uint32_t sG = 49152;                     // fp32 [64][GS]; later the u staging
constexpr uint32_t sIMG = sG + 64 * GS * 4;        // images; later T operands and w staging
constexpr uint32_t sIMGsz = 2 * R_IMG * LI * 2;
constexpr uint32_t sKG = sIMG + sIMGsz;            // bf16 [64][LKG]: exp(G) k / ||k||
constexpr uint32_t sAT = sKG + 64 * LKG * 2;       // fp32 [64][LDT]: A, then T
constexpr uint32_t sX = sAT + 64 * LDT * 4;        // fp32 [16][LDT]: scratch of the inverse
constexpr uint32_t sM = sX + 16 * LDT * 4;         // M image (hi rows 0..63, lo rows 64..127)
constexpr uint32_t sVec = sM + 16384;              // beta, 1/||k||, 1/||q||, flags
constexpr uint32_t sBar = sVec + 4 * 256;
constexpr uint32_t kSmemBytes = sBar + 64 + 1024;
static_assert(2 * 64 * LTW * 2 + 16384 <= sIMGsz, "T operands and w staging exceed the image region");
static_assert(kSmemBytes <= 232448, "shared memory over the per-CTA limit");

__device__ __forceinline__ uint32_t sw_off(int r, int ch) {
  return (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4);
}
// Byte offset of fp32 element (r, j), j < 32, in a [rows][32] tile with 16-byte chunks swizzled.
__device__ __forceinline__ uint32_t u_offset(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)((j >> 2) ^ (r & 7)) << 4) + (uint32_t)(j & 3) * 4u;
}
// Eight bf16 of row r, features 8 ch .. 8 ch + 7, of a two-half swizzled [64][128] tile.
__device__ __forceinline__ void tile_row8(const unsigned char* tile, int r, int ch, float (&x)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(tile + (ch >> 3) * 8192 + sw_off(r, ch & 7));
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ float tile_elem(const unsigned char* tile, int r, int f) {
  const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(
      tile + (f >> 6) * 8192 + sw_off(r, (f & 63) >> 3));
  return __bfloat162float(e[f & 7]);
}

__global__ void __launch_bounds__(kThr, 1)
kda_intra_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* G = reinterpret_cast<float*>(sm + sG);
  __nv_bfloat16* IMG = reinterpret_cast<__nv_bfloat16*>(sm + sIMG);
  __nv_bfloat16* KG = reinterpret_cast<__nv_bfloat16*>(sm + sKG);
  float* AT = reinterpret_cast<float*>(sm + sAT);
  float* X = reinterpret_cast<float*>(sm + sX);
  float* Bt = reinterpret_cast<float*>(sm + sVec);
  float* KR = Bt + 64;
  float* QR = KR + 64;
  int* flags = reinterpret_cast<int*>(QR + 64);  // [0] unsafe diagonal blocks, [1] failure
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + sBar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hv = blockIdx.y, h = hv / p.HG;
  pdl_wait();     // the chunk table (and the L2-norm factors) are written
  pdl_release();  // the scan may take SMs as this grid drains
  int t0, L, wslot;
  if (!resolve_slot(p, blockIdx.x, t0, L, wslot)) return;  // uniform over the CTA
  const size_t sl = (size_t)wslot * p.Hv + hv;

  if (tid == 0) {
    flags[0] = 0;
    flags[1] = 0;
    mbar_init(bar, 1);
    mbar_init_fence();
    mbar_expect_tx(bar, 49152);
    tma_load_3d(sm + sK, &tmk, 0, h, t0, bar);
    tma_load_3d(sm + sK + 8192, &tmk, 64, h, t0, bar);
    tma_load_3d(sm + sQ, &tmq, 0, h, t0, bar);
    tma_load_3d(sm + sQ + 8192, &tmq, 64, h, t0, bar);
    tma_load_3d(sm + sV, &tmv, 0, hv, t0, bar);
    tma_load_3d(sm + sV + 8192, &tmv, 64, hv, t0, bar);
  }
  __syncthreads();  // the barrier and the flags are initialised before anyone waits
  // gate rows (16-byte pieces; zero past the chunk end and for channels past D)
  for (int idx = tid; idx < 64 * 32; idx += kThr) {
    const int i = idx >> 5, c4 = (idx & 31) * 4;
    const bool ok = i < L && c4 < p.D;
    cp_async16(G + i * GS + c4, p.g + (((size_t)(ok ? t0 + i : t0) * p.Hv + hv) * p.D + (ok ? c4 : 0)),
               ok);
  }
  cp_async_commit();
  if (tid < 64) {
    const bool ok = tid < L;
    const size_t row = (size_t)(t0 + tid);
    Bt[tid] = ok ? p.beta[row * p.Hv + hv] : 0.f;
    KR[tid] = (ok && p.krn) ? p.krn[row * p.H + h] : 1.f;
    QR[tid] = (ok && p.qrn) ? p.qrn[row * p.H + h] : 1.f;
  }
  cp_async_wait<0>();
  if (!mbar_wait(bar, 0, kWaitIters)) flags[1] = 1;
  __syncthreads();
  // rows past the sequence end of the tiles read as zero (they hold the next sequence)
  for (int idx = tid; idx < 6 * (64 - L) * 8; idx += kThr) {
    const int part = idx / ((64 - L) * 8), rem = idx % ((64 - L) * 8);
    *reinterpret_cast<uint4*>(sm + sK + part * 8192 + (uint32_t)(L + (rem >> 3)) * 128u +
                              (rem & 7) * 16u) = make_uint4(0u, 0u, 0u, 0u);
  }
  {  // inclusive cumsum along the chunk: four threads per channel, 16 rows each, then each
     // segment adds the totals of the segments before it (in order), through X as scratch
    const int chn = tid & 127, seg = tid >> 7;
    float x[16], acc = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      acc += G[(16 * seg + r) * GS + chn];
      x[r] = acc;
    }
    X[seg * 128 + chn] = acc;
    __syncthreads();
    float off = 0.f;
    for (int s2 = 0; s2 < seg; ++s2) off += X[s2 * 128 + chn];
#pragma unroll
    for (int r = 0; r < 16; ++r) G[(16 * seg + r) * GS + chn] = x[r] + off;
  }
  for (int idx = tid; idx < 16384 / 16; idx += kThr)
    reinterpret_cast<uint4*>(sm + sM)[idx] = make_uint4(0u, 0u, 0u, 0u);
  for (int idx = tid; idx < 64 * LDT; idx += kThr) AT[idx] = 0.f;
  __syncthreads();
  if (tid < 128) {  // diagonal blocks whose gate range is too wide for the middle reference
    int bad = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (G[16 * b * GS + tid] - G[(16 * b + 15) * GS + tid] > kDiagRange) bad |= 1 << b;
    if (bad) atomicOr(&flags[0], bad);
  }

  // ---------------- decayed k (fp16), decayed q (bf16 hi/lo), exp(G) k (w operand), exp(G_L)
  {
    unsigned char* img = sm + sIMG;  // [k16 | q hi | q lo], each two 8 KB halves
    for (int idx = tid; idx < 64 * 16; idx += kThr) {
      const int i = idx >> 4, ch = idx & 15;
      float kx[8], qx[8];
      tile_row8(sm + sK, i, ch, kx);
      tile_row8(sm + sQ, i, ch, qx);
      uint32_t kt[4], qh[4], ql[4], kg[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int f = 8 * ch + e;
        const float gi0 = G[i * GS + f], gi1 = G[i * GS + f + 1];
        const float gl0 = G[63 * GS + f], gl1 = G[63 * GS + f + 1];
        const float k0 = kx[e] * KR[i], k1 = kx[e + 1] * KR[i];
        kt[e >> 1] = pack_f16(__expf(gl0 - gi0) * k0, __expf(gl1 - gi1) * k1);
        const float e0 = __expf(gi0), e1 = __expf(gi1);
        split_pack2(e0 * qx[e] * QR[i], e1 * qx[e + 1] * QR[i], qh[e >> 1], ql[e >> 1]);
        kg[e >> 1] = pack_bf16(e0 * k0, e1 * k1);
      }
      const uint32_t off = (ch >> 3) * 8192 + sw_off(i, ch & 7);
      *reinterpret_cast<uint4*>(img + off) = make_uint4(kt[0], kt[1], kt[2], kt[3]);
      *reinterpret_cast<uint4*>(img + 16384 + off) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
      *reinterpret_cast<uint4*>(img + 32768 + off) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
      *reinterpret_cast<uint4*>(KG + i * LKG + 8 * ch) = make_uint4(kg[0], kg[1], kg[2], kg[3]);
    }
    for (int f = tid; f < 128; f += kThr) p.gam[sl * 128 + f] = __expf(G[63 * GS + f]);
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_store(static_cast<unsigned char*>(p.k16) + sl * 16384, img, 16384);
      bulk_store(static_cast<unsigned char*>(p.qimg) + sl * 32768, img + 16384, 32768);
      bulk_commit();
      bulk_wait_read<0>();  // the image region is rewritten next
    }
    __syncthreads();
  }

  // ---------------- A and M: 20 blocks of 16 x 16 over four chunks of 32 channels
  // blocks 0-5: A of pair p, 6-11: M of pair p, 12-15: A of diagonal block b, 16-19: M
  // pairs (bi, bj), bj < bi: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
  auto pair_bi = [](int pr) { return pr < 1 ? 1 : (pr < 3 ? 2 : 3); };
  constexpr int kBlkPerWarp = (20 + kWarps - 1) / kWarps;
  float acc[kBlkPerWarp][2][4];
#pragma unroll
  for (int s = 0; s < kBlkPerWarp; ++s)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[s][nt][e] = 0.f;
#pragma unroll 1
  for (int fc = 0; fc < 4; ++fc) {
    // images of channels 32 fc .. 32 fc + 31: 416 rows x 4 groups of 8 channels
    for (int it = tid; it < R_IMG * 4; it += kThr) {
      const int R = it >> 2, fg = it & 3, f0 = 32 * fc + 8 * fg;
      int src, ref;           // token row and reference row
      bool from_q = false, ref_first = true;  // exp(G_src - G_ref) or exp(G_ref - G_src)
      if (R < R_DK) {                           // off-diagonal E rows (k, then q)
        src = R & 63;
        from_q = R >= R_EQ;
        ref = src & ~15;
      } else if (R < R_FD) {                    // diagonal E rows
        src = R & 63;
        from_q = R >= R_DQ;
        ref = (src & ~15) + 8;
      } else if (R < R_FO) {                    // diagonal F rows
        src = R - R_FD;
        ref = (src & ~15) + 8;
        ref_first = false;
      } else {                                  // off-diagonal F rows of pair pr
        const int c = R - R_FO, pr = c >> 4, bi = pair_bi(pr), bj = pr - (bi * (bi - 1)) / 2;
        src = 16 * bj + (c & 15);
        ref = 16 * bi;
        ref_first = false;
      }
      float x[8];
      tile_row8(from_q ? sm + sQ : sm + sK, src, f0 >> 3, x);
      const float rs = from_q ? QR[src] : KR[src];
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float gs0 = G[src * GS + f0 + e], gs1 = G[src * GS + f0 + e + 1];
        const float gr0 = G[ref * GS + f0 + e], gr1 = G[ref * GS + f0 + e + 1];
        const float d0 = ref_first ? gs0 - gr0 : gr0 - gs0;
        const float d1 = ref_first ? gs1 - gr1 : gr1 - gs1;
        split_pack2(x[e] * rs * __expf(d0), x[e + 1] * rs * __expf(d1), hi[e >> 1], lo[e >> 1]);
      }
      *reinterpret_cast<uint4*>(IMG + R * LI + 8 * fg) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(IMG + (R_IMG + R) * LI + 8 * fg) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kBlkPerWarp; ++s) {
      const int blk = warp + kWarps * s;
      if (blk >= 20) break;
      int eR, fR;
      if (blk < 12) {
        const int pr = blk % 6, bi = pair_bi(pr);
        eR = (blk < 6 ? R_EK : R_EQ) + 16 * bi;
        fR = R_FO + 16 * pr;
      } else {
        const int b = (blk - 12) & 3;
        eR = (blk < 16 ? R_DK : R_DQ) + 16 * b;
        fR = R_FD + 16 * b;
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t ah[4], al[4], bh[4], bl[4];
        load_a(ah, IMG, LI, eR, 16 * ks, lane);
        load_a(al, IMG + R_IMG * LI, LI, eR, 16 * ks, lane);
        load_b_nk(bh, IMG, LI, 16 * ks, fR, lane);
        load_b_nk(bl, IMG + R_IMG * LI, LI, 16 * ks, fR, lane);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma_bf16(acc[s][nt], ah, bh[2 * nt], bh[2 * nt + 1]);
          mma_bf16(acc[s][nt], ah, bl[2 * nt], bl[2 * nt + 1]);
          mma_bf16(acc[s][nt], al, bh[2 * nt], bh[2 * nt + 1]);
        }
      }
    }
    __syncthreads();
  }
  // accumulators into A (fp32, beta_i applied, strict lower) and the M image (lower incl.)
  {
    const int g = lane >> 2, c = 2 * (lane & 3);
    unsigned char* mimg = sm + sM;
#pragma unroll
    for (int s = 0; s < kBlkPerWarp; ++s) {
      const int blk = warp + kWarps * s;
      if (blk >= 20) break;
      int r0, c0;
      bool diag;
      if (blk < 12) {
        const int pr = blk % 6, bi = pair_bi(pr), bj = pr - (bi * (bi - 1)) / 2;
        r0 = 16 * bi;
        c0 = 16 * bj;
        diag = false;
      } else {
        r0 = c0 = 16 * ((blk - 12) & 3);
        diag = true;
      }
      const bool is_m = (blk >= 6 && blk < 12) || blk >= 16;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = r0 + g + 8 * hh, j = c0 + 8 * nt + c;
          float v0 = acc[s][nt][2 * hh], v1 = acc[s][nt][2 * hh + 1];
          if (is_m) {
            if (diag) {
              v0 = j <= i ? v0 : 0.f;
              v1 = j + 1 <= i ? v1 : 0.f;
            }
            uint32_t hi, lo;
            split_pack2(v0, v1, hi, lo);
            const uint32_t off = sw_off(i, j >> 3) + (j & 7) * 2;
            *reinterpret_cast<uint32_t*>(mimg + off) = hi;
            *reinterpret_cast<uint32_t*>(mimg + 8192 + off) = lo;
          } else {
            if (diag) {
              v0 = j < i ? v0 : 0.f;
              v1 = j + 1 < i ? v1 : 0.f;
            }
            AT[i * LDT + j] = Bt[i] * v0;
            AT[i * LDT + j + 1] = Bt[i] * v1;
          }
        }
    }
  }
  __syncthreads();
  // diagonal blocks with a wide gate range: entry by entry, exp(G_i - G_j) <= 1
  if (flags[0]) {
    for (int pidx = warp; pidx < 4 * 136; pidx += kThr / 32) {
      const int b = pidx / 136;
      if (!((flags[0] >> b) & 1)) continue;
      int rem = pidx % 136, ii = 0;
      while (rem > ii) {
        rem -= ii + 1;
        ++ii;
      }
      const int i = 16 * b + ii, j = 16 * b + rem;
      float sk = 0.f, sq = 0.f;
      for (int d = lane; d < 128; d += 32) {
        const float e = __expf(G[i * GS + d] - G[j * GS + d]) * tile_elem(sm + sK, j, d);
        sk = fmaf(tile_elem(sm + sK, i, d), e, sk);
        sq = fmaf(tile_elem(sm + sQ, i, d), e, sq);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      if (lane == 0) {
        if (j < i) AT[i * LDT + j] = Bt[i] * sk * KR[i] * KR[j];
        const float m = sq * QR[i] * KR[j];
        __nv_bfloat16 mh, ml;
        split_bf16(m, mh, ml);
        const uint32_t off = sw_off(i, j >> 3) + (j & 7) * 2;
        *reinterpret_cast<__nv_bfloat16*>(sm + sM + off) = mh;
        *reinterpret_cast<__nv_bfloat16*>(sm + sM + 8192 + off) = ml;
      }
    }
    __syncthreads();
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_store(static_cast<unsigned char*>(p.M) + sl * 16384, sm + sM, 16384);
    bulk_commit();
  }
  tri_inverse_64_tc<kThr / 32>(AT, LDT, X, tid);  // ends synchronized

  // ---------------- T diag(beta) as a bf16 hi / lo pair (the hi part is the w operand)
  __nv_bfloat16* TH = IMG;
  __nv_bfloat16* TL = IMG + 64 * LTW;
  for (int idx = tid; idx < 64 * 8; idx += kThr) {
    const int i = idx >> 3, j0 = 8 * (idx & 7);
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2)
      split_pack2(AT[i * LDT + j0 + e] * Bt[j0 + e], AT[i * LDT + j0 + e + 1] * Bt[j0 + e + 1],
                  hi[e >> 1], lo[e >> 1]);
    *reinterpret_cast<uint4*>(TH + i * LTW + j0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(TL + i * LTW + j0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  __syncthreads();

  constexpr int kNW = 128 / (kWarps / 4);  // output columns per warp (4 warps per 16-row tile)
  constexpr int kNT = kNW / 8;              // n8 tiles per warp
  const int mt = warp & 3, nh = warp >> 2;  // rows 16 mt.., columns kNW nh .. kNW nh + kNW - 1
  const int g = lane >> 2, c = 2 * (lane & 3);
  // ---------------- w = T diag(beta) (exp(G) k): T is lower triangular (k steps <= mt)
  {
    float wa[kNT][4];
#pragma unroll
    for (int n = 0; n < kNT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) wa[n][e] = 0.f;
    for (int ks = 0; ks <= mt; ++ks) {
      uint32_t a[4];
      load_a(a, TH, LTW, 16 * mt, 16 * ks, lane);
#pragma unroll
      for (int n2 = 0; n2 < kNT / 2; ++n2) {
        uint32_t b[4];
        load_b_kn(b, KG, LKG, 16 * ks, kNW * nh + 16 * n2, lane);
        mma_bf16(wa[2 * n2], a, b[0], b[1]);
        mma_bf16(wa[2 * n2 + 1], a, b[2], b[3]);
      }
    }
    unsigned char* wimg = reinterpret_cast<unsigned char*>(IMG + 2 * 64 * LTW);
#pragma unroll
    for (int n = 0; n < kNT; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = 16 * mt + g + 8 * hh, col = kNW * nh + 8 * n + c;
        *reinterpret_cast<uint32_t*>(wimg + (col >> 6) * 8192 + sw_off(i, (col & 63) >> 3) +
                                     (col & 7) * 2) = pack_bf16(wa[n][2 * hh], wa[n][2 * hh + 1]);
      }
  }
  // ---------------- u = T diag(beta) v (T hi and lo against the exact v tile)
  {
    float ua[kNT][4];
#pragma unroll
    for (int n = 0; n < kNT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) ua[n][e] = 0.f;
    const uint32_t vbase = smem_addr(sm + sV);
    for (int ks = 0; ks <= mt; ++ks) {
      uint32_t ah[4], al[4];
      load_a(ah, TH, LTW, 16 * mt, 16 * ks, lane);
      load_a(al, TL, LTW, 16 * mt, 16 * ks, lane);
#pragma unroll
      for (int n2 = 0; n2 < kNT / 2; ++n2) {
        // B = v tile [token][value column], swizzled: rows 16 ks.., columns 16-wide group
        const int m = lane >> 3;
        const int row = 16 * ks + (lane & 7) + (m & 1) * 8;
        const int col = kNW * nh + 16 * n2 + (m >> 1) * 8;
        uint32_t b[4];
        ldsm_x4_t_addr(b, vbase + (col >> 6) * 8192 + sw_off(row, (col & 63) >> 3));
        mma_bf16(ua[2 * n2], ah, b[0], b[1]);
        mma_bf16(ua[2 * n2 + 1], ah, b[2], b[3]);
        mma_bf16(ua[2 * n2], al, b[0], b[1]);
        mma_bf16(ua[2 * n2 + 1], al, b[2], b[3]);
      }
    }
    unsigned char* ust = sm + sG;  // the gates are consumed
#pragma unroll
    for (int n = 0; n < kNT; ++n)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = 16 * mt + g + 8 * hh, col = kNW * nh + 8 * n + c;
        *reinterpret_cast<float2*>(ust + (col >> 5) * 8192 + u_offset(i, col & 31)) =
            make_float2(ua[n][2 * hh], ua[n][2 * hh + 1]);
      }
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_store(static_cast<unsigned char*>(p.w) + sl * 16384,
               reinterpret_cast<unsigned char*>(IMG + 2 * 64 * LTW), 16384);
    bulk_store(reinterpret_cast<unsigned char*>(p.u + sl * 64 * 128), sm + sG, 32768);
    bulk_commit();
    bulk_wait<0>();  // every image written before the CTA's shared memory is released
    if (flags[1]) {
      mbar_wait(bar, 0, kWaitIters);  // the tile copies, bounded
      set_status(p.status, GDN_DEV_TIMEOUT);
    }
  }
}

}  // namespace

bool launch_kda_intra(const Params& p, cudaStream_t s) {
  CUtensorMap tmk, tmq, tmv;
  const int rows = p.T > 0 ? p.T : 1;
  if (!encode_rows_tmap(&tmk, p.k, rows, p.H, p.D) ||
      !encode_rows_tmap(&tmq, p.q, rows, p.H, p.D) ||
      !encode_rows_tmap(&tmv, p.v, rows, p.Hv, p.D))
    return false;
  ensure_smem_limit((const void*)kda_intra_kernel, (int)kSmemBytes);
  return launch_pdl(kda_intra_kernel, dim3(p.nt_max, p.Hv), dim3(kThr), kSmemBytes, s, p, tmk,
                    tmq, tmv) == cudaSuccess;
}

}  // namespace gdn
