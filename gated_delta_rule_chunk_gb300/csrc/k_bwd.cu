// Backward pass of the chunked gated delta rule (scalar gates), fp32 SIMT.
//
// The stage names follow the backward kernels listed in the FLA graph-capture
// RFC ("What needs to change", GDN bwd: the state-gradient scan, the local dv
// and dq/dk/dw/dg gradients and the WY-representation gradient). Per sequence
// and value head, with the chunk quantities of the forward (chunk-start state
// S, T = (I + A)^-1, w, u, v_new, M = Gamma * (Q K^T) and the decayed images
// Qt = exp(G) Q, Kt = exp(G_L - G) K), the gradient of
//   v_new = u - w S,   o = scale (Qt S + M v_new),   S' = exp(G_L) S + Kt^T v_new
// runs a reverse scan over the chunks (dS holds the gradient of the next
// chunk-start state):
//   dv_new = Kt dS + scale M^T dO,   dS <- exp(G_L) dS + scale Qt^T dO - w^T dv_new
// and then, per chunk, with dw = -dv_new S^T, Z = dv_new (beta V)^T + dw (beta exp(G) K)^T
// and dA = -(T^T Z T^T) on the strict lower triangle:
//   dv   = beta * (T^T dv_new)
//   dq   = scale exp(G) * (dO S^T) + (dP * Gamma) K,           dP = scale dO v_new^T (j <= i)
//   dk   = (dP * Gamma)^T Q + exp(G_L - G) * (v_new dS^T) + beta exp(G) * (T^T dw)
//          + (dAt + dAt^T) K,                                  dAt = dA * beta_i Gamma_ij
//   dbeta_i = (T^T dv_new)_i . v_i + exp(G_i) (T^T dw)_i . k_i + sum_j dA_ij Gamma_ij k_i . k_j
//   dG   from every exp(G) factor (rows and columns of Gamma, exp(G), exp(G_L));
//   dg   = reverse in-chunk cumsum of dG,  dS_0 = the scan's last dS.
// Each step is the derivative of one forward equation; together they equal the
// token-by-token adjoint of the recurrence.
#include <type_traits>

#include "gdn_common.cuh"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThr = 256;

template <int D>
constexpr int bv_of() { return D == 128 ? 32 : 16; }

__device__ __forceinline__ float ld_dout(const BwdParams& p, size_t idx) {
  return p.dout_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.dout)[idx])
                     : reinterpret_cast<const float*>(p.dout)[idx];
}

// ---------------------------------------------------------------- reverse scan
template <int D>
constexpr size_t scan_floats() {
  constexpr int BV = bv_of<D>(), SLD = BV + 4, LQ = D + 4;
  return (size_t)D * SLD + D * 68 + 64 * 68 + 2 * 64 * LQ + 2 * 64 * BV + D;
}

// fp32 SIMT reverse scan (fp32 inputs): the forward quantities are the general path's
// fp32 tiles (Kt = exp(G_L - G) k, Qt^T = (exp(G) q)^T, w^T, M^T, exp(G_L) per key row).
template <int D>
__global__ void __launch_bounds__(kThr) bwd_scan_kernel(BwdParams p) {
  constexpr int BV = bv_of<D>(), SLD = BV + 4, LQ = D + 4, RN = BV / 16;
  extern __shared__ __align__(16) float sm[];
  float* dS = sm;                  // [D][SLD] gradient of the next chunk-start state
  float* KtT = dS + D * SLD;       // [D][68]  Kt^T
  float* Mr = KtT + D * 68;        // [64][68] M (row-major)
  float* Qr = Mr + 64 * 68;        // [64][LQ] Qt (token-major)
  float* Wr = Qr + 64 * LQ;        // [64][LQ] w (token-major)
  float* dO = Wr + 64 * LQ;        // [64][BV]
  float* dV = dO + 64 * BV;        // [64][BV] dv_new
  float* gm = dV + 64 * BV;        // [D]

  const int tid = threadIdx.x;
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * BV;
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }
  const size_t sbase = ((size_t)n * p.Hv + hv) * D * D;
  for (int idx = tid; idx < D * BV; idx += kThr) {
    const int d = idx / BV, j = idx % BV;
    dS[d * SLD + j] = p.dfin ? p.dfin[sbase + (size_t)(c0 + j) * D + d] : 0.f;
  }
  for (int c = nch - 1; c >= 0; --c) {
    const size_t sl = (size_t)(sv.first_slot + c) * p.Hv + hv;
    const int t0 = sv.start + kChunk * c;
    const int L = min(kChunk, sv.len - kChunk * c);
    if (tid == 0 && c > 0) {  // the next (earlier) chunk's tiles into L2 while this one runs
      const size_t pl = sl - p.Hv;
      bulk_prefetch_l2(p.kt + pl * 64 * D, 64 * D * 4);
      bulk_prefetch_l2(p.qt + pl * 64 * D, 64 * D * 4);
      bulk_prefetch_l2(p.wT + pl * 64 * D, 64 * D * 4);
      bulk_prefetch_l2(p.MT + pl * 4096, 4096 * 4);
    }
    const float* kt = p.kt + sl * 64 * D;
    const float* qt = p.qt + sl * 64 * D;
    const float* wt = p.wT + sl * 64 * D;
    const float* mt = p.MT + sl * 4096;
    // Kt rows (lanes along features) into Kt^T; Qt^T and w^T rows (lanes along tokens)
    // into token-major tiles; M^T[i][t] = M[t][i] into M
    staged_copy<8>(64 * D, tid, kThr, [&](int i) { return kt[i]; },
                   [&](int i, float x) { KtT[(i % D) * 68 + i / D] = x; });
    staged_copy<8>(64 * D, tid, kThr, [&](int i) { return qt[i]; },
                   [&](int i, float x) { Qr[(i % 64) * LQ + i / 64] = x; });
    staged_copy<8>(64 * D, tid, kThr, [&](int i) { return wt[i]; },
                   [&](int i, float x) { Wr[(i % 64) * LQ + i / 64] = x; });
    staged_copy<8>(64 * 64, tid, kThr, [&](int i) { return mt[i]; },
                   [&](int i, float x) { Mr[(i & 63) * 68 + (i >> 6)] = x; });
    staged_copy<8>(64 * BV, tid, kThr,
                   [&](int i) {
                     return i / BV < L ? ld_dout(p, ((size_t)(t0 + i / BV) * p.Hv + hv) * D + c0 + i % BV)
                                       : 0.f;
                   },
                   [&](int i, float x) { dO[i] = x; });
    for (int d = tid; d < D; d += kThr) gm[d] = p.gam[sl * D + d];
    __syncthreads();
    {  // the incoming gradient is this chunk's dS_next; keep it for the chunk kernels
      float* dh = p.dhs + sl * D * D;
      for (int idx = tid; idx < D * BV; idx += kThr) {
        const int j = idx / D, d = idx % D;
        dh[(size_t)(c0 + j) * D + d] = dS[d * SLD + j];
      }
    }
    {  // dv_new = Kt dS + scale M^T dO (M[t][i] is zero for t < i)
      const int i0 = (tid >> 4) * 4, n0 = (tid & 15) * RN;
      float a[4][RN], b[4][RN];
      zero(a);
      zero(b);
      fma_tile<4, RN>(a, KtT, 68, dS, SLD, i0, n0, 0, D);
      fma_tile<4, RN>(b, Mr, 68, dO, BV, i0, n0, i0, 64);
      float* gout = p.dvn + sl * 64 * D + c0;
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < RN; ++cc) {
          const float x = fmaf(p.scale, b[r][cc], a[r][cc]);
          dV[(i0 + r) * BV + n0 + cc] = x;
          gout[(size_t)(i0 + r) * D + n0 + cc] = x;
        }
    }
    __syncthreads();
    // dS <- exp(G_L) dS + scale Qt^T dO - w^T dv_new (each entry owned by one thread)
    for (int t = tid; t < (D / 4) * 16; t += kThr) {
      const int d0 = (t >> 4) * 4, n0 = (t & 15) * RN;
      float a[4][RN], b[4][RN];
      zero(a);
      zero(b);
      fma_tile<4, RN>(a, Qr, LQ, dO, BV, d0, n0, 0, 64);
      fma_tile<4, RN>(b, Wr, LQ, dV, BV, d0, n0, 0, 64);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int cc = 0; cc < RN; ++cc) {
          float& s = dS[(d0 + r) * SLD + n0 + cc];
          s = fmaf(gm[d0 + r], s, fmaf(p.scale, a[r][cc], -b[r][cc]));
        }
    }
    __syncthreads();
  }
  __syncthreads();  // an empty sequence skips the loop: dS was written by other threads
  if (p.dh0)
    for (int idx = tid; idx < D * BV; idx += kThr) {
      const int j = idx / D, d = idx % D;
      p.dh0[sbase + (size_t)(c0 + j) * D + d] = dS[d * SLD + j];
    }
}

// ---------------------------------------------------------------- contractions with S, dS
// dos = dO S^T, dw = -dv_new S^T, ys = v_new dS_next^T (contractions over dv) and
// sdot = <S, dS_next>, per (chunk slot, value head), on warp-level tensor-core MMAs.
// With the state [dv][dk] row-major, each product is A [64 tokens][dv] times B = the
// state [dv][dk]: a dense 64 x D x D contraction. Both fp32 operands are split into a
// bf16 hi/lo pair in shared memory (x = hi + lo, about 16 significant bits) and the
// product takes the three terms hi*hi + hi*lo + lo*hi (a bf16 dO is exact: two terms).
template <int D>
constexpr size_t state_mma_bytes() {
  return (size_t)2 * (D + 64) * (D + 8) * sizeof(__nv_bfloat16) + 64;
}

__device__ __forceinline__ float4 ld_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Four consecutive dO elements (bf16 or fp32) as floats.
__device__ __forceinline__ float4 ld_dout4(const BwdParams& p, size_t idx) {
  if (p.dout_bf16) {
    const uint2 r = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.dout) + idx);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return ld_f4(reinterpret_cast<const float*>(p.dout) + idx);
}

// bf16 hi/lo copies of `rows` fp32 rows of D columns into row-major tiles with row
// stride D + 8 (16-byte padding: the 8 row addresses of an ldmatrix hit distinct bank
// groups). get(r, c4) returns columns 4 c4 .. 4 c4 + 3 of row r; eight loads in flight
// per thread.
template <int D, typename Get>
__device__ __forceinline__ void split_rows(__nv_bfloat16* hi, __nv_bfloat16* lo, int rows, int tid,
                                           Get get) {
  constexpr int RS = D + 8, Q = D / 4;
  const int n = rows * Q;
  for (int base = tid; base < n; base += 8 * kThr) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int idx = base + u * kThr;
      v[u] = idx < n ? get(idx / Q, idx % Q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int idx = base + u * kThr;
      if (idx < n) {
        const int off = (idx / Q) * RS + 4 * (idx % Q);
        uint2 h, l;
        split_pack2(v[u].x, v[u].y, h.x, l.x);
        split_pack2(v[u].z, v[u].w, h.y, l.y);
        *reinterpret_cast<uint2*>(hi + off) = h;
        *reinterpret_cast<uint2*>(lo + off) = l;
      }
    }
  }
}

// out[64][D] = sign * A B, A = Ah + Al ([64][D + 8]), B = Bh + Bl ([D][D + 8], row-major
// [k][n]); warp w owns rows 16 (w % 4).. and columns (w / 4) D/2 ..; the lo*lo term is
// dropped, and so is every Al term when A is exact in bf16.
template <int D>
__device__ __forceinline__ void state_product(const __nv_bfloat16* Ah, const __nv_bfloat16* Al,
                                              bool a_exact, const __nv_bfloat16* Bh,
                                              const __nv_bfloat16* Bl, float sign, float* out,
                                              int warp, int lane) {
  constexpr int RS = D + 8, NW = D / 2, NT = NW / 8;
  const int mt = warp & 3, n0 = (warp >> 2) * NW;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll 2
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t ah[4], al[4];
    load_a(ah, Ah, RS, 16 * mt, 16 * ks, lane);
    if (!a_exact) load_a(al, Al, RS, 16 * mt, 16 * ks, lane);
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t bh[4], bl[4];
      load_b_kn(bh, Bh, RS, 16 * ks, n0 + 16 * np, lane);
      load_b_kn(bl, Bl, RS, 16 * ks, n0 + 16 * np, lane);
      mma_bf16(acc[2 * np], ah, bh[0], bh[1]);
      mma_bf16(acc[2 * np + 1], ah, bh[2], bh[3]);
      mma_bf16(acc[2 * np], ah, bl[0], bl[1]);
      mma_bf16(acc[2 * np + 1], ah, bl[2], bl[3]);
      if (!a_exact) {
        mma_bf16(acc[2 * np], al, bh[0], bh[1]);
        mma_bf16(acc[2 * np + 1], al, bh[2], bh[3]);
      }
    }
  }
  const int g = lane >> 2, c2 = 2 * (lane & 3), r0 = 16 * mt + g;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = n0 + 8 * nt + c2;
    *reinterpret_cast<float2*>(out + (size_t)r0 * D + col) =
        make_float2(sign * acc[nt][0], sign * acc[nt][1]);
    *reinterpret_cast<float2*>(out + (size_t)(r0 + 8) * D + col) =
        make_float2(sign * acc[nt][2], sign * acc[nt][3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThr) bwd_state_kernel(BwdParams p) {
  constexpr int RS = D + 8;
  extern __shared__ __align__(16) unsigned char smb[];
  __nv_bfloat16* Bh = reinterpret_cast<__nv_bfloat16*>(smb);  // [D][RS] the state (then dS_next)
  __nv_bfloat16* Bl = Bh + D * RS;
  __nv_bfloat16* Ah = Bl + D * RS;                             // [64][RS] dO, dv_new, v_new
  __nv_bfloat16* Al = Ah + 64 * RS;
  float* red = reinterpret_cast<float*>(Al + 64 * RS);         // [8] warp partials

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, hv = blockIdx.y;
  int t0, L, wslot;
  if (!resolve_slot(p, blockIdx.x, t0, L, wslot)) return;
  const size_t sl = (size_t)wslot * p.Hv + hv;
  const float* hs = p.hs + sl * D * D;
  const float* dhs = p.dhs + sl * D * D;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);

  split_rows<D>(Bh, Bl, D, tid, [&](int r, int c4) { return ld_f4(hs + (size_t)r * D + 4 * c4); });
  split_rows<D>(Ah, Al, 64, tid, [&](int r, int c4) {  // rows past the sequence end: zero
    return r < L ? ld_dout4(p, ((size_t)(t0 + r) * p.Hv + hv) * D + 4 * c4) : z4;
  });
  __syncthreads();
  state_product<D>(Ah, Al, p.dout_bf16 != 0, Bh, Bl, 1.f, p.dos + sl * 64 * D, warp, lane);
  __syncthreads();
  split_rows<D>(Ah, Al, 64, tid,
                [&](int r, int c4) { return ld_f4(p.dvn + sl * 64 * D + (size_t)r * D + 4 * c4); });
  __syncthreads();
  state_product<D>(Ah, Al, false, Bh, Bl, -1.f, p.dw + sl * 64 * D, warp, lane);
  __syncthreads();
  float sd = 0.f;
  split_rows<D>(Bh, Bl, D, tid, [&](int r, int c4) {
    const float4 a = ld_f4(dhs + (size_t)r * D + 4 * c4), b = ld_f4(hs + (size_t)r * D + 4 * c4);
    sd += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
    return a;
  });
  split_rows<D>(Ah, Al, 64, tid,
                [&](int r, int c4) { return ld_f4(p.vn + sl * 64 * D + (size_t)r * D + 4 * c4); });
  __syncthreads();
  state_product<D>(Ah, Al, false, Bh, Bl, 1.f, p.ys + sl * 64 * D, warp, lane);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, o);
  if (lane == 0) red[warp] = sd;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kThr / 32; ++w) t += red[w];
    p.sdot[sl] = t;
  }
}

// ---------------------------------------------------------------- per-chunk gradients
constexpr int kLd = 72;    // row stride (8 mod 32) of the 64 x 64 matrices and the 64-wide blocks

constexpr size_t chunk_floats() {
  return (size_t)11 * 64 * kLd + 16 * kLd + 8 * 64 + 4 * 64 * 8;
}
// On a GB300 a launch of this kernel with 219,392 B of dynamic shared memory ran and one with
// 231,936 B was refused (the per-block total also holds about 4 KB beyond the dynamic size).
static_assert(chunk_floats() * sizeof(float) <= 219392, "per-chunk kernel shared memory");

// Threads of the per-chunk kernel: 16 warps, each owning a 16 x 16 tile of every 64-wide
// result, so that four warps per SM sub-partition cover the latency of the shared-memory
// operand loads and the MMAs.
constexpr int kThrC = 512;
constexpr int kBlkU = 64 * 32 / kThrC;

// A [64 x 32] block of a token-major source (tokens x 32 features) held in registers,
// kBlkU elements per thread, so that the next block's loads are in flight while the current
// one is used. Warp w, lane l holds token 4 w + l / 8 and features l % 8 + 8 u: each load
// instruction reads four 8-feature runs, and the 32 lanes of a token-major store fall in
// 32 distinct banks (8 t + f, row stride 8 mod 32; a feature-major store is two-way).
struct Blk {
  float r[kBlkU];
};
__device__ __forceinline__ int blk_token(int tid) { return 4 * (tid >> 5) + ((tid & 31) >> 3); }
__device__ __forceinline__ int blk_feature(int tid, int u) { return (tid & 7) + 8 * u; }
// get(i, f) returns token i, feature f; tokens at or past L read as zero.
template <typename Get>
__device__ __forceinline__ void load_blk(Blk& b, int L, int tid, Get get) {
  const int t = blk_token(tid);
#pragma unroll
  for (int u = 0; u < kBlkU; ++u) b.r[u] = t < L ? get(t, blk_feature(tid, u)) : 0.f;
}
// ... stored feature-major (32 rows of stride kLd) or token-major (64 rows of stride ld)
__device__ __forceinline__ void store_fm(float* dst, const Blk& b, int tid) {
  const int t = blk_token(tid);
#pragma unroll
  for (int u = 0; u < kBlkU; ++u) dst[blk_feature(tid, u) * kLd + t] = b.r[u];
}
__device__ __forceinline__ void store_tm(float* dst, const Blk& b, int tid, int ld) {
  const int t = blk_token(tid);
#pragma unroll
  for (int u = 0; u < kBlkU; ++u) dst[t * ld + blk_feature(tid, u)] = b.r[u];
}
// A [64 x 32] block held as one 4-feature vector per thread: warp w, lane l holds token
// 4 w + l / 8 and features 4 (l % 8) .. 4 (l % 8) + 3 (one vector load); for blocks stored
// token-major only, where each eight lanes write one contiguous 128-byte row segment.
struct Blk4 {
  float4 v;
};
template <typename TIn>
__device__ __forceinline__ float4 ld_in4(const void* base, size_t idx) {
  if constexpr (std::is_same<TIn, __nv_bfloat16>::value) {
    const uint2 r = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + idx);
  }
}
// get(i, f) returns features f..f+3 of token i; tokens at or past L read as zero.
template <typename Get>
__device__ __forceinline__ void load_blk4(Blk4& b, int L, int tid, Get get) {
  const int t = blk_token(tid);
  b.v = t < L ? get(t, 4 * (tid & 7)) : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ void store_tm4(float* dst, const Blk4& b, int tid, int ld) {
  *reinterpret_cast<float4*>(dst + blk_token(tid) * ld + 4 * (tid & 7)) = b.v;
}

// Element (i, j) of a 64 x 64 pass over index idx: each warp covers an 8 x 4 patch, so that
// both [i][j] and [j][i] accesses (row stride kLd) are at most two-way bank conflicts.
__device__ __forceinline__ void patch_ij(int idx, int& i, int& j) {
  const int blk = idx >> 5, l = idx & 31;
  i = 8 * (blk & 7) + (l & 7);
  j = 4 * (blk >> 3) + (l >> 3);
}

// acc[nt] += sum_{k0 <= k < k1} A[m0 + r][k] B[n0 + 8 nt + c'][k] over a 16 x 8 NT warp tile:
// both operands fp32 in shared memory with k contiguous (row strides lda, ldb = 8 mod 32, so
// that the 64-bit fragment loads of each half-warp fall in distinct banks), split into bf16
// hi + lo per fragment, three warp MMAs per step of 16 (hi*hi, hi*lo, lo*hi).
// Accumulator element e of tile nt: row m0 + g + 8 (e >> 1), column n0 + 8 nt + c + (e & 1)
// (g = lane / 4, c = 2 (lane % 4)).
// AX / BX: the A / B operand holds values exact in bf16 (the bf16 inputs k, q, v), whose
// lo halves are zero: the terms with them are skipped (two MMAs per step, or one when both
// are exact).
template <int NT, bool AX = false, bool BX = false>
__device__ __forceinline__ void mma_rowk(float (&acc)[NT][4], const float* A, int lda,
                                         const float* B, int ldb, int m0, int n0, int k0,
                                         int k1, int lane) {
  const int g = lane >> 2, c = 2 * (lane & 3);
#pragma unroll 2
  for (int k = k0; k < k1; k += 16) {
    const float* ap = A + (m0 + g) * lda + k + c;
    const float2 a0 = *reinterpret_cast<const float2*>(ap);
    const float2 a1 = *reinterpret_cast<const float2*>(ap + 8 * lda);
    const float2 a2 = *reinterpret_cast<const float2*>(ap + 8);
    const float2 a3 = *reinterpret_cast<const float2*>(ap + 8 * lda + 8);
    uint32_t ah[4], al[4];
    split_pack2(a0.x, a0.y, ah[0], al[0]);
    split_pack2(a1.x, a1.y, ah[1], al[1]);
    split_pack2(a2.x, a2.y, ah[2], al[2]);
    split_pack2(a3.x, a3.y, ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float* bp = B + (n0 + 8 * nt + g) * ldb + k + c;
      const float2 b0 = *reinterpret_cast<const float2*>(bp);
      const float2 b1 = *reinterpret_cast<const float2*>(bp + 8);
      uint32_t bh[2], bl[2];
      split_pack2(b0.x, b0.y, bh[0], bl[0]);
      split_pack2(b1.x, b1.y, bh[1], bl[1]);
      mma_bf16(acc[nt], ah, bh[0], bh[1]);
      if (!BX) mma_bf16(acc[nt], ah, bl[0], bl[1]);
      if (!AX) mma_bf16(acc[nt], al, bh[0], bh[1]);
    }
  }
}

// Sum of x over the four lanes that share a row of an MMA accumulator.
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Per (chunk slot, value head). Every product is a warp-MMA tile product of fp32 operands in
// shared memory stored with the contraction index contiguous (mma_rowk): token-major blocks
// for the sums over features, feature-major blocks and transposed matrices for the sums over
// tokens. Warp w owns rows 16 mt.. of each result, mt = w / 4, and
// columns 16 nh.. (of 64 tokens or of a pass of 64 features), nh = (w - mt) % 4:
// the warps of one SM sub-partition (w % 4) then hold every row block and every column
// block once, so that the products that skip the zero triangle of T, of the gate-masked
// matrices or of the lower-triangular results load the sub-partitions evenly.
template <typename TIn, int D>
__global__ void __launch_bounds__(kThrC) bwd_chunk_kernel(BwdParams p) {
  constexpr bool kX = std::is_same<TIn, __nv_bfloat16>::value;  // k, q, v exact in bf16
  extern __shared__ __align__(16) float sm[];
  float* Tm = sm;                  // T = (I + A)^-1, row-major
  float* Tt = Tm + 64 * kLd;       // T^T
  float* GK = Tt + 64 * kLd;       // Gamma * K K^T (strict lower); later dAt + dAt^T
  float* Mm = GK + 64 * kLd;       // Gamma * Q K^T (lower incl.)
  float* dP = Mm + 64 * kLd;       // scale dO v_new^T (lower incl.); later dP * Gamma
  float* Zm = dP + 64 * kLd;       // Z^T; later dA
  float* Tp = Zm + 64 * kLd;       // scratch: (Z^T T)^T; later (dP * Gamma)^T
  float* R0 = Tp;                  // before that, the feature-major block (dv_new, then dw)
  float* Xs = Tp + 64 * kLd;       // [16][kLd] scratch of the inverse
  float* B0 = Xs + 16 * kLd;       // [64][kLd] token-major blocks of 64 features
  float* B1 = B0 + 64 * kLd;
  float* B2 = B1 + 64 * kLd;
  float* B3 = B2 + 64 * kLd;
  float* G = B3 + 64 * kLd;        // [64] in-chunk cumulative gate
  float* eG = G + 64;              // exp(G)
  float* eL = eG + 64;             // exp(G_L - G)
  float* bt = eL + 64;             // beta
  float* dGv = bt + 64;            // dG
  float* dBv = dGv + 64;           // dbeta
  float* rsk = dBv + 64;           // (T^T dw)_i . k_i
  float* wsum = rsk + 64;          // W_i = exp(G_L - G_i) k_i . (v_new dS^T)_i
  float* pv = wsum + 64;           // [64][8] partial row dots (T^T dv_new) . v (slots 0-3)
  float* pk = pv + 64 * 8;         // [64][8] partial row dots (T^T dw) . k
  float* pq = pk + 64 * 8;         // [64][8] partial row dots q . (dO S^T)
  float* pw = pq + 64 * 8;         // [64][8] partial row dots k . (v_new dS^T)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, hv = blockIdx.y, h = hv / p.HG;
  const int g = lane >> 2, c = 2 * (lane & 3), mt = warp >> 2, nh = (warp - mt) & 3;
  const int r0 = 16 * mt + g;  // this thread's accumulator rows: r0 and r0 + 8
  int t0, L, wslot;
  if (!resolve_slot(p, blockIdx.x, t0, L, wslot)) return;
  const bool lower = nh <= mt;  // this warp's 64-wide tile meets the lower triangle
  const size_t sl = (size_t)wslot * p.Hv + hv;
  auto kin = [&](int i, int f) { return ld_in<TIn>(p.k, ((size_t)(t0 + i) * p.H + h) * D + f); };
  auto qin = [&](int i, int f) { return ld_in<TIn>(p.q, ((size_t)(t0 + i) * p.H + h) * D + f); };
  // element (row, column) of accumulator entry (nt, e) of a 64-wide result
  auto col64 = [&](int nt, int e) { return 16 * nh + 8 * nt + c + (e & 1); };
  auto row = [&](int e) { return r0 + 8 * (e >> 1); };

  const size_t krow = (size_t)p.H * D, vrow = (size_t)p.Hv * D;  // token strides
  const size_t kbase = ((size_t)t0 * p.H + h) * D, vbase = ((size_t)t0 * p.Hv + hv) * D;
  // k and q of features f0..f0+63 (two blocks each) for the first stage, token-major only
  // (vector loads); the first ones are in flight during the gate scan
  Blk4 k4[2], q4[2];
  auto load_kq4 = [&](int f0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      load_blk4(k4[hh], L, tid, [&](int i, int f) { return ld_in4<TIn>(p.k, kbase + i * krow + f0 + 32 * hh + f); });
      load_blk4(q4[hh], L, tid, [&](int i, int f) { return ld_in4<TIn>(p.q, kbase + i * krow + f0 + 32 * hh + f); });
    }
  };
  load_kq4(0);
  if (warp == 0) {  // G: inclusive in-chunk cumsum of g (two rows per lane, shuffle scan)
    const bool ok0 = lane < L, ok1 = lane + 32 < L;
    float g0 = ok0 ? p.g[(size_t)(t0 + lane) * p.Hv + hv] : 0.f;
    float g1 = ok1 ? p.g[(size_t)(t0 + lane + 32) * p.Hv + hv] : 0.f;
    bt[lane] = ok0 ? p.beta[(size_t)(t0 + lane) * p.Hv + hv] : 0.f;
    bt[lane + 32] = ok1 ? p.beta[(size_t)(t0 + lane + 32) * p.Hv + hv] : 0.f;
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
  }
  __syncthreads();
  if (tid < 64) {
    eG[tid] = expf(G[tid]);
    eL[tid] = expf(G[63] - G[tid]);
  }
  // ---------------- K K^T and Q K^T (64 features a pass)
  {
    float akk[2][4], aqk[2][4];
    zero(akk);
    zero(aqk);
    for (int fp = 0; fp < D / 64; ++fp) {
      __syncthreads();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        store_tm4(B0 + 32 * hh, k4[hh], tid, kLd);
        store_tm4(B1 + 32 * hh, q4[hh], tid, kLd);
      }
      __syncthreads();
      if (fp + 1 < D / 64) load_kq4(64 * (fp + 1));  // in flight under this pass's products
      if (lower) {  // both are masked to the lower triangle
        mma_rowk<2, kX, kX>(akk, B0, kLd, B0, kLd, 16 * mt, 16 * nh, 0, 64, lane);
        mma_rowk<2, kX, kX>(aqk, B1, kLd, B0, kLd, 16 * mt, 16 * nh, 0, 64, lane);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = row(e), j = col64(nt, e);
        const float gam = j <= i ? expf(G[i] - G[j]) : 0.f;
        GK[i * kLd + j] = j < i ? gam * akk[nt][e] : 0.f;
        Mm[i * kLd + j] = gam * aqk[nt][e];
        Tm[i * kLd + j] = j < i ? bt[i] * gam * akk[nt][e] : 0.f;  // A
      }
  }
  // value-feature blocks (dO, v_new, dv_new, v) of features f0..f0+63, two blocks each;
  // dv_new is also stored feature-major (scalar element map), the others by vectors
  Blk4 bdo[2], bvn[2], bv[2];
  Blk bdv[2];
  auto load_value_blocks = [&](int f0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int fh = f0 + 32 * hh;
      load_blk4(bdo[hh], L, tid, [&](int i, int f) { return ld_dout4(p, vbase + i * vrow + fh + f); });
      load_blk4(bvn[hh], 64, tid, [&](int i, int f) { return ld_f4(p.vn + sl * 64 * D + (size_t)i * D + fh + f); });
      load_blk(bdv[hh], 64, tid, [&](int i, int f) { return p.dvn[sl * 64 * D + (size_t)i * D + fh + f]; });
      load_blk4(bv[hh], L, tid, [&](int i, int f) { return ld_in4<TIn>(p.v, vbase + i * vrow + fh + f); });
    }
  };
  // key-feature blocks (dw, k) of features f0..f0+63: dw (also stored feature-major), and k
  // by vectors into k4
  Blk bdw[2];
  auto load_key_blocks = [&](int f0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int fh = f0 + 32 * hh;
      load_blk(bdw[hh], 64, tid, [&](int i, int f) { return p.dw[sl * 64 * D + (size_t)i * D + fh + f]; });
      load_blk4(k4[hh], L, tid, [&](int i, int f) { return ld_in4<TIn>(p.k, kbase + i * krow + fh + f); });
    }
  };
  load_value_blocks(0);  // in flight during the inverse
  __syncthreads();
  tri_inverse_64_tc<kThrC / 32>(Tm, kLd, Xs, tid);  // Tm = T, ends synchronized
  for (int idx = tid; idx < 64 * 64; idx += kThrC) {
    int i, j;
    patch_ij(idx, i, j);
    Tt[j * kLd + i] = Tm[i * kLd + j];
  }
  // ---------------- value features: dP, Z1, T^T dv_new (dv and the dbeta part)
  float az[2][4];
  zero(az);
  {
    float adp[2][4];
    zero(adp);
    float rv[2] = {0.f, 0.f};
    for (int fp = 0; fp < D / 64; ++fp) {
      __syncthreads();
      const int f0 = fp * 64;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        store_tm4(B0 + 32 * h, bdo[h], tid, kLd);
        store_tm4(B1 + 32 * h, bvn[h], tid, kLd);
        store_tm(B2 + 32 * h, bdv[h], tid, kLd);
        store_tm4(B3 + 32 * h, bv[h], tid, kLd);
        store_fm(R0 + 32 * h * kLd, bdv[h], tid);
      }
      __syncthreads();
      if (fp + 1 < D / 64)
        load_value_blocks(f0 + 64);
      else
        load_key_blocks(0);
      if (lower) mma_rowk<2>(adp, B0, kLd, B1, kLd, 16 * mt, 16 * nh, 0, 64, lane);
      mma_rowk<2, false, kX>(az, B2, kLd, B3, kLd, 16 * mt, 16 * nh, 0, 64, lane);
      float tu[2][4];  // (T^T dv_new)[j][n]: T[i][j] = 0 for i < j
      zero(tu);
      mma_rowk<2>(tu, Tt, kLd, R0, kLd, 16 * mt, 16 * nh, 16 * mt, 64, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // entries 2 hh, 2 hh + 1: adjacent columns
          const int j = r0 + 8 * hh, n = col64(nt, 0);
          const float t0v = tu[nt][2 * hh], t1v = tu[nt][2 * hh + 1];
          rv[hh] = fmaf(t0v, B3[j * kLd + n], rv[hh]);
          rv[hh] = fmaf(t1v, B3[j * kLd + n + 1], rv[hh]);
          if (j < L)
            *reinterpret_cast<float2*>(p.dv + ((size_t)(t0 + j) * p.Hv + hv) * D + f0 + n) =
                make_float2(bt[j] * t0v, bt[j] * t1v);
        }
    }
    rv[0] = quad_sum(rv[0]);
    rv[1] = quad_sum(rv[1]);
    if ((lane & 3) == 0) {
      pv[r0 * 8 + nh] = rv[0];
      pv[(r0 + 8) * 8 + nh] = rv[1];
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = row(e), j = col64(nt, e);
        dP[i * kLd + j] = j <= i ? p.scale * adp[nt][e] : 0.f;
      }
  }
  // ---------------- key features: Z2, T^T dw (the dk and dbeta / dG parts)
  {
    float rk[2] = {0.f, 0.f};
    for (int fp = 0; fp < D / 64; ++fp) {
      __syncthreads();
      const int f0 = fp * 64;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        store_tm(B0 + 32 * h, bdw[h], tid, kLd);
        store_tm4(B1 + 32 * h, k4[h], tid, kLd);
        store_fm(R0 + 32 * h * kLd, bdw[h], tid);
      }
      __syncthreads();
      if (fp + 1 < D / 64) load_key_blocks(f0 + 64);
      {  // Z2[i][j] = sum_d dw[i][d] exp(G_j) k[j][d]: scale column j after the sum
        float z2[2][4];
        zero(z2);
        mma_rowk<2, false, kX>(z2, B0, kLd, B1, kLd, 16 * mt, 16 * nh, 0, 64, lane);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) az[nt][e] = fmaf(eG[col64(nt, e)], z2[nt][e], az[nt][e]);
      }
      float tw[2][4];
      zero(tw);
      mma_rowk<2>(tw, Tt, kLd, R0, kLd, 16 * mt, 16 * nh, 16 * mt, 64, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // entries 2 hh, 2 hh + 1: adjacent columns
          const int j = r0 + 8 * hh, n = col64(nt, 0);
          const float t0v = tw[nt][2 * hh], t1v = tw[nt][2 * hh + 1];
          rk[hh] = fmaf(t0v, B1[j * kLd + n], rk[hh]);
          rk[hh] = fmaf(t1v, B1[j * kLd + n + 1], rk[hh]);
          *reinterpret_cast<float2*>(p.ttdw + sl * 64 * D + (size_t)j * D + f0 + n) = make_float2(t0v, t1v);
        }
    }
    rk[0] = quad_sum(rk[0]);
    rk[1] = quad_sum(rk[1]);
    if ((lane & 3) == 0) {
      pk[r0 * 8 + nh] = rk[0];
      pk[(r0 + 8) * 8 + nh] = rk[1];
    }
  }
  // Z = (Z1 + Z2) diag(beta), stored transposed
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = col64(nt, e);
      Zm[j * kLd + row(e)] = bt[j] * az[nt][e];
    }
  __syncthreads();
  {  // Z^T T (T[k][n] = 0 for k < n), stored transposed
    float acc[2][4];
    zero(acc);
    mma_rowk<2>(acc, Zm, kLd, Tt, kLd, 16 * mt, 16 * nh, 16 * nh, 64, lane);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) Tp[col64(nt, e) * kLd + row(e)] = acc[nt][e];
  }
  __syncthreads();
  {  // dA[j][m] = -sum_l (Z^T T)[l][j] T[m][l] on the strict lower triangle (T[m][l] = 0 for
     // l > m)
    float acc[2][4];
    zero(acc);
    if (lower) mma_rowk<2>(acc, Tp, kLd, Tm, kLd, 16 * mt, 16 * nh, 0, 16 * nh + 16, lane);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = row(e), j = col64(nt, e);
        Zm[i * kLd + j] = j < i ? -acc[nt][e] : 0.f;
      }
  }
  __syncthreads();
  // k and q of features f0..f0+63 (two blocks each) for the dq / dk stage, stored
  // feature-major (scalar element map); the first pass's are in flight during the row sums
  // and the PG pass
  Blk bk[2], bq[2];
  auto load_kq64 = [&](int f0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      load_blk(bk[hh], L, tid, [&](int i, int f) { return kin(i, f0 + 32 * hh + f); });
      load_blk(bq[hh], L, tid, [&](int i, int f) { return qin(i, f0 + 32 * hh + f); });
    }
  };
  load_kq64(0);
  // ---------------- row and column sums: dbeta and dG parts from A and from dP
  {  // eight threads per row i, each over columns j = 8 m + sub, then a fixed shuffle sum
    const int i = tid >> 3, sub = tid & 7;
    float db = 0.f, dg = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int j = 8 * m + sub;
      const float da = Zm[i * kLd + j], gk = GK[i * kLd + j];
      db = fmaf(da, gk, db);
      dg = fmaf(da, bt[i] * gk, dg);                      // row of dA * A
      dg = fmaf(dP[i * kLd + j], Mm[i * kLd + j], dg);    // row of dP * M
      dg -= Zm[j * kLd + i] * bt[j] * GK[j * kLd + i];    // column of dA * A
      dg -= dP[j * kLd + i] * Mm[j * kLd + i];            // column of dP * M
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      db += __shfl_xor_sync(0xffffffffu, db, o);
      dg += __shfl_xor_sync(0xffffffffu, dg, o);
    }
    if (sub == 0) {
      const float sv = (pv[i * 8] + pv[i * 8 + 1]) + (pv[i * 8 + 2] + pv[i * 8 + 3]);
      const float sk = (pk[i * 8] + pk[i * 8 + 1]) + (pk[i * 8 + 2] + pk[i * 8 + 3]);
      rsk[i] = sk;
      dBv[i] = sv + eG[i] * sk + db;
      dGv[i] = dg + bt[i] * eG[i] * sk;
    }
  }
  __syncthreads();
  // PG = dP * Gamma (lower incl.) into dP and, transposed, into Tp; GK = dAt + dAt^T with
  // dAt = dA * beta_i Gamma_ij
  for (int idx = tid; idx < 64 * 64; idx += kThrC) {
    int i, j;
    patch_ij(idx, i, j);
    const float ex = expf(j <= i ? G[i] - G[j] : G[j] - G[i]);  // one of the two is used
    const float gij = j <= i ? ex : 0.f;
    const float gji = i <= j ? ex : 0.f;
    const float pg = dP[i * kLd + j] * gij;
    dP[i * kLd + j] = pg;  // in place: this pass reads dP at (i, j) only
    Tp[j * kLd + i] = pg;
    GK[i * kLd + j] = Zm[i * kLd + j] * bt[i] * gij + Zm[j * kLd + i] * bt[j] * gji;
  }
  // (the dq / dk stage's first barrier orders these writes before its products)
  // ---------------- key features again: dq and dk parts of this value head, 64 features a
  // pass; the feature-major k and q tiles take the T and T^T buffers, dead from here on
  {
    float* Rk = Tm;
    float* Rq = Tt;
    float rq[2] = {0.f, 0.f}, rw[2] = {0.f, 0.f};
    for (int fp = 0; fp < D / 64; ++fp) {
      __syncthreads();
      const int f0 = fp * 64;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        store_fm(Rk + 32 * h * kLd, bk[h], tid);
        store_fm(Rq + 32 * h * kLd, bq[h], tid);
      }
      __syncthreads();
      if (fp + 1 < D / 64) load_kq64(f0 + 64);
      // the epilogue's inputs (dO S^T, v_new dS^T, T^T dw of this thread's elements) are
      // loaded before the products, which cover their latency
      float2 os2[2][2], y2[2][2], tw2[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const size_t at = sl * 64 * D + (size_t)(r0 + 8 * hh) * D + f0 + col64(nt, 0);
          os2[nt][hh] = *reinterpret_cast<const float2*>(p.dos + at);
          y2[nt][hh] = *reinterpret_cast<const float2*>(p.ys + at);
          tw2[nt][hh] = *reinterpret_cast<const float2*>(p.ttdw + at);
        }
      float aq[2][4], ak[2][4];
      zero(aq);
      zero(ak);
      // PG is lower triangular: (PG K)[i] takes tokens j <= i, (PG^T Q)[i] tokens j >= i
      mma_rowk<2, false, kX>(aq, dP, kLd, Rk, kLd, 16 * mt, 16 * nh, 0, 16 * mt + 16, lane);
      mma_rowk<2, false, kX>(ak, Tp, kLd, Rq, kLd, 16 * mt, 16 * nh, 16 * mt, 64, lane);
      mma_rowk<2, false, kX>(ak, GK, kLd, Rk, kLd, 16 * mt, 16 * nh, 0, 64, lane);  // (dAt + dAt^T) K
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = r0 + 8 * hh, d = col64(nt, 0);
          const size_t at = sl * 64 * D + (size_t)i * D + f0 + d;
          const float os[2] = {os2[nt][hh].x, os2[nt][hh].y};
          const float y[2] = {y2[nt][hh].x, y2[nt][hh].y};
          const float tw[2] = {tw2[nt][hh].x, tw2[nt][hh].y};
          float dq[2], dk[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 2 * hh + u;
            const float qv = Rq[(d + u) * kLd + i], kv = Rk[(d + u) * kLd + i];
            rq[hh] = fmaf(qv, os[u], rq[hh]);
            rw[hh] = fmaf(kv, y[u], rw[hh]);
            dq[u] = fmaf(p.scale * eG[i], os[u], aq[nt][e]);
            dk[u] = ak[nt][e] + eL[i] * y[u] + bt[i] * eG[i] * tw[u];
          }
          *reinterpret_cast<float2*>(p.dqp + at) = make_float2(dq[0], dq[1]);
          *reinterpret_cast<float2*>(p.dkp + at) = make_float2(dk[0], dk[1]);
        }
    }
    rq[0] = quad_sum(rq[0]);
    rq[1] = quad_sum(rq[1]);
    rw[0] = quad_sum(rw[0]);
    rw[1] = quad_sum(rw[1]);
    if ((lane & 3) == 0) {
      pq[r0 * 8 + nh] = rq[0];
      pq[(r0 + 8) * 8 + nh] = rq[1];
      pw[r0 * 8 + nh] = rw[0];
      pw[(r0 + 8) * 8 + nh] = rw[1];
    }
  }
  __syncthreads();
  if (tid < 64) {
    const int i = tid;
    const float sq = (pq[i * 8] + pq[i * 8 + 1]) + (pq[i * 8 + 2] + pq[i * 8 + 3]);
    const float sw = (pw[i * 8] + pw[i * 8 + 1]) + (pw[i * 8 + 2] + pw[i * 8 + 3]);
    wsum[i] = eL[i] * sw;
    dGv[i] += p.scale * eG[i] * sq - eL[i] * sw;
  }
  __syncthreads();
  if (warp == 0) {  // rows lane and lane + 32, fixed shuffle orders
    // exp(G_L) terms go to the last row (G is flat past the chunk end)
    float sw = wsum[lane] + wsum[lane + 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
    float d0 = dGv[lane], d1 = dGv[lane + 32];
    if (lane == 31) d1 += sw + expf(G[63]) * p.sdot[sl];
    // dg = reverse in-chunk cumsum of dG: suffix sums within each half, then the upper
    // half's total added to the lower half
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y0 = __shfl_down_sync(0xffffffffu, d0, o);
      const float y1 = __shfl_down_sync(0xffffffffu, d1, o);
      if (lane + o < 32) {
        d0 += y0;
        d1 += y1;
      }
    }
    d0 += __shfl_sync(0xffffffffu, d1, 0);
    if (lane < L) {
      p.dg[(size_t)(t0 + lane) * p.Hv + hv] = d0;
      p.dbeta[(size_t)(t0 + lane) * p.Hv + hv] = dBv[lane];
    }
    if (lane + 32 < L) {
      p.dg[(size_t)(t0 + lane + 32) * p.Hv + hv] = d1;
      p.dbeta[(size_t)(t0 + lane + 32) * p.Hv + hv] = dBv[lane + 32];
    }
  }
}

// dq, dk = sum over the value heads of each key head group (fixed order)
template <int D>
__global__ void __launch_bounds__(kThr) bwd_reduce_kernel(BwdParams p) {
  const int tid = threadIdx.x, h = blockIdx.y;
  int t0, L, wslot;
  if (!resolve_slot(p, blockIdx.x, t0, L, wslot)) return;
  for (int idx = 4 * tid; idx < L * D; idx += 4 * kThr) {  // four features at a time
    const int i = idx / D, d = idx % D;
    float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
    for (int r = 0; r < p.HG; ++r) {
      const size_t at = ((size_t)wslot * p.Hv + h * p.HG + r) * 64 * D + idx;
      const float4 a = *reinterpret_cast<const float4*>(p.dqp + at);
      const float4 b = *reinterpret_cast<const float4*>(p.dkp + at);
      sq.x += a.x; sq.y += a.y; sq.z += a.z; sq.w += a.w;
      sk.x += b.x; sk.y += b.y; sk.z += b.z; sk.w += b.w;
    }
    const size_t o = ((size_t)(t0 + i) * p.H + h) * D + d;
    *reinterpret_cast<float4*>(p.dq + o) = sq;
    *reinterpret_cast<float4*>(p.dk + o) = sk;
  }
}

template <typename TIn, int D, bool TC>
bool launch_bwd_t(const BwdParams& p, cudaStream_t s, cudaEvent_t* ev) {
  constexpr int BV = bv_of<D>();
  const int s1 = (int)(scan_floats<D>() * sizeof(float));
  const int s2 = (int)state_mma_bytes<D>();
  const int s3 = (int)(chunk_floats() * sizeof(float));
  if (!TC) ensure_smem_limit((const void*)bwd_scan_kernel<D>, s1);
  ensure_smem_limit((const void*)bwd_state_kernel<D>, s2);
  ensure_smem_limit((const void*)bwd_chunk_kernel<TIn, D>, s3);
  if constexpr (TC) {  // the tensor-core bridge (bf16 inputs): the warp-MMA scan
    if (!launch_bwd_scan_tc(p, D, s)) return false;
  } else {
    bwd_scan_kernel<D><<<dim3(p.N, p.Hv, D / BV), kThr, s1, s>>>(p);
  }
  if (ev) cudaEventRecord(ev[0], s);
  if (p.nt_max > 0) bwd_state_kernel<D><<<dim3(p.nt_max, p.Hv), kThr, s2, s>>>(p);
  if (ev) cudaEventRecord(ev[1], s);
  if (p.nt_max > 0) {
    bwd_chunk_kernel<TIn, D><<<dim3(p.nt_max, p.Hv), kThrC, s3, s>>>(p);
    bwd_reduce_kernel<D><<<dim3(p.nt_max, p.H), kThr, 0, s>>>(p);
  }
  if (ev) cudaEventRecord(ev[2], s);
  return cudaPeekAtLastError() == cudaSuccess;
}

}  // namespace

bool launch_bwd(const BwdParams& p, int D, bool bf16_inputs, bool tc_bridge, cudaStream_t s,
                cudaEvent_t* ev) {
  if (tc_bridge)  // the tensor-core bridge exists for bf16 inputs only
    return D == 128 ? launch_bwd_t<__nv_bfloat16, 128, true>(p, s, ev)
                    : launch_bwd_t<__nv_bfloat16, 64, true>(p, s, ev);
  if (D == 128)
    return bf16_inputs ? launch_bwd_t<__nv_bfloat16, 128, false>(p, s, ev)
                       : launch_bwd_t<float, 128, false>(p, s, ev);
  return bf16_inputs ? launch_bwd_t<__nv_bfloat16, 64, false>(p, s, ev)
                     : launch_bwd_t<float, 64, false>(p, s, ev);
}

}  // namespace gdn
