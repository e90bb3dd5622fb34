// K2, bf16 inputs: fused intra-chunk kernel over [chunk slots, key heads].
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 4: K K^T is
// computed once per (chunk, key head) and reused by the value heads of the
// group; per value head the decay/beta-scaled A, its triangular inverse and
// the products that need it are formed without writing A to global memory.
// Section 8: triangular work stays triangular (only tiles on or below the
// diagonal of K K^T, Q K^T and T K are multiplied).
//
// Per (chunk, key head h), with rows past the end of the sequence masked
// (k = q = 0, beta = 0, g = 0):
//   P = K K^T, R = Q K^T        (bf16 MMA, fp32 accumulate: exact products),
//                                kept in registers across the value-head loop
//   per value head hv of the group:
//     G = inclusive in-chunk cumsum of g (fp32, left to right)
//     A_ij = beta_i exp(G_i - G_j) P_ij (j < i);  T = (I + A)^-1 in place (fp32 diagonal
//            blocks, off-diagonal blocks on tensor-core MMAs with split operands)
//     w    = (T diag(beta exp(G))) K        (bf16 operand and store)
//     u    = (T diag(beta)) V               (T operand split into bf16 hi + lo; fp32 store)
//     M_ij = exp(G_i - G_j) R_ij (j <= i)   (stored as a bf16 hi/lo pair)
// The hi/lo split keeps about 16 significant bits where one bf16 rounding
// would cost ~1e-2 of the output's rms. MMA A-fragments of the scaled T are
// built in registers straight from the fp32 T tile.
//
// The bridge is written as the exact shared-memory images the inter-chunk
// kernel's tensor cores read, so that kernel moves each with one bulk copy:
//   w: two 64-column halves, each [64 rows][128 B] with the 128-byte swizzle
//      (16-byte chunk c of row r stored at chunk c ^ (r % 8));
//   M: [128 rows: hi then lo][128 B], same swizzle;
//   u: [dv/32 blocks][64 rows][32 fp32], 16-byte chunk c of row r at c ^ (r % 8);
//   k (once per key head): fp16, scaled by 1/||k|| when the L2 norm is on, zero past
//      the sequence end, two 64-column halves of [64 rows][128 B] with the 128-byte swizzle.
//
// Occupancy: ~75 KB of shared memory and 128 threads per CTA, so that several
// CTAs share an SM and hide each other's latency.
#include "gdn_common.cuh"
#include "tri_inverse.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int LDB = 136;  // bf16 stride of 128-wide tiles (272 B rows: conflict-free ldmatrix)
constexpr int LDT = 68;   // fp32 stride of the A/T tile (16-byte rows)

struct IntraSmem {
  __nv_bfloat16 K[64 * LDB], Q[64 * LDB], V[64 * LDB];
  float AT[64 * LDT];
  float X[16 * LDT];
  float G[64], B[64], E[64], KR[64];
};

// Byte offset of bf16 element (r, k), k < 64, in a [rows][128 B] tile with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  return (uint32_t)r * 128u + ((uint32_t)((k >> 3) ^ (r & 7)) << 4) + (uint32_t)(k & 7) * 2u;
}
// Byte offset of fp32 element (r, j), j < 32, in a [rows][32] tile with 16-byte chunks swizzled.
__device__ __forceinline__ uint32_t u_offset(int r, int j) {
  return (uint32_t)r * 128u + ((uint32_t)((j >> 2) ^ (r & 7)) << 4) + (uint32_t)(j & 3) * 4u;
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

// 64 rows x 128 bf16 of a [T, heads, 128] tensor into a padded tile; rows >= L read as zero.
__device__ __forceinline__ void load_rows(__nv_bfloat16* dst, const __nv_bfloat16* src, int t0,
                                          int L, int heads, int head, int tid) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int idx = tid + it * 128;  // 1024 chunks of 16 bytes
    const int i = idx >> 4, c = (idx & 15) * 8;
    const bool ok = i < L;
    const __nv_bfloat16* g = src + (((size_t)(ok ? t0 + i : t0) * heads + head) * kDk + c);
    cp_async16(dst + i * LDB + c, g, ok);
  }
}

__global__ void __launch_bounds__(128, 3) tc_intra_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  IntraSmem& s = *reinterpret_cast<IntraSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = 2 * (lane & 3);
  const int h = blockIdx.y;
  int t0, L, wslot;
  if (!resolve(p, blockIdx.x, t0, L, wslot)) return;

  load_rows(s.K, static_cast<const __nv_bfloat16*>(p.k), t0, L, p.H, h, tid);
  load_rows(s.Q, static_cast<const __nv_bfloat16*>(p.q), t0, L, p.H, h, tid);
  cp_async_commit();
  if (tid < 64) {  // optional L2-norm factors (1 when off)
    s.KR[tid] = (tid < L && p.krn) ? p.krn[(size_t)(t0 + tid) * p.H + h] : 1.f;
  }
  const int r0 = 16 * warp;
  float qra = 1.f, qrb = 1.f;  // 1/||q|| of this thread's two rows
  if (p.qrn) {
    qra = (r0 + g < L) ? p.qrn[(size_t)(t0 + r0 + g) * p.H + h] : 1.f;
    qrb = (r0 + g + 8 < L) ? p.qrn[(size_t)(t0 + r0 + g + 8) * p.H + h] : 1.f;
  }
  cp_async_wait<0>();
  __syncthreads();

  {  // fp16 image of the (normalised) k tile for the inter-chunk state update
    unsigned char* kimg = static_cast<unsigned char*>(p.k16) + ((size_t)wslot * p.H + h) * 64 * kDk * 2;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int idx = tid + it * 128;  // 1024 chunks of 8 elements
      const int half = idx >> 9, t = (idx >> 3) & 63, ch = idx & 7;
      const uint4 raw = *reinterpret_cast<const uint4*>(&s.K[t * LDB + half * 64 + ch * 8]);
      const uint32_t* r = reinterpret_cast<const uint32_t*>(&raw);
      uint4 v;
      uint32_t* o = reinterpret_cast<uint32_t*>(&v);
      const float sc = s.KR[t];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[e]));
        o[e] = pack_f16(f.x * sc, f.y * sc);
      }
      *reinterpret_cast<uint4*>(kimg + half * 8192 + t * 128 + ((ch ^ (t & 7)) << 4)) = v;
    }
  }

  // P = K K^T and R = Q K^T, rows r0..r0+15, column tiles on or below the diagonal.
  float kk[8][4], qk[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) kk[nt][e] = qk[nt][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t ak[4], aq[4];
    load_a(ak, s.K, LDB, r0, 16 * ks, lane);
    load_a(aq, s.Q, LDB, r0, 16 * ks, lane);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      if (np <= warp) {
        uint32_t b[4];
        load_b_nk(b, s.K, LDB, 16 * ks, 16 * np, lane);
        mma_bf16(kk[2 * np], ak, b[0], b[1]);
        mma_bf16(kk[2 * np + 1], ak, b[2], b[3]);
        mma_bf16(qk[2 * np], aq, b[0], b[1]);
        mma_bf16(qk[2 * np + 1], aq, b[2], b[3]);
      }
    }
  }

  for (int r = 0; r < p.HG; ++r) {
    const int hv = h * p.HG + r;
    const size_t sl = (size_t)wslot * p.Hv + hv;
    load_rows(s.V, static_cast<const __nv_bfloat16*>(p.v), t0, L, p.Hv, hv, tid);
    cp_async_commit();
    if (warp == 0) {  // gates and their in-chunk inclusive cumsum (64 rows, 2 per lane)
      const size_t b0 = (size_t)(t0 + lane) * p.Hv + hv, b1 = (size_t)(t0 + lane + 32) * p.Hv + hv;
      float g0 = lane < L ? p.g[b0] : 0.f, g1 = lane + 32 < L ? p.g[b1] : 0.f;
      const float be0 = lane < L ? p.beta[b0] : 0.f, be1 = lane + 32 < L ? p.beta[b1] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y0 = __shfl_up_sync(0xffffffffu, g0, o);
        const float y1 = __shfl_up_sync(0xffffffffu, g1, o);
        if (lane >= o) { g0 += y0; g1 += y1; }
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      s.G[lane] = g0;
      s.G[lane + 32] = g1;
      s.E[lane] = expf(g0);
      s.E[lane + 32] = expf(g1);
      s.B[lane] = be0;
      s.B[lane + 32] = be1;
      p.G[sl * 64 + lane] = g0;
      p.G[sl * 64 + lane + 32] = g1;
    }
    __syncthreads();

    // A (strictly lower, to shared memory) and M (hi/lo, to global) from the register tiles.
    {
      unsigned char* Mimg = static_cast<unsigned char*>(p.M) + sl * 2 * 64 * 64 * 2;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = r0 + g + 8 * hh;
        const float gi = s.G[i], bi = s.B[i] * s.KR[i], qi = hh ? qrb : qra;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int j = 8 * nt + c;
          float a2[2], m2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int jj = j + e;
            const float dec = (jj <= i) ? __expf(gi - s.G[jj]) : 0.f;
            a2[e] = (jj < i) ? bi * dec * s.KR[jj] * kk[nt][2 * hh + e] : 0.f;
            m2[e] = dec * qi * s.KR[jj] * qk[nt][2 * hh + e];
          }
          *reinterpret_cast<float2*>(&s.AT[i * LDT + j]) = make_float2(a2[0], a2[1]);
          split2_store(reinterpret_cast<__nv_bfloat16*>(Mimg + sw128_offset(i, j)),
                       reinterpret_cast<__nv_bfloat16*>(Mimg + sw128_offset(64 + i, j)), m2[0], m2[1]);
        }
      }
    }
    __syncthreads();
    tri_inverse_64_tc(s.AT, LDT, s.X, tid);

    // w = (T diag(beta exp(G) krn)) K, rows r0..r0+15; T is lower triangular (k-tiles <= warp).
    {
      float acc[16][4];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (ks <= warp) {
          uint32_t a[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // a0: (g, c) a1: (g+8, c) a2: (g, c+8) a3: (g+8, c+8)
            const int i = r0 + g + 8 * (q4 & 1), j = 16 * ks + c + 8 * (q4 >> 1);
            const float2 t = *reinterpret_cast<const float2*>(&s.AT[i * LDT + j]);
            a[q4] = pack_bf16(t.x * s.B[j] * s.E[j] * s.KR[j], t.y * s.B[j + 1] * s.E[j + 1] * s.KR[j + 1]);
          }
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            uint32_t b[4];
            load_b_kn(b, s.K, LDB, 16 * ks, 16 * np, lane);
            mma_bf16(acc[2 * np], a, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
          }
        }
      }
      unsigned char* wimg = static_cast<unsigned char*>(p.w) + sl * 64 * kDk * 2;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int col = 8 * nt + c;
        unsigned char* half = wimg + (col >> 6) * 8192;
        *reinterpret_cast<uint32_t*>(half + sw128_offset(r0 + g, col & 63)) = pack_bf16(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<uint32_t*>(half + sw128_offset(r0 + g + 8, col & 63)) = pack_bf16(acc[nt][2], acc[nt][3]);
      }
    }
    // u = (T diag(beta)) V with the T operand split into bf16 hi + lo.
    cp_async_wait<0>();
    __syncthreads();
    {
      float acc[16][4];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (ks <= warp) {
          uint32_t ah[4], al[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int i = r0 + g + 8 * (q4 & 1), j = 16 * ks + c + 8 * (q4 >> 1);
            const float2 t = *reinterpret_cast<const float2*>(&s.AT[i * LDT + j]);
            const float x0 = t.x * s.B[j], x1 = t.y * s.B[j + 1];
            const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
            ah[q4] = *reinterpret_cast<const uint32_t*>(&hi);
            al[q4] = *reinterpret_cast<const uint32_t*>(&lo);
          }
#pragma unroll
          for (int np = 0; np < 8; ++np) {
            uint32_t b[4];
            load_b_kn(b, s.V, LDB, 16 * ks, 16 * np, lane);
            mma_bf16(acc[2 * np], ah, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], ah, b[2], b[3]);
            mma_bf16(acc[2 * np], al, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], al, b[2], b[3]);
          }
        }
      }
      unsigned char* uimg = reinterpret_cast<unsigned char*>(p.u + sl * 64 * kDv);
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int col = 8 * nt + c;
        unsigned char* blk = uimg + (col >> 5) * 64 * 32 * 4;
        *reinterpret_cast<float2*>(blk + u_offset(r0 + g, col & 31)) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(blk + u_offset(r0 + g + 8, col & 31)) = make_float2(acc[nt][2], acc[nt][3]);
      }
    }
    __syncthreads();  // A/T and the gates are rewritten for the next value head
  }
}

}  // namespace

void launch_tc_intra(const Params& p, cudaStream_t s) {
  const int smem = (int)sizeof(IntraSmem);
  ensure_smem_limit((const void*)tc_intra_kernel, smem);
  tc_intra_kernel<<<dim3(p.nt_max, p.H), 128, smem, s>>>(p);
}

}  // namespace gdn
