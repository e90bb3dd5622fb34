// General chunk path: fp32 SIMT arithmetic for every case the bf16 tensor-core
// path does not take: fp32 inputs, head dimension 64, and per-channel gates.
// The decomposition is the same intra/inter split as the tensor-core path
// ("Optimizing GDN Chunk Prefill on Intel AMX CPU", sections 4 and 5), written
// once for a gate vector per key channel; a scalar gate is the case where all
// channels carry the same value.
//
// Intra (grid [nt_max, H], one CTA per chunk and key head, value heads of the
// group in turn). With G the in-chunk cumulative log-decay (per channel d):
//   A_ij = beta_i sum_d k_id k_jd exp(G_id - G_jd)   (j < i)     T = (I + A)^-1
//   M_ij =        sum_d q_id k_jd exp(G_id - G_jd)   (j <= i)
//   w    = T diag(beta) (exp(G) * K),   u = T diag(beta) V
//   Qt   = exp(G) * Q,   Kt = exp(G_L - G) * K,   gam = exp(G_L)
// Inter (grid [N, Hv, D / BV]), per chunk, with the fp32 state S [D x BV]:
//   v_new = u - w S,   o = scale (Qt S + M v_new),   S <- diag(gam) S + Kt^T v_new
//
// Exponent ranges (gates g <= 0, G non-increasing along the chunk): per-channel
// A and M entries of two different 16-row blocks bi > bj are products of
// k_i exp(G_i - G_r) and k_j exp(G_r - G_j) with the reference row r = 16 bi,
// both factors <= 1; entries inside one 16-row block exponentiate G_i - G_j
// directly. No factor ever exceeds 1, so no gate value can overflow.
#include "gdn_common.cuh"
#include "simt_tile.cuh"
#include "tri_inverse.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kThr = 256;
constexpr uint32_t kGenWaitIters = 1u << 22;

// Shared-memory floats of the intra kernel.
template <int D, bool CH>
constexpr int intra_floats() {
  return 64 * D                       // Kr
         + (CH ? 64 * D : 0)          // Gc (per-channel cumulative gates)
         + (CH ? 192 * D : 136 * D)   // E: operand images, then q / (exp(G) k) / v
         + 64 + 64 * 65 + 64 * 64 + 16 * 65 + 2 * 64;
}

template <typename TIn, int D, bool CH>
__global__ void __launch_bounds__(kThr) gen_intra_kernel(Params p) {
  extern __shared__ __align__(16) float sm[];
  float* Kr = sm;                          // [64][D] k rows (zero past the chunk end)
  float* Gc = Kr + 64 * D;                 // CH: [64][D] cumulative gates
  float* E = Gc + (CH ? 64 * D : 0);       // operand images
  float* Gs = E + (CH ? 192 * D : 136 * D);  // [64] cumulative scalar gate
  float* A = Gs + 64;                      // [64][65] A, then T = (I + A)^-1 in place
  float* TT = A + 64 * 65;                 // [64][64] M^T, then the w / u left operands
  float* Xs = TT + 64 * 64;                // [16][65] scratch of the inverse
  float* Bt = Xs + 16 * 65;                // [64] beta
  float* Eg = Bt + 64;                     // [64] exp(G) (scalar gates)

  const int tid = threadIdx.x, h = blockIdx.y;
  int t0, L, wslot;
  if (!resolve_slot(p, blockIdx.x, t0, L, wslot)) return;

  auto qk_row_scale = [&](const float* rn, int i) {
    return rn ? rn[(size_t)(t0 + i) * p.H + h] : 1.f;
  };
  staged_copy<8>(64 * D, tid, kThr,
                 [&](int idx) {
                   const int i = idx / D;
                   return i < L ? ld_in<TIn>(p.k, ((size_t)(t0 + i) * p.H + h) * D + idx % D) *
                                      qk_row_scale(p.krn, i)
                                : 0.f;
                 },
                 [&](int idx, float x) { Kr[idx] = x; });

  for (int r = 0; r < p.HG; ++r) {
    const int hv = h * p.HG + r;
    const size_t sl = (size_t)wslot * p.Hv + hv;
    if (tid < 64) {
      const bool ok = tid < L;
      Bt[tid] = ok ? p.beta[(size_t)(t0 + tid) * p.Hv + hv] : 0.f;
      if (!CH) Gs[tid] = ok ? p.g[(size_t)(t0 + tid) * p.Hv + hv] : 0.f;
    }
    for (int idx = tid; idx < 64 * 65; idx += kThr) A[idx] = 0.f;
    for (int idx = tid; idx < 64 * 64; idx += kThr) TT[idx] = 0.f;
    if constexpr (CH) {  // gate rows in (coalesced), zero past the chunk end
      staged_copy<8>(64 * D, tid, kThr,
                     [&](int idx) {
                       const int i = idx / D;
                       return i < L ? p.g[((size_t)(t0 + i) * p.Hv + hv) * D + idx % D] : 0.f;
                     },
                     [&](int idx, float x) { Gc[idx] = x; });
    }
    __syncthreads();
    if constexpr (CH) {  // inclusive cumsum along the chunk, one thread per channel
      for (int d = tid; d < D; d += kThr) {
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < 64; ++i) {
          acc += Gc[i * D + d];
          Gc[i * D + d] = acc;
        }
      }
    }
    if (!CH && tid == 0) {  // inclusive cumsum, left to right
      float acc = 0.f;
      for (int i = 0; i < 64; ++i) {
        acc += Gs[i];
        Gs[i] = acc;
      }
    }
    __syncthreads();
    if (!CH && tid < 64) Eg[tid] = expf(Gs[tid]);

    if constexpr (!CH) {
      // ------------------------------------------------ scalar gate: k and q images [D][68]
      float* KT = E;
      float* QT = E + 68 * D;
      {  // element e: lane = e % 32 covers 8 d x 4 i, e / 32 picks the (d, i) block
        auto dof = [&](int e) { return ((e >> 5) % (D / 8)) * 8 + (e & 7); };
        auto iof = [&](int e) { return ((e >> 5) / (D / 8)) * 4 + ((e >> 3) & 3); };
        staged_copy<8>(64 * D, tid, kThr,
                       [&](int e) {
                         const int i = iof(e);
                         return i < L ? ld_in<TIn>(p.q, ((size_t)(t0 + i) * p.H + h) * D + dof(e)) *
                                            qk_row_scale(p.qrn, i)
                                      : 0.f;
                       },
                       [&](int e, float x) {
                         const int d = dof(e), i = iof(e);
                         KT[d * 68 + i] = Kr[i * D + d];
                         QT[d * 68 + i] = x;
                       });
      }
      __syncthreads();
      // A and M over 4x4 tiles of the lower triangle (one tile per thread)
      {
        const int i0 = (tid >> 4) * 4, j0 = (tid & 15) * 4;
        if (j0 <= i0) {
          float ak[4][4], aq[4][4];
          zero(ak);
          zero(aq);
#pragma unroll 2
          for (int d = 0; d < D; ++d) {
            float ki[4], qi[4], kj[4];
            ldv<4>(KT + d * 68 + i0, ki);
            ldv<4>(QT + d * 68 + i0, qi);
            ldv<4>(KT + d * 68 + j0, kj);
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                ak[a][b] = fmaf(ki[a], kj[b], ak[a][b]);
                aq[a][b] = fmaf(qi[a], kj[b], aq[a][b]);
              }
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const int i = i0 + a, j = j0 + b;
              if (j <= i) {
                const float dec = expf(Gs[i] - Gs[j]);
                if (j < i) A[i * 65 + j] = Bt[i] * dec * ak[a][b];
                TT[j * 64 + i] = dec * aq[a][b];
              }
            }
        }
      }
      // Qt^T = exp(G_i) q_i (from the q image), Kt = exp(G_L - G_i) k_i, gam = exp(G_L)
      float* qt = p.qt + sl * 64 * D;
      float* kt = p.kt + sl * 64 * D;
      const float gl = Gs[63];
      for (int idx = tid; idx < 64 * D; idx += kThr) {
        qt[idx] = Eg[idx & 63] * QT[(idx >> 6) * 68 + (idx & 63)];  // [D][64]
        kt[idx] = expf(gl - Gs[idx / D]) * Kr[idx];                 // [64][D]
      }
      for (int d = tid; d < D; d += kThr) p.gam[sl * D + d] = expf(gl);
      __syncthreads();
    } else {
      // ------------------------------------------------ per-channel gates
      float* EkT = E;             // [D][48]: k_i exp(G_i - G_r(i)), rows i = 16..63
      float* EqT = E + 48 * D;    // [D][48]: same for q
      float* FT = E + 96 * D;     // [D][96]: k_j exp(G_r - G_j), one 16-block per pair
      {
        const int dl = tid & 7, il = (tid >> 3) & 3, grp = tid >> 5;
        auto dof = [&](int e) { return ((e >> 5) % (D / 8)) * 8 + (e & 7); };
        auto iof = [&](int e) { return 16 + ((e >> 5) / (D / 8)) * 4 + ((e >> 3) & 3); };
        staged_copy<8>(48 * D, tid, kThr,
                       [&](int e) {
                         const int i = iof(e);
                         return i < L ? ld_in<TIn>(p.q, ((size_t)(t0 + i) * p.H + h) * D + dof(e)) *
                                            qk_row_scale(p.qrn, i)
                                      : 0.f;
                       },
                       [&](int e, float qv) {
                         const int d = dof(e), i = iof(e);
                         const int ref = i & ~15;  // first row of i's block
                         const float ex = __expf(Gc[i * D + d] - Gc[ref * D + d]);
                         EkT[d * 48 + i - 16] = Kr[i * D + d] * ex;
                         EqT[d * 48 + i - 16] = qv * ex;
                       });
        // pairs (bi, bj), bj < bi, in the order (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
        for (int blk = grp; blk < (D / 8) * 24; blk += kThr / 32) {
          const int d = (blk % (D / 8)) * 8 + dl, c = (blk / (D / 8)) * 4 + il;  // column 0..95
          const int pr = c >> 4, jj = c & 15;
          const int bi = pr < 1 ? 1 : (pr < 3 ? 2 : 3);
          const int bj = pr - (bi * (bi - 1)) / 2;
          const int j = 16 * bj + jj, ref = 16 * bi;
          FT[d * 96 + c] = Kr[j * D + d] * __expf(Gc[ref * D + d] - Gc[j * D + d]);
        }
      }
      __syncthreads();
      // off-diagonal blocks: 6 pairs x 64 tiles of 2x2
      for (int t = tid; t < 6 * 64; t += kThr) {
        const int pr = t >> 6, tt = t & 63;
        const int bi = pr < 1 ? 1 : (pr < 3 ? 2 : 3);
        const int bj = pr - (bi * (bi - 1)) / 2;
        const int ii = (tt >> 3) * 2, jj = (tt & 7) * 2;
        const int i0 = 16 * bi + ii, c0 = 16 * pr + jj;
        float ak[2][2], aq[2][2];
        zero(ak);
        zero(aq);
#pragma unroll 4
        for (int d = 0; d < D; ++d) {
          float ki[2], qi[2], fj[2];
          ldv<2>(EkT + d * 48 + i0 - 16, ki);
          ldv<2>(EqT + d * 48 + i0 - 16, qi);
          ldv<2>(FT + d * 96 + c0, fj);
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              ak[a][b] = fmaf(ki[a], fj[b], ak[a][b]);
              aq[a][b] = fmaf(qi[a], fj[b], aq[a][b]);
            }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int i = i0 + a, j = 16 * bj + jj + b;
            A[i * 65 + j] = Bt[i] * ak[a][b];
            TT[j * 64 + i] = aq[a][b];
          }
      }
      __syncthreads();
      // q rows into E (the images are consumed)
      float* Qr = E;
      staged_copy<8>(64 * D, tid, kThr,
                     [&](int idx) {
                       const int i = idx / D;
                       return i < L ? ld_in<TIn>(p.q, ((size_t)(t0 + i) * p.H + h) * D + idx % D) *
                                          qk_row_scale(p.qrn, i)
                                    : 0.f;
                     },
                     [&](int idx, float x) { Qr[idx] = x; });
      __syncthreads();
      // diagonal blocks: one warp per (i, j) pair, lanes over channels
      {
        const int warp = tid >> 5, lane = tid & 31;
        for (int pidx = warp; pidx < 4 * 136; pidx += kThr / 32) {
          const int b = pidx / 136;
          int rem = pidx % 136, ii = 0;
          while (rem > ii) {  // pairs (ii, jj) with jj <= ii, row by row
            rem -= ii + 1;
            ++ii;
          }
          const int i = 16 * b + ii, j = 16 * b + rem;
          float sk = 0.f, sq = 0.f;
          for (int d = lane; d < D; d += 32) {
            const float e = __expf(Gc[i * D + d] - Gc[j * D + d]) * Kr[j * D + d];
            sk = fmaf(Kr[i * D + d], e, sk);
            sq = fmaf(Qr[i * D + d], e, sq);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
          }
          if (lane == 0) {
            if (j < i) A[i * 65 + j] = Bt[i] * sk;
            TT[j * 64 + i] = sq;
          }
        }
      }
      // Qt^T = exp(G) q (transposed), Kt = exp(G_L - G) k, gam = exp(G_L)
      float* qt = p.qt + sl * 64 * D;
      float* kt = p.kt + sl * 64 * D;
      for (int idx = tid; idx < 64 * D; idx += kThr) {
        kt[idx] = __expf(Gc[63 * D + idx % D] - Gc[idx]) * Kr[idx];  // [64][D]
        const int d = idx >> 6, i = idx & 63;                          // [D][64]
        qt[idx] = __expf(Gc[i * D + d]) * Qr[i * D + d];
      }
      for (int d = tid; d < D; d += kThr) p.gam[sl * D + d] = __expf(Gc[63 * D + d]);
      __syncthreads();
    }

    // M^T out (zeros above the diagonal)
    {
      float4* mo = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.M) + sl * 64 * 64);
      const float4* ms = reinterpret_cast<const float4*>(TT);
      for (int idx = tid; idx < 64 * 16; idx += kThr) mo[idx] = ms[idx];
    }
    tri_inverse_64_inplace(A, 65, Xs, tid, kThr);  // ends synchronized

    // ------------------------------------------------ w = T diag(beta) (exp(G) * K)
    float* Y = E;  // [64][D] right operand
    for (int idx = tid; idx < 64 * 64; idx += kThr) {
      const int j = idx >> 6, i = idx & 63;
      TT[idx] = A[i * 65 + j] * Bt[j] * (CH ? 1.f : Eg[j]);  // (T diag(beta [exp G]))^T
    }
    for (int idx = tid; idx < 64 * D; idx += kThr)
      Y[idx] = CH ? __expf(Gc[idx]) * Kr[idx] : Kr[idx];
    __syncthreads();
    constexpr int NT = D / 4;  // column tiles of 4
    {
      float* wo = reinterpret_cast<float*>(p.w) + sl * 64 * D;  // [D][64] (w^T)
      for (int t = tid; t < 16 * NT; t += kThr) {
        const int i0 = (t / NT) * 4, d0 = (t % NT) * 4;
        float acc[4][4];
        zero(acc);
        fma_tile<4, 4>(acc, TT, 64, Y, D, i0, d0, 0, i0 + 4);  // T is lower triangular
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<float4*>(wo + (d0 + c) * 64 + i0) =
              make_float4(acc[0][c], acc[1][c], acc[2][c], acc[3][c]);
      }
    }
    __syncthreads();
    // ------------------------------------------------ u = T diag(beta) V
    for (int idx = tid; idx < 64 * 64; idx += kThr) {
      const int j = idx >> 6, i = idx & 63;
      TT[idx] = A[i * 65 + j] * Bt[j];
    }
    staged_copy<8>(64 * D, tid, kThr,
                   [&](int idx) {
                     const int i = idx / D;
                     return i < L ? ld_in<TIn>(p.v, ((size_t)(t0 + i) * p.Hv + hv) * D + idx % D)
                                  : 0.f;
                   },
                   [&](int idx, float x) { Y[idx] = x; });
    __syncthreads();
    {
      constexpr int BV = D == 128 ? 32 : 16;
      float* uo = p.u + sl * 64 * D;  // [D / BV][64][BV]
      for (int t = tid; t < 16 * NT; t += kThr) {
        const int i0 = (t / NT) * 4, d0 = (t % NT) * 4;
        float acc[4][4];
        zero(acc);
        fma_tile<4, 4>(acc, TT, 64, Y, D, i0, d0, 0, i0 + 4);
        float* ub = uo + (size_t)(d0 / BV) * 64 * BV + (d0 % BV);
#pragma unroll
        for (int a = 0; a < 4; ++a)
          *reinterpret_cast<float4*>(ub + (i0 + a) * BV) =
              make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- inter (scan)
template <int D>
constexpr int scan_bv() { return D == 128 ? 32 : 16; }

template <int D>
constexpr int scan_sld() { return scan_bv<D>() + 4; }  // state row stride (fewer bank conflicts)

template <int D>
constexpr size_t scan_smem_bytes() {
  constexpr int BV = scan_bv<D>(), SLD = scan_sld<D>();
  return sizeof(float) * (2 * D * SLD + 2 * D * 64 + 64 * D + 64 * 64 + 2 * 64 * BV + D) + 64;
}

template <int D>
__global__ void __launch_bounds__(kThr) gen_inter_kernel(Params p) {
  constexpr int BV = scan_bv<D>(), SLD = scan_sld<D>();
  extern __shared__ __align__(16) float sm[];
  float* S0 = sm;                    // [2][D][SLD] state (BV columns used), double buffered
  float* Wt = S0 + 2 * D * SLD;      // [D][64] w^T
  float* Qt = Wt + D * 64;           // [D][64] (exp(G) q)^T
  float* Kt = Qt + D * 64;           // [64][D] exp(G_L - G) k
  float* Mt = Kt + 64 * D;           // [64][64] M^T
  float* U = Mt + 64 * 64;           // [2][64][BV] u, then v_new
  float* gam = U + 2 * 64 * BV;      // [D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(gam + D);  // 0-1 u, 2 w, 3 rest

  const int tid = threadIdx.x;
  const int n = blockIdx.x, hv = blockIdx.y, cb = blockIdx.z, c0 = cb * BV;
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    if (tid == 0) set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }
  const size_t state_base = ((size_t)n * p.Hv + hv) * D * D;

  auto slot_of = [&](int c) { return (size_t)(sv.first_slot + c) * p.Hv + hv; };
  int issued[4] = {0, 0, 0, 0};  // copies issued per barrier (thread 0)
  auto issue_u = [&](int c) {
    const size_t sl = slot_of(c);
    uint64_t* b = &bars[c & 1];
    ++issued[c & 1];
    mbar_expect_tx(b, 64 * BV * 4);
    bulk_load(U + (c & 1) * 64 * BV, p.u + sl * 64 * D + (size_t)cb * 64 * BV, 64 * BV * 4, b);
  };
  auto issue_w = [&](int c) {
    const size_t sl = slot_of(c);
    ++issued[2];
    mbar_expect_tx(&bars[2], D * 64 * 4);
    bulk_load(Wt, reinterpret_cast<const float*>(p.w) + sl * 64 * D, D * 64 * 4, &bars[2]);
  };
  auto issue_rest = [&](int c) {
    const size_t sl = slot_of(c);
    ++issued[3];
    mbar_expect_tx(&bars[3], (2 * D * 64 + 64 * 64 + D) * 4);
    bulk_load(Qt, p.qt + sl * 64 * D, D * 64 * 4, &bars[3]);
    bulk_load(Kt, p.kt + sl * 64 * D, D * 64 * 4, &bars[3]);
    bulk_load(Mt, reinterpret_cast<const float*>(p.M) + sl * 64 * 64, 64 * 64 * 4, &bars[3]);
    bulk_load(gam, p.gam + sl * D, D * 4, &bars[3]);
  };

  if (tid == 0) {
    for (int b = 0; b < 4; ++b) mbar_init(&bars[b], 1);
    mbar_init_fence();
    if (nch > 0) {
      issue_u(0);
      issue_w(0);
      issue_rest(0);
    }
  }
  for (int idx = tid; idx < D * BV; idx += kThr) {
    const int d = idx / BV, j = idx % BV;
    S0[d * SLD + j] = p.s0 ? p.s0[state_base + (size_t)(c0 + j) * D + d] : 0.f;
  }
  __syncthreads();

  bool failed = false;
  int cur = 0;
  for (int c = 0; c < nch; ++c) {
    const float* S = S0 + cur * D * SLD;
    float* Sn = S0 + (cur ^ 1) * D * SLD;
    float* Uc = U + (c & 1) * 64 * BV;
    if (p.hs) {  // chunk-start state, [dv][dk] rows of the slot (for the backward pass)
      float* hs = p.hs + slot_of(c) * D * D;
      for (int idx = tid; idx < D * BV; idx += kThr) {
        const int j = idx / D, d = idx % D;
        hs[(size_t)(c0 + j) * D + d] = S[d * SLD + j];
      }
    }
    bool ok = mbar_wait(&bars[c & 1], (uint32_t)((c >> 1) & 1), kGenWaitIters);
    ok = ok && mbar_wait(&bars[2], (uint32_t)(c & 1), kGenWaitIters);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    // v_new = u - w S: 64 x BV outputs, 4 x (BV / 16) per thread
    {
      constexpr int RN = BV / 16;
      const int i0 = (tid >> 4) * 4, n0 = (tid & 15) * RN;
      float acc[4][RN];
      zero(acc);
      fma_tile<4, RN>(acc, Wt, 64, S, SLD, i0, n0, 0, D);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) Uc[(i0 + a) * BV + n0 + b] -= acc[a][b];
    }
    __syncthreads();
    if (p.vn_out) {
      float* vo = p.vn_out + slot_of(c) * 64 * D + c0;
      for (int idx = tid; idx < 64 * BV; idx += kThr) vo[(idx / BV) * D + idx % BV] = Uc[idx];
    }
    if (tid == 0 && c + 1 < nch) {
      fence_async_smem();
      issue_w(c + 1);
      issue_u(c + 1);
    }
    ok = mbar_wait(&bars[3], (uint32_t)(c & 1), kGenWaitIters);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    // o = scale (Qt S + M v_new) for rows < L, and S' = diag(gam) S + Kt^T v_new
    {
      const int t0 = sv.start + kChunk * c;
      const int L = min(kChunk, sv.len - kChunk * c);
      constexpr int RN = BV / 16;
      constexpr int OT = 16 * 16;              // output tiles of 4 x RN
      constexpr int ST = (D / 4) * 16;         // state tiles of 4 x RN
      for (int t = tid; t < OT + ST; t += kThr) {
        float acc[4][RN];
        zero(acc);
        if (t < OT) {
          const int i0 = (t >> 4) * 4, n0 = (t & 15) * RN;
          if (i0 >= L || !p.out) continue;  // no output when only the states are wanted
          fma_tile<4, RN>(acc, Qt, 64, S, SLD, i0, n0, 0, D);
          fma_tile<4, RN>(acc, Mt, 64, Uc, BV, i0, n0, 0, min(i0 + 4, 64));
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            if (i0 + a >= L) break;
            const size_t oi = ((size_t)(t0 + i0 + a) * p.Hv + hv) * D + c0 + n0;
#pragma unroll
            for (int b = 0; b < RN; ++b) {
              const float o = p.scale * acc[a][b];
              if (p.out_bf16)
                reinterpret_cast<__nv_bfloat16*>(p.out)[oi + b] = __float2bfloat16_rn(o);
              else
                reinterpret_cast<float*>(p.out)[oi + b] = o;
            }
          }
        } else {
          const int s = t - OT;
          const int d0 = (s >> 4) * 4, n0 = (s & 15) * RN;
          fma_tile<4, RN>(acc, Kt, D, Uc, BV, d0, n0, 0, 64);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < RN; ++b) {
              const int idx = (d0 + a) * SLD + n0 + b;
              Sn[idx] = fmaf(gam[d0 + a], S[idx], acc[a][b]);
            }
        }
      }
    }
    __syncthreads();
    if (tid == 0 && c + 1 < nch) {
      fence_async_smem();
      issue_rest(c + 1);
    }
    cur ^= 1;
  }
  if (failed) {
    if (tid == 0) {
      set_status(p.status, GDN_DEV_TIMEOUT);
      // let copies still in flight land before the CTA's shared memory is released
      // (phases complete in order: waiting for the last one issued covers the rest)
      for (int b = 0; b < 4; ++b)
        if (issued[b] > 0) mbar_wait(&bars[b], (uint32_t)((issued[b] - 1) & 1), kGenWaitIters);
    }
    return;
  }
  if (p.sT) {
    const float* S = S0 + cur * D * SLD;
    for (int idx = tid; idx < D * BV; idx += kThr) {
      const int j = idx / D, d = idx % D;
      p.sT[state_base + (size_t)(c0 + j) * D + d] = S[d * SLD + j];
    }
  }
}

template <typename TIn, int D, bool CH>
bool launch_intra_t(const Params& p, cudaStream_t s) {
  const int smem = intra_floats<D, CH>() * (int)sizeof(float);
  ensure_smem_limit((const void*)gen_intra_kernel<TIn, D, CH>, smem);
  gen_intra_kernel<TIn, D, CH><<<dim3(p.nt_max, p.H), kThr, smem, s>>>(p);
  return cudaPeekAtLastError() == cudaSuccess;
}

template <int D>
bool launch_inter_t(const Params& p, cudaStream_t s) {
  const int smem = (int)scan_smem_bytes<D>();
  ensure_smem_limit((const void*)gen_inter_kernel<D>, smem);
  gen_inter_kernel<D><<<dim3(p.N, p.Hv, D / scan_bv<D>()), kThr, smem, s>>>(p);
  return cudaPeekAtLastError() == cudaSuccess;
}

template <typename TIn>
bool launch_intra_d(const Params& p, int D, bool ch, cudaStream_t s) {
  if (D == 128) return ch ? launch_intra_t<TIn, 128, true>(p, s) : launch_intra_t<TIn, 128, false>(p, s);
  return ch ? launch_intra_t<TIn, 64, true>(p, s) : launch_intra_t<TIn, 64, false>(p, s);
}

}  // namespace

bool launch_gen_intra(const Params& p, int D, bool ch, bool bf16_inputs, cudaStream_t s) {
  return bf16_inputs ? launch_intra_d<__nv_bfloat16>(p, D, ch, s)
                     : launch_intra_d<float>(p, D, ch, s);
}

bool launch_gen_inter(const Params& p, int D, cudaStream_t s) {
  return D == 128 ? launch_inter_t<128>(p, s) : launch_inter_t<64>(p, s);
}

}  // namespace gdn
