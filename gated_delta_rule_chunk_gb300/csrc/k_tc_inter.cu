// K3, bf16 inputs: fused inter-chunk scan over [sequences, value heads, dv blocks].
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", section 5: the state
// contribution, the local-attention output and the state update are fused per
// sequence and value head, walking the chunks in order with the fp32 state
// updated in place; the [sequences, Hv] domain is chosen for parallelism over
// [sequences, H]. "Chunking Qwen3.5's gated DeltaNet ... on Apple Silicon"
// (section "How do you parallelize a recurrence for prefill?"): the value
// dimension of the state tile is blocked so that it stays on chip. Here a CTA
// owns 32 value columns of one (sequence, value head): its 128x32 fp32 state
// lives in registers as the accumulators of the state-update MMA for the whole
// sequence.
//
// Per chunk (S = chunk-start state, dk x 32):
//   X     = w S_hi                          (chain; w and S_hi bf16)
//   v_new = u - X                           (fp32)
//   o     = scale (diag(exp(G)) Q (S_hi + S_lo) + (M_hi + M_lo)(vn_hi + vn_lo) - M_lo vn_lo)
//   S    <- exp(G_L) S + K^T (vh_hi + vh_lo),  vh = diag(exp(G_L - G)) v_new
// where x_hi + x_lo is a bf16 hi/lo split of an fp32 value (the lo*lo product
// is dropped). S is split after every update; the next chunk's operands are
// prefetched with cp.async while the current chunk is computed.
#include "gdn_common.cuh"
#include "warp_mma.cuh"

namespace gdn {

namespace {

constexpr int BV = 32;         // value columns of the state per CTA
constexpr int LDB = 136;       // bf16 stride of 128-wide tiles
constexpr int LDB64 = 72;      // bf16 stride of 64-wide tiles
constexpr int LDS = BV + 8;    // bf16 stride of 32-wide tiles (80 B rows)
constexpr int LDU = BV + 4;    // fp32 stride of the u tile

struct Stage {
  __nv_bfloat16 W[64 * LDB], Q[64 * LDB], K[64 * LDB];
  __nv_bfloat16 Mh[64 * LDB64], Ml[64 * LDB64];
  float U[64 * LDU];
  float G[64], QR[64], KR[64], pad[64];
};

struct InterSmem {
  Stage st[2];
  __nv_bfloat16 Sh[128 * LDS], Sl[128 * LDS];                        // [dk][BV]
  __nv_bfloat16 Vnh[64 * LDS], Vnl[64 * LDS], Vhh[64 * LDS], Vhl[64 * LDS];  // [token][BV]
};

__device__ __forceinline__ void load_chunk(Stage& st, const Params& p, int slot, int hv, int h,
                                           int c0, int t0, int L, int tid) {
  const size_t sl = (size_t)slot * p.Hv + hv;
  const __nv_bfloat16* wg = static_cast<const __nv_bfloat16*>(p.w) + sl * 64 * kDk;
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k);
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int idx = tid + it * 128;
    const int i = idx >> 4, c = (idx & 15) * 8;
    const bool ok = i < L;
    const size_t row = ((size_t)(ok ? t0 + i : t0) * p.H + h) * kDk + c;
    cp_async16(&st.W[i * LDB + c], wg + i * kDk + c, true);
    cp_async16(&st.Q[i * LDB + c], qg + row, ok);
    cp_async16(&st.K[i * LDB + c], kg + row, ok);
  }
  const __nv_bfloat16* mg = static_cast<const __nv_bfloat16*>(p.M) + sl * 2 * 64 * 64;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int idx = tid + it * 128;  // 512 chunks per 64x64 bf16 tile
    const int i = idx >> 3, c = (idx & 7) * 8;
    cp_async16(&st.Mh[i * LDB64 + c], mg + i * 64 + c, true);
    cp_async16(&st.Ml[i * LDB64 + c], mg + 64 * 64 + i * 64 + c, true);
    cp_async16(&st.U[i * LDU + (idx & 7) * 4], p.u + (sl * 64 + i) * kDv + c0 + (idx & 7) * 4,
               true);
  }
  if (tid < 16) cp_async16(&st.G[tid * 4], p.G + sl * 64 + tid * 4, true);
  if (tid >= 64) {
    const int i = tid - 64;
    const bool ok = i < L && p.qrn;
    st.QR[i] = ok ? p.qrn[(size_t)(t0 + i) * p.H + h] : 1.f;
    st.KR[i] = ok ? p.krn[(size_t)(t0 + i) * p.H + h] : 1.f;
  }
}

__global__ void __launch_bounds__(128) tc_inter_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  InterSmem& s = *reinterpret_cast<InterSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = 2 * (lane & 3);
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * BV;
  const int h = hv / p.HG;
  const SeqView sv = seq_view(p, n);
  int nch = (sv.len + kChunk - 1) / kChunk;
  if (sv.first_slot + nch > p.nt_max) {
    set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
    nch = max(0, p.nt_max - sv.first_slot);
  }
  const size_t state_base = ((size_t)n * p.Hv + hv) * kDv * kDk;

  // State rows (dk) 32*warp + 16*mt + {g, g+8}, columns 8*nt + c + {0,1}.
  float S[2][4][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 32 * warp + 16 * mt + g + (e >> 1) * 8, col = 8 * nt + c + (e & 1);
        S[mt][nt][e] = p.s0 ? p.s0[state_base + (size_t)(c0 + col) * kDk + row] : 0.f;
      }
  auto store_split_state = [&]() {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = 32 * warp + 16 * mt + g + hh * 8, col = 8 * nt + c;
          split2_store(&s.Sh[row * LDS + col], &s.Sl[row * LDS + col], S[mt][nt][2 * hh],
                       S[mt][nt][2 * hh + 1]);
        }
  };
  store_split_state();

  if (nch > 0) load_chunk(s.st[0], p, sv.first_slot, hv, h, c0, sv.start, min(kChunk, sv.len), tid);
  cp_async_commit();

  for (int ci = 0; ci < nch; ++ci) {
    const int t0 = sv.start + kChunk * ci;
    const int L = min(kChunk, sv.len - kChunk * ci);
    if (ci + 1 < nch) {
      const int t1 = t0 + kChunk;
      load_chunk(s.st[(ci + 1) & 1], p, sv.first_slot + ci + 1, hv, h, c0, t1,
                 min(kChunk, sv.len - kChunk * (ci + 1)), tid);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    Stage& st = s.st[ci & 1];
    const int r0 = 16 * warp;

    // X = w S_hi (chain) and Q S = Q (S_hi + S_lo) (output), rows r0..r0+15.
    float xa[4][4], qa[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) xa[nt][e] = qa[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t aw[4], aq[4];
      load_a(aw, st.W, LDB, r0, 16 * ks, lane);
      load_a(aq, st.Q, LDB, r0, 16 * ks, lane);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t bh[4], bl[4];
        load_b_kn(bh, s.Sh, LDS, 16 * ks, 16 * np, lane);
        load_b_kn(bl, s.Sl, LDS, 16 * ks, 16 * np, lane);
        mma_bf16(xa[2 * np], aw, bh[0], bh[1]);
        mma_bf16(xa[2 * np + 1], aw, bh[2], bh[3]);
        mma_bf16(qa[2 * np], aq, bh[0], bh[1]);
        mma_bf16(qa[2 * np + 1], aq, bh[2], bh[3]);
        mma_bf16(qa[2 * np], aq, bl[0], bl[1]);
        mma_bf16(qa[2 * np + 1], aq, bl[2], bl[3]);
      }
    }
    // v_new = u - X; vh = exp(G_L - G) v_new * krn (row factors); both split hi/lo.
    const float gl = st.G[63];
    const float fa = expf(gl - st.G[r0 + g]) * st.KR[r0 + g];
    const float fb = expf(gl - st.G[r0 + g + 8]) * st.KR[r0 + g + 8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = 8 * nt + c;
      const float v0 = st.U[(r0 + g) * LDU + col] - xa[nt][0];
      const float v1 = st.U[(r0 + g) * LDU + col + 1] - xa[nt][1];
      const float v2 = st.U[(r0 + g + 8) * LDU + col] - xa[nt][2];
      const float v3 = st.U[(r0 + g + 8) * LDU + col + 1] - xa[nt][3];
      split2_store(&s.Vnh[(r0 + g) * LDS + col], &s.Vnl[(r0 + g) * LDS + col], v0, v1);
      split2_store(&s.Vnh[(r0 + g + 8) * LDS + col], &s.Vnl[(r0 + g + 8) * LDS + col], v2, v3);
      split2_store(&s.Vhh[(r0 + g) * LDS + col], &s.Vhl[(r0 + g) * LDS + col], fa * v0, fa * v1);
      split2_store(&s.Vhh[(r0 + g + 8) * LDS + col], &s.Vhl[(r0 + g + 8) * LDS + col], fb * v2,
                   fb * v3);
    }
    __syncthreads();

    // Output rows r0..r0+15: diag(exp(G) * qrn) Q S + M v_new (M causal: k-tiles <= warp).
    {
      const float ea = expf(st.G[r0 + g]) * st.QR[r0 + g];
      const float eb = expf(st.G[r0 + g + 8]) * st.QR[r0 + g + 8];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        qa[nt][0] *= ea; qa[nt][1] *= ea; qa[nt][2] *= eb; qa[nt][3] *= eb;
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (ks <= warp) {
          uint32_t mh[4], ml[4];
          load_a(mh, st.Mh, LDB64, r0, 16 * ks, lane);
          load_a(ml, st.Ml, LDB64, r0, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t bh[4], bl[4];
            load_b_kn(bh, s.Vnh, LDS, 16 * ks, 16 * np, lane);
            load_b_kn(bl, s.Vnl, LDS, 16 * ks, 16 * np, lane);
            mma_bf16(qa[2 * np], mh, bh[0], bh[1]);
            mma_bf16(qa[2 * np + 1], mh, bh[2], bh[3]);
            mma_bf16(qa[2 * np], ml, bh[0], bh[1]);
            mma_bf16(qa[2 * np + 1], ml, bh[2], bh[3]);
            mma_bf16(qa[2 * np], mh, bl[0], bl[1]);
            mma_bf16(qa[2 * np + 1], mh, bl[2], bl[3]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = c0 + 8 * nt + c;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = r0 + g + 8 * hh;
          if (row < L) {
            const size_t oi = ((size_t)(t0 + row) * p.Hv + hv) * kDv + col;
            const float o0 = p.scale * qa[nt][2 * hh], o1 = p.scale * qa[nt][2 * hh + 1];
            if (p.out_bf16)
              *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + oi) = pack_bf16(o0, o1);
            else
              *reinterpret_cast<float2*>(static_cast<float*>(p.out) + oi) = make_float2(o0, o1);
          }
        }
      }
    }

    // S <- exp(G_L) S + K^T (vh_hi + vh_lo); this warp owns dk rows 32*warp..+31.
    {
      const float gam = expf(gl);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[mt][nt][e] *= gam;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t bh[2][4], bl[2][4];
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          load_b_kn(bh[np], s.Vhh, LDS, 16 * ks, 16 * np, lane);
          load_b_kn(bl[np], s.Vhl, LDS, 16 * ks, 16 * np, lane);
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a[4];
          load_a_trans(a, st.K, LDB, 32 * warp + 16 * mt, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            mma_bf16(S[mt][2 * np], a, bh[np][0], bh[np][1]);
            mma_bf16(S[mt][2 * np + 1], a, bh[np][2], bh[np][3]);
            mma_bf16(S[mt][2 * np], a, bl[np][0], bl[np][1]);
            mma_bf16(S[mt][2 * np + 1], a, bl[np][2], bl[np][3]);
          }
        }
      }
    }
    store_split_state();   // readers of the old split finished before the v_new barrier
    __syncthreads();       // stage ci&1 and the v_new tiles are reused next
  }
  cp_async_wait<0>();

  if (p.sT) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = 32 * warp + 16 * mt + g + (e >> 1) * 8, col = 8 * nt + c + (e & 1);
          p.sT[state_base + (size_t)(c0 + col) * kDk + row] = S[mt][nt][e];
        }
  }
}

}  // namespace

void launch_tc_inter(const Params& p, cudaStream_t s) {
  const int smem = (int)sizeof(InterSmem);
  ensure_smem_limit((const void*)tc_inter_kernel, smem);
  tc_inter_kernel<<<dim3(p.N, p.Hv, kDv / BV), 128, smem, s>>>(p);
}

}  // namespace gdn
