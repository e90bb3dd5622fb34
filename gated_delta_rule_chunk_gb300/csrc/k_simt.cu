// fp32 SIMT path (used for fp32 inputs): the same intra/inter decomposition
// as the tensor-core path, in plain fp32 FMA arithmetic, so that fp32 inputs
// are computed without any reduced-precision operand.
//
// Intra (grid [nt_max, H]), following "Optimizing GDN Chunk Prefill on Intel
// AMX CPU" section 4 (K K^T once per key head, then per value head of the
// group: decay/beta scaling, triangular solve, w and u):
//   G_i  = sum_{j<=i} g_j                          (in-chunk cumulative log-decay)
//   A_ij = beta_i exp(G_i - G_j) k_i.k_j  (j < i)   T = (I + A)^-1
//   w    = T diag(beta exp(G)) K,   u = T diag(beta) V
//   M_ij = exp(G_i - G_j) q_i.k_j  (j <= i)         (causal decay-masked q.k)
// Inter (grid [N, Hv, dv/32]), section 5 of the same note (state output and
// state update fused per sequence and value head; fp32 state updated in place):
//   v_new = u - w S
//   o     = scale (diag(exp(G)) Q S + M v_new)
//   S    <- exp(G_L) S + (diag(exp(G_L - G)) K)^T v_new
// with the plus sign of (I + A) fixed by unrolling the per-token recurrence.
#include "gdn_common.cuh"
#include "tri_inverse.cuh"

namespace gdn {

namespace {

constexpr int kLd = 129;   // padded fp32 row stride of 128-wide tiles
constexpr int kLd64 = 65;  // padded fp32 row stride of 64-wide tiles

template <typename TIn>
__device__ __forceinline__ float load_in(const void* base, size_t idx) {
  return to_f32(reinterpret_cast<const TIn*>(base)[idx]);
}

// Resolve the chunk of this slot; returns false (after flagging) if the CTA has nothing to do.
__device__ __forceinline__ bool resolve_chunk(const Params& p, int slot, int& n, int& t0,
                                              int& L, int& wslot) {
  const int2 e = p.chunk_table[slot];
  if (e.x < 0) return false;  // sentinel slot: early exit
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
  n = e.x;
  t0 = sv.start + kChunk * e.y;
  L = min(kChunk, sv.len - kChunk * e.y);
  return true;
}

template <typename TIn>
__global__ void __launch_bounds__(256) simt_intra_kernel(Params p) {
  extern __shared__ float sm[];
  float* Ks = sm;                     // [64][129]
  float* Qs = Ks + 64 * kLd;          // [64][129]
  float* Vs = Qs + 64 * kLd;          // [64][129]
  float* KK = Vs + 64 * kLd;          // [64][65]
  float* QK = KK + 64 * kLd64;        // [64][65]
  float* A = QK + 64 * kLd64;         // [64][65]
  float* Tm = A + 64 * kLd64;         // [64][65]
  float* X = Tm + 64 * kLd64;         // [16][65] scratch of the inverse
  float* Gs = X + 16 * kLd64;         // [64]
  float* Bs = Gs + 64;                // [64]
  float* Es = Bs + 64;                // [64]

  const int tid = threadIdx.x, h = blockIdx.y;
  int n, t0, L, wslot;
  if (!resolve_chunk(p, blockIdx.x, n, t0, L, wslot)) return;

  for (int idx = tid; idx < 64 * 128; idx += 256) {
    const int i = idx >> 7, d = idx & 127;
    float kv = 0.f, qv = 0.f;
    if (i < L) {
      const size_t row = (size_t)(t0 + i) * p.H + h;
      kv = load_in<TIn>(p.k, row * kDk + d);
      qv = load_in<TIn>(p.q, row * kDk + d);
      if (p.krn) {
        kv *= p.krn[row];
        qv *= p.qrn[row];
      }
    }
    Ks[i * kLd + d] = kv;
    Qs[i * kLd + d] = qv;
  }
  __syncthreads();
  for (int idx = tid; idx < 64 * 64; idx += 256) {
    const int i = idx >> 6, j = idx & 63;
    float kk = 0.f, qk = 0.f;
    if (j <= i) {
      for (int d = 0; d < kDk; ++d) {
        kk = fmaf(Ks[i * kLd + d], Ks[j * kLd + d], kk);
        qk = fmaf(Qs[i * kLd + d], Ks[j * kLd + d], qk);
      }
    }
    KK[i * kLd64 + j] = kk;
    QK[i * kLd64 + j] = qk;
  }
  __syncthreads();

  for (int r = 0; r < p.HG; ++r) {
    const int hv = h * p.HG + r;
    const size_t sl = (size_t)wslot * p.Hv + hv;
    if (tid < 64) {
      const bool ok = tid < L;
      Gs[tid] = ok ? p.g[(size_t)(t0 + tid) * p.Hv + hv] : 0.f;
      Bs[tid] = ok ? p.beta[(size_t)(t0 + tid) * p.Hv + hv] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // inclusive in-chunk cumsum, left to right
      float acc = 0.f;
      for (int i = 0; i < 64; ++i) {
        acc += Gs[i];
        Gs[i] = acc;
      }
    }
    __syncthreads();
    if (tid < 64) {
      Es[tid] = expf(Gs[tid]);
      p.G[sl * 64 + tid] = Gs[tid];
    }
    float* Mo = reinterpret_cast<float*>(p.M) + sl * 64 * 64;
    for (int idx = tid; idx < 64 * 64; idx += 256) {
      const int i = idx >> 6, j = idx & 63;
      const float dec = (j <= i) ? expf(Gs[i] - Gs[j]) : 0.f;
      A[i * kLd64 + j] = (j < i) ? Bs[i] * dec * KK[i * kLd64 + j] : 0.f;
      Mo[idx] = dec * QK[i * kLd64 + j];
    }
    for (int idx = tid; idx < 64 * 128; idx += 256) {
      const int i = idx >> 7, d = idx & 127;
      Vs[i * kLd + d] = (i < L) ? load_in<TIn>(p.v, ((size_t)(t0 + i) * p.Hv + hv) * kDv + d) : 0.f;
    }
    __syncthreads();
    tri_inverse_64(A, kLd64, Tm, kLd64, X, tid, 256);
    __syncthreads();
    float* wo = reinterpret_cast<float*>(p.w) + sl * 64 * kDk;
    float* uo = p.u + sl * 64 * kDv;
    for (int idx = tid; idx < 64 * 128; idx += 256) {
      const int i = idx >> 7, d = idx & 127;
      float wa = 0.f, ua = 0.f;
      for (int j = 0; j <= i; ++j) {
        const float t = Tm[i * kLd64 + j] * Bs[j];
        wa = fmaf(t * Es[j], Ks[j * kLd + d], wa);
        ua = fmaf(t, Vs[j * kLd + d], ua);
      }
      wo[idx] = wa;
      uo[idx] = ua;
    }
    __syncthreads();
  }
}

constexpr int kBV = 32;  // value columns of the state per inter CTA

template <typename TIn>
__global__ void __launch_bounds__(256) simt_inter_kernel(Params p) {
  extern __shared__ float sm[];
  float* S = sm;                      // [128][33]  dk x BV
  float* Ws = S + 128 * 33;           // [64][129]
  float* Qs = Ws + 64 * kLd;          // [64][129]
  float* Ks = Qs + 64 * kLd;          // [64][129]
  float* Ms = Ks + 64 * kLd;          // [64][65]
  float* Un = Ms + 64 * kLd64;        // [64][33]  u, then v_new
  float* Gs = Un + 64 * 33;           // [64]

  const int tid = threadIdx.x;
  const int n = blockIdx.x, hv = blockIdx.y, c0 = blockIdx.z * kBV;
  const int h = hv / p.HG;
  const SeqView sv = seq_view(p, n);
  const int nch = (sv.len + kChunk - 1) / kChunk;
  const size_t state_base = ((size_t)n * p.Hv + hv) * kDv * kDk;

  for (int idx = tid; idx < 128 * kBV; idx += 256) {
    const int d = idx / kBV, j = idx % kBV;
    S[d * 33 + j] = p.s0 ? p.s0[state_base + (size_t)(c0 + j) * kDk + d] : 0.f;
  }
  __syncthreads();

  for (int c = 0; c < nch; ++c) {
    const int slot = sv.first_slot + c;
    if (slot >= p.nt_max) {
      set_status(p.status, GDN_DEV_CHUNK_OVERFLOW);
      break;
    }
    const int t0 = sv.start + kChunk * c;
    const int L = min(kChunk, sv.len - kChunk * c);
    const size_t sl = (size_t)slot * p.Hv + hv;
    const float* wi = reinterpret_cast<const float*>(p.w) + sl * 64 * kDk;
    const float* Mi = reinterpret_cast<const float*>(p.M) + sl * 64 * 64;
    for (int idx = tid; idx < 64 * 128; idx += 256) {
      const int i = idx >> 7, d = idx & 127;
      float qv = 0.f, kv = 0.f;
      if (i < L) {
        const size_t row = (size_t)(t0 + i) * p.H + h;
        qv = load_in<TIn>(p.q, row * kDk + d);
        kv = load_in<TIn>(p.k, row * kDk + d);
        if (p.krn) {
          qv *= p.qrn[row];
          kv *= p.krn[row];
        }
      }
      Ws[i * kLd + d] = wi[idx];
      Qs[i * kLd + d] = qv;
      Ks[i * kLd + d] = kv;
    }
    for (int idx = tid; idx < 64 * 64; idx += 256) Ms[(idx >> 6) * kLd64 + (idx & 63)] = Mi[idx];
    for (int idx = tid; idx < 64 * kBV; idx += 256) {
      const int i = idx / kBV, j = idx % kBV;
      Un[i * 33 + j] = p.u[(sl * 64 + i) * kDv + c0 + j];
    }
    if (tid < 64) Gs[tid] = p.G[sl * 64 + tid];
    __syncthreads();
    // v_new = u - w S (in place over u)
    for (int idx = tid; idx < 64 * kBV; idx += 256) {
      const int i = idx / kBV, j = idx % kBV;
      float x = 0.f;
      for (int d = 0; d < kDk; ++d) x = fmaf(Ws[i * kLd + d], S[d * 33 + j], x);
      Un[i * 33 + j] -= x;
    }
    __syncthreads();
    // o = scale (exp(G) Q S + M v_new), rows past the sequence end are not stored
    for (int idx = tid; idx < 64 * kBV; idx += 256) {
      const int i = idx / kBV, j = idx % kBV;
      if (i >= L) continue;
      float a = 0.f, b = 0.f;
      for (int d = 0; d < kDk; ++d) a = fmaf(Qs[i * kLd + d], S[d * 33 + j], a);
      for (int m = 0; m <= i; ++m) b = fmaf(Ms[i * kLd64 + m], Un[m * 33 + j], b);
      const float o = p.scale * (expf(Gs[i]) * a + b);
      const size_t oi = ((size_t)(t0 + i) * p.Hv + hv) * kDv + c0 + j;
      if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(o);
      else
        reinterpret_cast<float*>(p.out)[oi] = o;
    }
    __syncthreads();
    // S <- exp(G_L) S + (diag(exp(G_L - G)) K)^T v_new; G is flat past the last valid row
    const float gl = Gs[63];
    for (int idx = tid; idx < 128 * kBV; idx += 256) {
      const int d = idx / kBV, j = idx % kBV;
      float acc = 0.f;
      for (int i = 0; i < 64; ++i) acc = fmaf(Ks[i * kLd + d] * expf(gl - Gs[i]), Un[i * 33 + j], acc);
      S[d * 33 + j] = fmaf(expf(gl), S[d * 33 + j], acc);
    }
    __syncthreads();
  }
  if (p.sT)
    for (int idx = tid; idx < 128 * kBV; idx += 256) {
      const int d = idx / kBV, j = idx % kBV;
      p.sT[state_base + (size_t)(c0 + j) * kDk + d] = S[d * 33 + j];
    }
}

constexpr size_t kIntraSmem = sizeof(float) * (3 * 64 * kLd + 4 * 64 * kLd64 + 16 * kLd64 + 3 * 64);
constexpr size_t kInterSmem = sizeof(float) * (128 * 33 + 3 * 64 * kLd + 64 * kLd64 + 64 * 33 + 64);

template <typename TIn>
void launch_intra_t(const Params& p, cudaStream_t s) {
  ensure_smem_limit((const void*)simt_intra_kernel<TIn>, (int)kIntraSmem);
  simt_intra_kernel<TIn><<<dim3(p.nt_max, p.H), 256, kIntraSmem, s>>>(p);
}

template <typename TIn>
void launch_inter_t(const Params& p, cudaStream_t s) {
  ensure_smem_limit((const void*)simt_inter_kernel<TIn>, (int)kInterSmem);
  simt_inter_kernel<TIn><<<dim3(p.N, p.Hv, kDv / kBV), 256, kInterSmem, s>>>(p);
}

}  // namespace

void launch_simt_intra(const Params& p, bool bf16_inputs, cudaStream_t s) {
  if (bf16_inputs) launch_intra_t<__nv_bfloat16>(p, s); else launch_intra_t<float>(p, s);
}

void launch_simt_inter(const Params& p, bool bf16_inputs, cudaStream_t s) {
  if (bf16_inputs) launch_inter_t<__nv_bfloat16>(p, s); else launch_inter_t<float>(p, s);
}

}  // namespace gdn
