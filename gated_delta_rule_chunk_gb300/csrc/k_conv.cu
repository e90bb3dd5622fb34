// Front end: qkv projection output -> q, k, v.
//
// The llama.cpp page (PrismML-Eng/llama.cpp pull 399, "What", item 1, and "How
// (exactness)"): a causal depthwise convolution of width d_conv over each channel
// of the projection output, whose inputs are the d_conv - 1 inputs saved from
// before the sequence (the conv state) followed by the sequence's rows, summed
// in tap order (sum += w[j] * xx[t + j], j = 0 .. d_conv - 1, no bias), then SiLU,
// then the per-head L2 norm of q and k (x / sqrt(sum x^2 + eps), one warp per
// head and token). The new conv state is the last d_conv - 1 inputs of each
// sequence; snapshot s, for rolling a speculative batch back, is the state after
// the sequence's token s.
//
// Channel order of the projection output: q (H x dk), k (H x dk), v (Hv x dv).
//
// conv_kernel: grid (token tiles of 32, channel tiles of 512); a thread owns 4
// consecutive channels (one 8- or 16-byte load per token), a warp one 128-channel
// head, and keeps the causal window in registers across the tile's tokens.
// state_kernel (launched after it, so that the new state may overwrite the old
// one): each thread reads every input of its channels' new state and snapshots
// before writing any.
#include "gdn_common.cuh"

namespace gdn {

namespace {

constexpr int kTile = 32;     // tokens per CTA
constexpr int kMaxConv = 8;   // d_conv <= 8

__device__ __forceinline__ void load4(const void* x, size_t idx, bool bf16, float (&o)[4]) {
  if (bf16) {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + idx);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  } else {
    const float4 f = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx);
    o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
  }
}

__device__ __forceinline__ void store4(void* y, size_t idx, bool bf16, const float (&o)[4]) {
  if (bf16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(o[2], o[3]);
    uint2 r;
    r.x = *reinterpret_cast<const uint32_t*>(&a);
    r.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + idx) = r;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(y) + idx) = make_float4(o[0], o[1], o[2], o[3]);
  }
}

// Clamped bounds of sequence n (status bit for a malformed cu_seqlens).
__device__ __forceinline__ int2 seq_bounds(const ConvParams& p, int n) {
  if (!p.cu) return make_int2(0, p.T);
  const int a = p.cu[n], b = p.cu[n + 1];
  const int ac = min(max(a, 0), p.T), bc = min(max(b, 0), p.T);
  return make_int2(ac, max(bc, ac));
}

// Sequence containing row t (the first n with end > t), or N if none.
__device__ __forceinline__ int seq_of(const ConvParams& p, int t) {
  if (!p.cu) return t < p.T ? 0 : 1;
  int lo = 0, hi = p.N;  // invariant: answer in [lo, hi]
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (seq_bounds(p, mid).y > t) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Input of channel c at row p of sequence n (rows before the start come from the state).
__device__ __forceinline__ void input4(const ConvParams& p, int n, int start, int row, int c,
                                       float (&o)[4]) {
  if (row >= start) {
    load4(p.x, (size_t)row * p.C + c, p.bf16, o);
  } else if (p.s_in) {
    const int i = (p.d - 1) - (start - row);  // state entry (0 = oldest)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = p.s_in[((size_t)n * p.C + c + e) * (p.d - 1) + i];
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = 0.f;
  }
}

// D = d_conv as a compile-time constant: the tap loop and the window shift unroll
// without predicates (the kernel is instruction-bound otherwise).
template <int D>
__global__ void __launch_bounds__(128) conv_kernel(ConvParams p) {
  const int tid = threadIdx.x;
  const int c = blockIdx.y * 512 + 4 * tid;  // first of this thread's 4 channels
  if (c >= p.C) return;
  const int t0 = blockIdx.x * kTile;
  const int t1 = min(t0 + kTile, p.T);
  const bool qk = c < 2 * p.H * kDk;  // q or k channels (whole warps: heads are 128 wide)
  float w[4][D];
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int j = 0; j < D; ++j) w[e][j] = p.w[(size_t)(c + e) * D + j];

  int n = seq_of(p, t0);
  int2 sb = n < p.N ? seq_bounds(p, n) : make_int2(p.T, p.T);
  float win[D > 1 ? D - 1 : 1][4];  // win[j]: input at row t - (D - 1) + j
  auto fill = [&](int t) {
#pragma unroll
    for (int j = 0; j < D - 1; ++j) input4(p, n, sb.x, t - (D - 1) + j, c, win[j]);
  };
  bool stale = true;  // the window is filled at the first row of each sequence run
  constexpr int G = 8;  // rows loaded together (memory-level parallelism)
  for (int tb = t0; tb < t1; tb += G) {
    float rowv[G][4];
#pragma unroll
    for (int u = 0; u < G; ++u)
      if (tb + u < t1) load4(p.x, (size_t)(tb + u) * p.C + c, p.bf16, rowv[u]);
#pragma unroll
    for (int u = 0; u < G; ++u) {
      const int t = tb + u;
      if (t >= t1 || n >= p.N) break;  // rows past the last sequence are not part of any
      if (t >= sb.y) {                  // next sequence (skipping empty ones)
        while (n < p.N && seq_bounds(p, n).y <= t) ++n;
        if (n >= p.N) break;
        sb = seq_bounds(p, n);
        stale = true;
      }
      if (t < sb.x) continue;           // a row before the sequence (no sequence owns it)
      if (stale) {
        fill(t);
        stale = false;
      }
      const float (&cur)[4] = rowv[u];
      float y[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float acc = 0.f;  // taps in order j = 0 .. D - 1 (the current row is tap D - 1)
#pragma unroll
        for (int j = 0; j < D - 1; ++j) acc = fmaf(w[e][j], win[j][e], acc);
        acc = fmaf(w[e][D - 1], cur[e], acc);
        y[e] = __fdividef(acc, 1.f + __expf(-acc));  // SiLU
      }
      if (p.l2norm && qk) {
        float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = 1.f / sqrtf(ss + p.eps);
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] *= r;
      }
      // q [T,H,dk], k [T,H,dk], v [T,Hv,dv]: channel c is element c of row t of q, then k, v
      const int qkc = p.H * kDk;
      if (c < qkc)
        store4(p.q, (size_t)t * qkc + c, p.bf16, y);
      else if (c < 2 * qkc)
        store4(p.k, (size_t)t * qkc + (c - qkc), p.bf16, y);
      else
        store4(p.v, (size_t)t * (p.Hv * kDv) + (c - 2 * qkc), p.bf16, y);
      // slide the window (slot D - 2 takes the current row)
#pragma unroll
      for (int j = 0; j < D - 1; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) win[j][e] = j + 1 < D - 1 ? win[j + 1][e] : cur[e];
    }
  }
}

// New conv state and snapshots of sequence blockIdx.x for channels 4 tid .. of tile blockIdx.y.
__global__ void __launch_bounds__(128) state_kernel(ConvParams p) {
  const int n = blockIdx.x;
  const int c = blockIdx.y * 512 + 4 * threadIdx.x;
  if (p.cu && threadIdx.x == 0 && blockIdx.y == 0) {
    const int a = p.cu[n], b = p.cu[n + 1];
    if (a < 0 || b > p.T || b < a) set_status(p.status, GDN_DEV_BAD_CU_SEQLENS);
  }
  if (c >= p.C || p.d < 2) return;
  const int2 sb = seq_bounds(p, n);
  const int L = sb.y - sb.x;
  const int dm = p.d - 1;
  // xx[i] = state entry i for i < d - 1, else x[start + i - (d - 1)]
  auto xx = [&](int i, float (&o)[4]) { input4(p, n, sb.x, sb.x + i - dm, c, o); };
  float fin[kMaxConv - 1][4];
#pragma unroll
  for (int i = 0; i < kMaxConv - 1; ++i)
    if (i < dm) xx(L + i, fin[i]);
  // snapshots (which must not alias the input state), then the new state, whose
  // inputs were all read above
  if (p.snaps) {
    for (int s = 0; s < p.n_snap; ++s) {
      const int e = L > 0 ? min(s, L - 1) + 1 : 0;
      float v[kMaxConv - 1][4];
#pragma unroll
      for (int i = 0; i < kMaxConv - 1; ++i)
        if (i < dm) xx(e + i, v[i]);
#pragma unroll
      for (int i = 0; i < kMaxConv - 1; ++i)
        if (i < dm) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            p.snaps[(((size_t)n * p.n_snap + s) * p.C + c + q) * dm + i] = v[i][q];
        }
    }
  }
  if (p.s_out) {
#pragma unroll
    for (int i = 0; i < kMaxConv - 1; ++i)
      if (i < dm) {
#pragma unroll
        for (int q = 0; q < 4; ++q) p.s_out[((size_t)n * p.C + c + q) * dm + i] = fin[i][q];
      }
  }
}

}  // namespace

void launch_conv_front(const ConvParams& p, cudaStream_t s) {
  const dim3 tiles((unsigned)((p.C + 511) / 512));
  if (p.T > 0) {
    const dim3 grid((unsigned)((p.T + kTile - 1) / kTile), tiles.x);
    switch (p.d) {
      case 1: conv_kernel<1><<<grid, 128, 0, s>>>(p); break;
      case 2: conv_kernel<2><<<grid, 128, 0, s>>>(p); break;
      case 3: conv_kernel<3><<<grid, 128, 0, s>>>(p); break;
      case 4: conv_kernel<4><<<grid, 128, 0, s>>>(p); break;
      case 5: conv_kernel<5><<<grid, 128, 0, s>>>(p); break;
      case 6: conv_kernel<6><<<grid, 128, 0, s>>>(p); break;
      case 7: conv_kernel<7><<<grid, 128, 0, s>>>(p); break;
      default: conv_kernel<8><<<grid, 128, 0, s>>>(p); break;
    }
  }
  if (p.N > 0) state_kernel<<<dim3((unsigned)p.N, tiles.x), 128, 0, s>>>(p);
}

}  // namespace gdn
