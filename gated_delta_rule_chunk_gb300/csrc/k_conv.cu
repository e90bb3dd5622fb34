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
// conv_kernel: grid (token tiles of 16 rows, channel tiles of 512); a warp owns one
// 128-channel head slice, a thread 4 consecutive channels. Each warp brings its
// slice of the tile's rows and the d_conv - 1 rows before them into shared memory
// with one TMA box, keeps the causal window in registers, overwrites each row with
// its output in place and writes the 16 output rows back with one TMA store (or,
// for a tile that touches rows outside every sequence, with per-thread stores of
// the rows a sequence owns). state_kernel (launched after it, so that the new state
// may overwrite the old one): each thread reads every input of its channels' new
// state and snapshots before writing any.
#include <cuda.h>

#include "gdn_common.cuh"
#include "umma.cuh"

namespace gdn {

namespace {

constexpr int kTile = 16;     // tokens per CTA
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
__global__ void __launch_bounds__(128)
conv_kernel(const __grid_constant__ ConvParams p, const __grid_constant__ CUtensorMap tm_x,
            const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v) {
  constexpr int kRows = kTile + D - 1;  // tile rows plus the window's rows before them
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int esz = p.bf16 ? 2 : 4;
  const int c_w = blockIdx.y * 512 + 128 * warp;  // this warp's head slice
  const int c = c_w + 4 * lane;                   // first of this thread's 4 channels
  const int t0 = blockIdx.x * kTile;
  const int t1 = min(t0 + kTile, p.T);
  unsigned char* tile = smem + warp * kRows * 128 * esz;  // [kRows][128 channels]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 4 * kRows * 128 * esz) + warp;
  if (c_w >= p.C) return;  // whole warps (C is a multiple of 128)
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
    mbar_expect_tx(bar, (uint32_t)(kRows * 128 * esz));
    tma_load_2d(tile, &tm_x, c_w, t0 - (D - 1), bar);
  }
  const bool qk = c_w < 2 * p.H * kDk;  // q or k head
  float w[4][D];  // this thread's taps, loaded while the tile is in flight
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int j = 0; j < D; ++j) w[e][j] = p.w[(size_t)(c + e) * D + j];
  // the sequences owning the tile's rows (cu_seqlens reads, also while the tile is in flight)
  int n = seq_of(p, t0);
  int2 sb = n < p.N ? seq_bounds(p, n) : make_int2(p.T, p.T);
  // the TMA store may write the whole tile only if a sequence owns every row of it
  const int lo = p.cu ? min(max(p.cu[0], 0), p.T) : 0;
  const int hi = p.cu ? min(max(p.cu[p.N], 0), p.T) : p.T;
  const bool whole = t0 >= lo && t1 <= hi;
  __syncwarp();
  const bool loaded = mbar_wait(bar, 0, 1u << 22);
  if (!loaded && lane == 0) set_status(p.status, GDN_DEV_TIMEOUT);

  auto row_ptr = [&](int t) { return tile + (t - t0 + D - 1) * 128 * esz + 4 * lane * esz; };
  auto smem4 = [&](int t, float (&o)[4]) {
    const unsigned char* src = row_ptr(t);
    if (p.bf16) {
      const uint2 r = *reinterpret_cast<const uint2*>(src);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
      o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    } else {
      const float4 f = *reinterpret_cast<const float4*>(src);
      o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
    }
  };
  float win[D > 1 ? D - 1 : 1][4];  // win[j]: input at row t - (D - 1) + j
  auto fill = [&](int t) {
#pragma unroll
    for (int j = 0; j < D - 1; ++j) {
      const int r = t - (D - 1) + j;
      if (r >= sb.x) {
        smem4(r, win[j]);
      } else if (p.s_in) {
        const int i = (D - 1) - (sb.x - r);
#pragma unroll
        for (int e = 0; e < 4; ++e) win[j][e] = p.s_in[((size_t)n * p.C + c + e) * (D - 1) + i];
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) win[j][e] = 0.f;
      }
    }
  };
  const int qkc = p.H * kDk;
  // One output row: the taps in order, SiLU, the optional L2 norm of a q or k head, the
  // store (in place in the tile when the tile is stored whole), then the window slides
  // (slot D - 2 takes the current row).
  auto emit = [&](int t) {
    float cur[4], y[4];
    smem4(t, cur);
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
      const float r = rsqrtf(ss + p.eps);
#pragma unroll
      for (int e = 0; e < 4; ++e) y[e] *= r;
    }
    if (whole) {  // in place: this thread's channels of row t are no longer read
      unsigned char* dst = row_ptr(t);
      if (p.bf16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(y[2], y[3]);
        uint2 r;
        r.x = *reinterpret_cast<const uint32_t*>(&a);
        r.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(dst) = r;
      } else {
        *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
      }
    } else if (c < qkc) {
      store4(p.q, (size_t)t * qkc + c, p.bf16, y);
    } else if (c < 2 * qkc) {
      store4(p.k, (size_t)t * qkc + (c - qkc), p.bf16, y);
    } else {
      store4(p.v, (size_t)t * (p.Hv * kDv) + (c - 2 * qkc), p.bf16, y);
    }
#pragma unroll
    for (int j = 0; j < D - 1; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) win[j][e] = j + 1 < D - 1 ? win[j + 1][e] : cur[e];
  };
  if (n < p.N && t0 >= sb.x && t0 + kTile <= sb.y) {
    // the common case: one sequence owns every row of the tile (no per-row checks)
    fill(t0);
#pragma unroll 3
    for (int t = t0; t < t0 + kTile; ++t) emit(t);
  } else {
    bool stale = true;  // the window is filled at the first row of each sequence run
    for (int t = t0; t < t1; ++t) {
      if (n >= p.N) break;  // rows past the last sequence are not part of any
      if (t >= sb.y) {      // next sequence (skipping empty ones)
        while (n < p.N && seq_bounds(p, n).y <= t) ++n;
        if (n >= p.N) break;
        sb = seq_bounds(p, n);
        stale = true;
      }
      if (t < sb.x) continue;  // a row before the sequence (no sequence owns it)
      if (stale) {
        fill(t);
        stale = false;
      }
      emit(t);
    }
  }
  if (whole) {
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      const unsigned char* src = tile + (D - 1) * 128 * esz;
      if (c_w < qkc)
        tma_store_2d(&tm_q, c_w, t0, src);
      else if (c_w < 2 * qkc)
        tma_store_2d(&tm_k, c_w - qkc, t0, src);
      else
        tma_store_2d(&tm_v, c_w - 2 * qkc, t0, src);
      bulk_commit();
      bulk_wait<0>();
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

bool launch_conv_front(const ConvParams& p, cudaStream_t s) {
  const unsigned tiles = (unsigned)((p.C + 511) / 512);
  if (p.T > 0) {
    const bool bf16 = p.bf16 != 0;
    const int qkc = p.H * kDk, vc = p.Hv * kDv;
    CUtensorMap tm_x, tm_q, tm_k, tm_v;
    const int rows = kTile + p.d - 1;
    if (!encode_2d_tmap(&tm_x, p.x, bf16, p.C, p.T, 128, rows) ||
        !encode_2d_tmap(&tm_q, p.q, bf16, qkc, p.T, 128, kTile) ||
        !encode_2d_tmap(&tm_k, p.k, bf16, qkc, p.T, 128, kTile) ||
        !encode_2d_tmap(&tm_v, p.v, bf16, vc, p.T, 128, kTile))
      return false;
    const int smem = 4 * rows * 128 * (bf16 ? 2 : 4) + 4 * 8;
    const dim3 grid((unsigned)((p.T + kTile - 1) / kTile), tiles);
#define GDN_CONV_LAUNCH(D)                                                              \
  ensure_smem_limit((const void*)conv_kernel<D>, smem);                                 \
  conv_kernel<D><<<grid, 128, smem, s>>>(p, tm_x, tm_q, tm_k, tm_v);
    switch (p.d) {
      case 1: GDN_CONV_LAUNCH(1) break;
      case 2: GDN_CONV_LAUNCH(2) break;
      case 3: GDN_CONV_LAUNCH(3) break;
      case 4: GDN_CONV_LAUNCH(4) break;
      case 5: GDN_CONV_LAUNCH(5) break;
      case 6: GDN_CONV_LAUNCH(6) break;
      case 7: GDN_CONV_LAUNCH(7) break;
      default: GDN_CONV_LAUNCH(8) break;
    }
#undef GDN_CONV_LAUNCH
  }
  if (p.N > 0) state_kernel<<<dim3((unsigned)p.N, tiles), 128, 0, s>>>(p);
  return true;
}

}  // namespace gdn
