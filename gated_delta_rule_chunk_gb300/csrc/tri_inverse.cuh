// Inverse of a 64x64 unit lower-triangular matrix I + A in shared memory, fp32.
//
// "Optimizing GDN Chunk Prefill on Intel AMX CPU", sections 4 and 8: the
// triangular solve of the intra stage stays triangular. Blocked forward
// substitution with 16x16 blocks: the four diagonal blocks are inverted
// column by column in parallel, then block row a = 1..3 is
//   T[a, 0:a] = -T[a, a] * (A[a, 0:a] * T[0:a, 0:a]),
// which only needs block rows < a (already final).
#pragma once

namespace gdn {

// A: strictly lower triangular part (row stride lda; entries on and above the
// diagonal are ignored). Tm: output (row stride ldt), fully written (zeros above
// the diagonal). X: scratch of 16 rows x 64 (row stride ldt). All threads of
// the block call this with the same nthr; it ends with the block synchronized.
__device__ inline void tri_inverse_64(const float* A, int lda, float* Tm, int ldt, float* X,
                                      int tid, int nthr) {
  for (int idx = tid; idx < 64 * 64; idx += nthr) Tm[(idx >> 6) * ldt + (idx & 63)] = 0.f;
  __syncthreads();
  if (tid < 64) {  // diagonal blocks, one thread per (block, column)
    const int base = (tid >> 4) * 16, c = tid & 15;
    float col[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (m < i) acc = fmaf(A[(base + i) * lda + base + m], col[m], acc);
      col[i] = (i < c) ? 0.f : (i == c ? 1.f : -acc);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Tm[(base + i) * ldt + base + c] = col[i];
  }
  __syncthreads();
  for (int a = 1; a < 4; ++a) {
    const int r0 = 16 * a, w = 16 * a;
    for (int idx = tid; idx < 16 * w; idx += nthr) {
      const int i = idx / w, j = idx % w;
      float acc = 0.f;
      for (int m = j; m < w; ++m) acc = fmaf(A[(r0 + i) * lda + m], Tm[m * ldt + j], acc);
      X[i * ldt + j] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < 16 * w; idx += nthr) {
      const int i = idx / w, j = idx % w;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m) acc = fmaf(Tm[(r0 + i) * ldt + r0 + m], X[m * ldt + j], acc);
      Tm[(r0 + i) * ldt + j] = -acc;
    }
    __syncthreads();
  }
}

}  // namespace gdn

namespace gdn {

// In-place variant: AT holds A (strictly lower part, zeros on and above the
// diagonal) on entry and T = (I + A)^-1 on exit (row stride ld). Each block row
// of A is consumed (into the scratch X) before T overwrites it. X: 16 rows x
// ld scratch. Ends with the block synchronized.
__device__ inline void tri_inverse_64_inplace(float* AT, int ld, float* X, int tid, int nthr) {
  float col[16];
  const int base = (tid >> 4) * 16, c = tid & 15;
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (m < i) acc = fmaf(AT[(base + i) * ld + base + m], col[m], acc);
      col[i] = (i < c) ? 0.f : (i == c ? 1.f : -acc);
    }
  }
  __syncthreads();  // every diagonal block of A has been read
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) AT[(base + i) * ld + base + c] = col[i];
  }
  __syncthreads();
  for (int a = 1; a < 4; ++a) {
    const int r0 = 16 * a, w = 16 * a;
    for (int idx = tid; idx < 16 * w; idx += nthr) {
      const int i = idx / w, j = idx % w;
      float acc = 0.f;
      for (int m = j; m < w; ++m) acc = fmaf(AT[(r0 + i) * ld + m], AT[m * ld + j], acc);
      X[i * ld + j] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < 16 * w; idx += nthr) {
      const int i = idx / w, j = idx % w;
      float acc = 0.f;
      for (int m = 0; m <= i; ++m) acc = fmaf(AT[(r0 + i) * ld + r0 + m], X[m * ld + j], acc);
      AT[(r0 + i) * ld + j] = -acc;
    }
    __syncthreads();
  }
}

}  // namespace gdn

#include "warp_mma.cuh"

namespace gdn {

// Split A fragment (16 x 16 at (r0, c0)) of a row-major fp32 tile with stride ld.
__device__ __forceinline__ void frag_a_split(const float* base, int ld, int r0, int c0, int lane,
                                             uint32_t (&hi)[4], uint32_t (&lo)[4]) {
  const int g = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 v = *reinterpret_cast<const float2*>(
        &base[(r0 + g + 8 * (q & 1)) * ld + c0 + c + 8 * (q >> 1)]);
    split_pack2(v.x, v.y, hi[q], lo[q]);
  }
}

// Split B fragment (16 k x 8 n at (k0, n0)) of a row-major [k][n] fp32 tile.
__device__ __forceinline__ void frag_b_split(const float* base, int ld, int k0, int n0, int lane,
                                             uint32_t (&hi)[2], uint32_t (&lo)[2]) {
  const int g = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float x0 = base[(k0 + c + 8 * q) * ld + n0 + g];
    const float x1 = base[(k0 + c + 8 * q + 1) * ld + n0 + g];
    split_pack2(x0, x1, hi[q], lo[q]);
  }
}

// D += A * B with both operands split into bf16 hi/lo (the lo*lo product dropped).
__device__ __forceinline__ void mma_split3(float (&d)[4], const uint32_t (&ah)[4],
                                           const uint32_t (&al)[4], const uint32_t (&bh)[2],
                                           const uint32_t (&bl)[2]) {
  mma_bf16(d, ah, bh[0], bh[1]);
  mma_bf16(d, ah, bl[0], bl[1]);
  mma_bf16(d, al, bh[0], bh[1]);
}

// In-place inverse of I + A (64 x 64, A strictly lower triangular with zeros on and
// above the diagonal) for a CTA of 32 * kWarps threads (kWarps >= 2). The four
// diagonal 16 x 16 blocks are inverted column by column (SIMT, fp32); block row
// a = 1..3 then needs two small
// products, X = A[a, 0:a] T[0:a, 0:a] and T[a, 0:a] = -T[a, a] X, done on warp-level
// tensor-core MMAs with the fp32 operands split into bf16 hi + lo (about 16
// significant bits, fp32 accumulate). X: 16 rows x ld scratch.
template <int kWarps = 4>
__device__ inline void tri_inverse_64_tc(float* AT, int ld, float* X, int tid) {
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = 2 * (lane & 3);
  float col[16];
  const int base = (tid >> 4) * 16, cc = tid & 15;
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (m < i) acc = fmaf(AT[(base + i) * ld + base + m], col[m], acc);
      col[i] = (i < cc) ? 0.f : (i == cc ? 1.f : -acc);
    }
  }
  __syncthreads();  // every diagonal block of A has been read
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) AT[(base + i) * ld + base + cc] = col[i];
  }
  __syncthreads();
#pragma unroll
  for (int a = 1; a < 4; ++a) {
    const int r0 = 16 * a;
    for (int nt = warp; nt < 2 * a; nt += kWarps) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < a; ++ks) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        frag_a_split(AT, ld, r0, 16 * ks, lane, ah, al);
        frag_b_split(AT, ld, 16 * ks, 8 * nt, lane, bh, bl);
        mma_split3(acc, ah, al, bh, bl);
      }
      *reinterpret_cast<float2*>(&X[g * ld + 8 * nt + c]) = make_float2(acc[0], acc[1]);
      *reinterpret_cast<float2*>(&X[(g + 8) * ld + 8 * nt + c]) = make_float2(acc[2], acc[3]);
    }
    __syncthreads();
    for (int nt = warp; nt < 2 * a; nt += kWarps) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t ah[4], al[4], bh[2], bl[2];
      frag_a_split(AT, ld, r0, r0, lane, ah, al);
      frag_b_split(X, ld, 0, 8 * nt, lane, bh, bl);
      mma_split3(acc, ah, al, bh, bl);
      *reinterpret_cast<float2*>(&AT[(r0 + g) * ld + 8 * nt + c]) = make_float2(-acc[0], -acc[1]);
      *reinterpret_cast<float2*>(&AT[(r0 + g + 8) * ld + 8 * nt + c]) = make_float2(-acc[2], -acc[3]);
    }
    __syncthreads();
  }
}

}  // namespace gdn

namespace gdn {

// In-place inverse of I + A (64 x 64, A strictly lower triangular with zeros on and above
// the diagonal) for a CTA of 8 warps, by recursive doubling: the four diagonal 16 x 16
// blocks by column substitution (fp32, one thread per column); then the two 32 x 32
// diagonal blocks, T = [[T11, 0], [-T22 A21 T11, T22]] with 16 x 16 parts (both at once);
// then the whole 64 x 64 the same way with 32 x 32 parts. Four dependent products in
// place of the six of the block-row order, with all eight warps busy in the last level.
// The products run on warp-level MMAs with fp32 operands split into bf16 hi + lo (about
// 16 significant bits, fp32 accumulate). X: scratch of 32 rows x ldx fp32 (ldx >= 32).
__device__ inline void tri_inverse_64_rd(float* AT, int ld, float* X, int ldx, int tid) {
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = 2 * (lane & 3);
  float col[16];
  const int base = (tid >> 4) * 16, cc = tid & 15;
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        if (m < i) acc = fmaf(AT[(base + i) * ld + base + m], col[m], acc);
      col[i] = (i < cc) ? 0.f : (i == cc ? 1.f : -acc);
    }
  }
  __syncthreads();  // every diagonal block of A has been read
  if (tid < 64) {
#pragma unroll
    for (int i = 0; i < 16; ++i) AT[(base + i) * ld + base + cc] = col[i];
  }
  __syncthreads();
  // Level 1: blocks (1, 0) and (3, 2). Warp w < 4: pair q = w / 2 (rows r, columns o),
  // n-tile w % 2. Y = A[r, o] T[o, o] into X columns 16 q..; then T[r, o] = -T[r, r] Y.
  const int q = warp >> 1, n1 = warp & 1;
  const int r1 = 16 + 32 * q, o1 = 32 * q;
  if (warp < 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t ah[4], al[4], bh[2], bl[2];
    frag_a_split(AT, ld, r1, o1, lane, ah, al);
    frag_b_split(AT, ld, o1, o1 + 8 * n1, lane, bh, bl);
    mma_split3(acc, ah, al, bh, bl);
    *reinterpret_cast<float2*>(&X[g * ldx + 16 * q + 8 * n1 + c]) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(&X[(g + 8) * ldx + 16 * q + 8 * n1 + c]) =
        make_float2(acc[2], acc[3]);
  }
  __syncthreads();
  if (warp < 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t ah[4], al[4], bh[2], bl[2];
    frag_a_split(AT, ld, r1, r1, lane, ah, al);
    frag_b_split(X, ldx, 0, 16 * q + 8 * n1, lane, bh, bl);
    mma_split3(acc, ah, al, bh, bl);
    *reinterpret_cast<float2*>(&AT[(r1 + g) * ld + o1 + 8 * n1 + c]) = make_float2(-acc[0], -acc[1]);
    *reinterpret_cast<float2*>(&AT[(r1 + g + 8) * ld + o1 + 8 * n1 + c]) =
        make_float2(-acc[2], -acc[3]);
  }
  __syncthreads();
  // Level 2: rows 32..63, columns 0..31. Warp w: row tile m2 = w / 4 (16 rows), n-tile
  // w % 4. Y = A21 T11 (T11[0:16, 16:32] is zero, so column tiles 2, 3 skip k-step 0)
  // into X rows 16 m2..; then T21 = -T22 Y (T22[0:16, 16:32] is zero, so row tile 0 skips
  // k-step 1).
  const int m2 = warp >> 2, n2 = warp & 3;
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      if (ks == 0 && n2 >= 2) continue;
      uint32_t ah[4], al[4], bh[2], bl[2];
      frag_a_split(AT, ld, 32 + 16 * m2, 16 * ks, lane, ah, al);
      frag_b_split(AT, ld, 16 * ks, 8 * n2, lane, bh, bl);
      mma_split3(acc, ah, al, bh, bl);
    }
    *reinterpret_cast<float2*>(&X[(16 * m2 + g) * ldx + 8 * n2 + c]) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(&X[(16 * m2 + g + 8) * ldx + 8 * n2 + c]) =
        make_float2(acc[2], acc[3]);
  }
  __syncthreads();
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      if (ks == 1 && m2 == 0) continue;
      uint32_t ah[4], al[4], bh[2], bl[2];
      frag_a_split(AT, ld, 32 + 16 * m2, 32 + 16 * ks, lane, ah, al);
      frag_b_split(X, ldx, 16 * ks, 8 * n2, lane, bh, bl);
      mma_split3(acc, ah, al, bh, bl);
    }
    *reinterpret_cast<float2*>(&AT[(32 + 16 * m2 + g) * ld + 8 * n2 + c]) =
        make_float2(-acc[0], -acc[1]);
    *reinterpret_cast<float2*>(&AT[(32 + 16 * m2 + g + 8) * ld + 8 * n2 + c]) =
        make_float2(-acc[2], -acc[3]);
  }
  __syncthreads();
}

}  // namespace gdn
