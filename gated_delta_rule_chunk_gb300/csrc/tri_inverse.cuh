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
