// Warp-level bf16 MMA (m16n8k16, fp32 accumulate), ldmatrix and cp.async
// helpers, written from the PTX ISA's fragment definitions.
//
// Fragment ownership for mma.m16n8k16 (lane = threadIdx.x % 32, g = lane / 4,
// c = 2 * (lane % 4)):
//   A (16x16, row-major): a0 = A[g][c..c+1], a1 = A[g+8][c..c+1],
//                         a2 = A[g][c+8..c+9], a3 = A[g+8][c+8..c+9]
//   B (16x8, k x n):      b0 = B[c..c+1][g],   b1 = B[c+8..c+9][g]
//   C/D (16x8 fp32):      d0,d1 = D[g][c..c+1], d2,d3 = D[g+8][c..c+1]
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Barrier over `count` threads (a multiple of 32) with hardware barrier `id` (1..15).
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void ldsm_x4_t_addr(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_addr(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four 8x8 b16 matrices; lanes 8i..8i+7 give the row addresses of matrix i.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row_addr)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(row_addr)));
}

// A fragment of the 16x16 tile at (r0, c0) of a row-major bf16 array (row stride ld).
__device__ __forceinline__ void load_a(uint32_t (&a)[4], const __nv_bfloat16* base, int ld, int r0,
                                       int c0, int lane) {
  const int m = lane >> 3;
  ldsm_x4(a, base + (r0 + (lane & 7) + (m & 1) * 8) * ld + c0 + (m >> 1) * 8);
}

// A fragment of the 16x16 tile A = X^T where X is stored row-major [k][m]:
// A rows m0..m0+15 (columns of X), A cols k0..k0+15 (rows of X).
__device__ __forceinline__ void load_a_trans(uint32_t (&a)[4], const __nv_bfloat16* base, int ld,
                                             int m0, int k0, int lane) {
  const int m = lane >> 3;
  ldsm_x4_t(a, base + (k0 + (lane & 7) + (m >> 1) * 8) * ld + m0 + (m & 1) * 8);
}

// B fragments of two n-tiles (n0..n0+7 and n0+8..n0+15) over k0..k0+15, for B
// stored row-major as [k][n]: b[0],b[1] -> first n-tile, b[2],b[3] -> second.
__device__ __forceinline__ void load_b_kn(uint32_t (&b)[4], const __nv_bfloat16* base, int ld,
                                          int k0, int n0, int lane) {
  const int m = lane >> 3;
  ldsm_x4_t(b, base + (k0 + (lane & 7) + (m & 1) * 8) * ld + n0 + (m >> 1) * 8);
}

// Same, for B stored row-major as [n][k] (the "col" operand layout).
__device__ __forceinline__ void load_b_nk(uint32_t (&b)[4], const __nv_bfloat16* base, int ld,
                                          int k0, int n0, int lane) {
  const int m = lane >> 3;
  ldsm_x4(b, base + (n0 + (lane & 7) + (m >> 1) * 8) * ld + k0 + (m & 1) * 8);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// fp32 pair -> bf16 hi pair and bf16 lo pair (x = hi + lo to about 16 bits).
__device__ __forceinline__ void split_pack2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The same with fp16 halves: x = hi + lo, hi = fp16(x), lo = fp16(x - hi), about 22
// significant bits within the fp16 range.
__device__ __forceinline__ void split_pack2_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): about 16 significant bits.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ void split2_store(__nv_bfloat16* hi, __nv_bfloat16* lo, float x0,
                                             float x1) {
  __nv_bfloat16 h0, l0, h1, l1;
  split_bf16(x0, h0, l0);
  split_bf16(x1, h1, l1);
  *reinterpret_cast<__nv_bfloat162*>(hi) = __halves2bfloat162(h0, h1);
  *reinterpret_cast<__nv_bfloat162*>(lo) = __halves2bfloat162(l0, l1);
}

}  // namespace gdn
