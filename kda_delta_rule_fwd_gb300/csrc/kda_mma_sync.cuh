// Warp-level tensor-core products on the legacy mma.sync path (m16n8k8, tf32),
// used where a product has 16 rows: below the tensor-memory MMA's minimum M.
#pragma once
#include <cstdint>

namespace kda {

// Warp-level m16n8k8 tf32 product with fp32 accumulation, split three ways
// for float32 accuracy: acc[0] += hi(a) hi(b), acc[1] += hi(a) lo(b),
// acc[2] += lo(a) hi(b).  hi keeps the sign, the exponent and the top 10
// mantissa bits of x (truncation, one bitwise AND), lo = x - hi (exact) cut the
// same way, so the dropped lo(a) lo(b) term and the cuts leave about 2^-20 of
// each product.
// Fragments: a = (row g, col t), (g+8, t), (g, t+4), (g+8, t+4);
// b = (row t, col g), (t+4, g); c = (g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
// with g = lane/4, t = lane%4.
__device__ __forceinline__ uint32_t tf32_hi(float x) { return __float_as_uint(x) & 0xffffe000u; }
__device__ __forceinline__ uint32_t tf32_lo(float x, uint32_t hi) {
  return __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma_tf32x3(float (&acc)[3][4], const float (&a)[4],
                                           const float (&b)[2]) {
  uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ah[i] = tf32_hi(a[i]);
    al[i] = tf32_lo(a[i], ah[i]);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    bh[i] = tf32_hi(b[i]);
    bl[i] = tf32_lo(b[i], bh[i]);
  }
  mma_tf32(acc[0], ah, bh);
  mma_tf32(acc[1], ah, bl);
  mma_tf32(acc[2], al, bh);
}

}  // namespace kda
