// Warp-level tensor-core products on sm_103a: mma.sync m16n8k8 with tf32
// operands and fp32 accumulation, for the small dense contractions of the
// prefill scan and of the decode fold.
#pragma once

#include <cstdint>

namespace rssm {

// ---- warp-level tensor-core products (mma m16n8k8, tf32 in, fp32 accumulate).
// Fragments, g = lane / 4, t = lane % 4: A (16 x 8) a0 (g, t), a1 (g + 8, t),
// a2 (g, t + 4), a3 (g + 8, t + 4); B (8 x 8) b0 (t, g), b1 (t + 4, g);
// C (16 x 8) c0 (g, 2t), c1 (g, 2t + 1), c2 (g + 8, 2t), c3 (g + 8, 2t + 1).
// fp32 operands are split into a tf32 head and tail, x = hi + lo, and a
// product takes hi*hi + hi*lo + lo*hi, which keeps it near fp32 accuracy; an
// operand that is exact in tf32 (bf16 values) has no tail.

struct Tf32 {
  uint32_t hi, lo;
};

// The head is the operand truncated to tf32 (its low 13 bits cleared), the
// tail the exact fp32 remainder truncated to tf32 in the same way: the pair
// carries about 21 significant bits of the operand.
template <bool EXACT>
__device__ __forceinline__ Tf32 tf32_split(float x) {
  if (EXACT) return Tf32{__float_as_uint(x), 0u};
  const uint32_t hi = __float_as_uint(x) & 0xffffe000u;
  return Tf32{hi, __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u};
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// c += A B for split operands (the tail products first)
template <bool EXACT_A, bool EXACT_B>
__device__ __forceinline__ void mma_split(float (&c)[4], const Tf32 (&a)[4], const Tf32 (&b)[2]) {
  if (!EXACT_A) mma_tf32(c, a[0].lo, a[1].lo, a[2].lo, a[3].lo, b[0].hi, b[1].hi);
  if (!EXACT_B) mma_tf32(c, a[0].hi, a[1].hi, a[2].hi, a[3].hi, b[0].lo, b[1].lo);
  mma_tf32(c, a[0].hi, a[1].hi, a[2].hi, a[3].hi, b[0].hi, b[1].hi);
}

// Fragment order of the mat-vec inputs of a window with 8 NTN vectors (NTN
// n-tiles of eight): for rows [8s, 8s + 8) lane (g, t) finds at
// [2 NTN (32 s + 4 g + t) + 2 nt + h] vector 8 nt + g of row 8s + 2t + h.
// x_slot maps slot e back to its (row ch, vector v).
template <int NTN>
__device__ __forceinline__ void x_slot(int e, int& ch, int& v) {
  constexpr int CPL = 2 * NTN;  // values per lane and step
  const int s8 = e / (32 * CPL), ln = (e / CPL) & 31, comp = e % CPL;
  ch = 8 * s8 + 2 * (ln & 3) + (comp & 1);
  v = 8 * (comp >> 1) + (ln >> 2);
}

}  // namespace rssm
