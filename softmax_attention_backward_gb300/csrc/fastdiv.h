// Unsigned 32-bit division by a runtime-invariant divisor without a divide
// instruction: a multiply-high by a magic number computed once on the host
// (T. Granlund and P. L. Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, the unsigned N-bit method of their Figure 4.1).
//
// The kernels decode work items (batch, head, tile) from linear indices.  A
// plain `/` by a runtime value compiles to a reciprocal estimate on the
// special-function unit, where it waits behind the exponentials of the
// softmax warps that share the unit; the multiply-high does not.
//
// With l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1:
//   t = mulhi(m, n),  n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0)
// for every n < 2^32 and 1 <= d < 2^32.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

struct FastDiv {
  uint32_t d;    // divisor
  uint32_t m;    // magic multiplier
  uint32_t s1;   // min(l, 1)
  uint32_t s2;   // max(l - 1, 0)
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{};
  if (d == 0) d = 1;   // never used with 0; keeps the table well defined
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;
  f.d = d;
  f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 1 ? l - 1 : 0;
  return f;
}

ATTN_HD uint32_t mulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return static_cast<uint32_t>((static_cast<uint64_t>(a) * b) >> 32);
#endif
}

ATTN_HD uint32_t fdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = mulhi32(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

ATTN_HD uint32_t fmod_u(uint32_t n, const FastDiv& f) { return n - fdiv(n, f) * f.d; }

}  // namespace attn
