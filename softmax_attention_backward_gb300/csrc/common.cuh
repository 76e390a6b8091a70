// Shared host/device definitions of the attention kernels: problem
// descriptors passed to kernels, work decoding for dense and THD-packed
// layouts, and small math helpers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "fastdiv.h"
#include "sm100.cuh"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Kernel-side view of a dense (BSHD) or THD-packed problem.  For THD the
// tensors are treated as batch 1 with `rows_total` = capacity rows.
struct Problem {
  int batch;        // dense batch (1 for THD)
  int rows_total;   // rows of the S dimension of every tensor (seqlen or capacity)
  int heads_q;
  int heads_kv;
  int causal;
  float scale;
  const int32_t* cu_seqlens;  // null for dense
  int num_seqs;
  int max_seqlen;   // THD: bound on any sequence length
  int32_t* err;
  FastDiv fd_hq, fd_hkv, fd_grp;   // heads_q, heads_kv, heads_q / heads_kv
  FastDiv fd_ns;                   // num_seqs (1 for dense)
};

// One sequence of a problem: rows [row0, row0 + len) of batch entry `b`.
struct SeqRef {
  int b;
  int row0;
  int len;
};

// Decodes the linear tile index `x` (tiles of `tile_rows` rows) into a
// sequence and the local tile index inside it.  Returns false when `x` maps to
// no work (grids are sized by an upper bound for THD).
__device__ __forceinline__ bool decode_tile(const Problem& p, int x, int bz, int tile_rows,
                                            SeqRef& s, int& tile) {
  if (p.cu_seqlens == nullptr) {
    s.b = bz;
    s.row0 = 0;
    s.len = p.rows_total;
    const int n = (p.rows_total + tile_rows - 1) / tile_rows;
    if (x >= n) return false;
    tile = x;
    return true;
  }
  int rem = x;
  int prev = __ldg(p.cu_seqlens);
  for (int n = 0; n < p.num_seqs; ++n) {
    const int next = __ldg(p.cu_seqlens + n + 1);
    const int len = next > prev ? next - prev : 0;
    const int nt = (len + tile_rows - 1) / tile_rows;
    if (rem < nt) {
      s.b = 0;
      s.row0 = prev;
      s.len = len;
      tile = rem;
      return true;
    }
    rem -= nt;
    prev = next;
  }
  return false;
}

// Upper bound on the number of tiles of `tile_rows` rows over all sequences.
inline int tile_bound(int rows_total, int num_seqs, int tile_rows, bool packed) {
  const int base = (rows_total + tile_rows - 1) / tile_rows;
  return packed ? base + num_seqs : base;
}

// End of the valid rows of a THD problem (cu_seqlens[num_seqs], kept within
// [0, rows_total] so that a list breaking its contract cannot move the passes
// that use it out of their buffers); rows_total for dense.
__device__ __forceinline__ int valid_end(const Problem& p) {
  return p.cu_seqlens ? min(max(__ldg(p.cu_seqlens + p.num_seqs), 0), p.rows_total) : p.rows_total;
}

}  // namespace attn

namespace attn {

// Packed fp32x2 arithmetic (sm_100 family): two lanes of work per instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// bf16x2 of (lo, hi), lo in the low half.
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  return pack_bf16(lo, hi);
}

}  // namespace attn
