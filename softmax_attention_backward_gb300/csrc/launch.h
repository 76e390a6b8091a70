// Argument blocks and launch wrappers shared by the kernel translation units
// and the C ABI layer.
#pragma once

#include <cuda_runtime.h>

#include "attn.h"
#include "common.cuh"

namespace attn {

// The argument checks of every dense/THD entry point (status codes of attn.h);
// sets *empty when there is nothing to compute.
attn_status_t validate_dense_problem(const attn_problem_t* p, bool* empty);

// 4-D TMA map over a bf16 tensor [batch, rows, heads, dim] (dim contiguous): box
// of 64 dims x 1 head x box_rows rows x 1 batch, 128-byte swizzle, zero fill
// out of bounds.  False when the driver entry point is missing or refuses it.
bool make_bf16_tile_map(CUtensorMap* m, const void* ptr, int batch, int rows, int heads, int dim,
                        int box_rows);

// Streaming multiprocessors of the current device (0 if it cannot be read).
int sm_count();

// Grid of a grid-stride kernel: at most `waves` whole waves of co-resident
// blocks (SMs x the blocks of `threads` threads that fit on one SM at the
// kernel's register and shared-memory use), fewer when the work is smaller.
// A grid that is not a whole number of waves ends in a partial wave that
// leaves most of every SM idle.
template <typename Kernel>
inline int resident_grid(Kernel kernel, size_t work, int threads, int waves = 1) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int sms = sm_count();
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 1) * per_sm * (waves > 0 ? waves : 1);
  size_t g = (work + threads - 1) / threads;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

struct FwdArgs {
  Problem p;
  __nv_bfloat16* o;
  float* lse;
  float scale_log2;
  int total_items;      // work items: query-tile-pair slots x heads x batch
  int n_x;              // query-tile-pair slots per (batch, head)
  int x_major;          // item numbering, see next_fwd_item
  FastDiv fd_nx, fd_nbh; // n_x and heads_q * batch
};

struct BwdArgs {
  Problem p;
  const float* lse;
  const float* delta;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dq_acc;        // ATOMIC: accumulator [B, Hq, rows, D]; SPLIT: slab base
  size_t slab_elems;    // SPLIT, head_dim 64: elements per slab (0 otherwise)
  int n_split;          // SPLIT, head_dim 64: number of slabs
  int* dq_ticket;       // SPLIT, head_dim 128: order tickets [batch, head, n_x] (else null)
  int split;            // 1 = SPLIT
  int dq_tma;           // 1 = dQ tiles leave through the TMA map of the accumulator / slabs
  int total_items;      // work items: K/V tile slots x kv heads x batch
  int n_x;              // K/V tile slots per (batch, kv head)
  int x_major;          // item numbering, see next_bwd_item
  int pad_zero;         // THD, head_dim 128: the kernel writes the padding rows of dK and dV
  float scale_log2;
  FastDiv fd_nx, fd_nbh; // n_x and heads_kv * batch
};

template <int D>
cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x, cudaStream_t st);
template <int D>
cudaError_t launch_attn_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dO, const CUtensorMap& dq, const CUtensorMap& dk,
                            const CUtensorMap& dv, const BwdArgs& a, int grid, cudaStream_t st);
// head_dim 128 (attn_bwd_d128.cu): 128 x 128 steps; dQ, dK and dV leave from
// registers with plain global accesses
cudaError_t launch_attn_bwd128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dO,
                               const BwdArgs& a, int grid, cudaStream_t st);
// `clear` (n_clear 4-byte words, a multiple of 4) is zeroed as well when not
// null (the order tickets of SPLIT at head_dim 128).
template <int D>
cudaError_t launch_bwd_preprocess(const Problem& p, const __nv_bfloat16* o,
                                  const __nv_bfloat16* dout, float* delta, float* dq_acc,
                                  size_t acc_elems, float* clear, size_t n_clear,
                                  cudaStream_t st);
template <int D>
cudaError_t launch_dq_finalize(const Problem& p, const float* acc, size_t slab_elems, int split,
                               int n_split, __nv_bfloat16* dq, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t st);

}  // namespace attn

namespace attn {

// Key slots per chunk of the sparse backward main kernel.
constexpr int kSparseChunk = 64;
// Private fp32 dKV accumulators of the deterministic sparse backward: its
// main kernel runs this many CTAs (fewer when there are fewer items), one slab
// each.  A fixed count, not the device's SM count, so that the result does not
// depend on the device.
constexpr int kSparseSlabs = 152;

struct SparseArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const int32_t* idx;
  __nv_bfloat16* o;
  float* lse;
  const __nv_bfloat16* dout;
  const float* lse_in;
  const float* delta;
  __nv_bfloat16* dq;
  float* dkv_acc;        // fp32 dKV accumulator [T, 576], or slabs x [T, 576]
  int32_t* nch;          // backward: chunks of 64 slots per token (preprocess output)
  int slabs;             // 0: one shared accumulator; else the number of private slabs
  int T, H, K;
  float scale, scale_log2;
  int32_t* err;
};

cudaError_t launch_sparse_fwd(const SparseArgs& a, cudaStream_t st);
// Backward: preprocess (Delta, chunk counts, clearing the accumulator or
// slabs), main kernel, then the bf16 cast (shared accumulator) or the
// slab-order sum and cast (slabs).
cudaError_t launch_sparse_bwd(const SparseArgs& a, float* delta, __nv_bfloat16* dkv,
                              cudaStream_t st);
cudaError_t launch_sparse_bwd_main(const SparseArgs& a, cudaStream_t st);

}  // namespace attn
