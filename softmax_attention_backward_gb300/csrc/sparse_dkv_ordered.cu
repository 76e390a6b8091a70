// Deterministic dKV for the top-k sparse backward: disjoint ownership instead
// of atomics (the ordering discipline of "[2/2] Add TileLang fused DSA kernels
// support with THD and CP", Megatron-LM #5049, whose sparse MLA backward adds
// dKV with fp32 atomics; its review thread and the CSA kernels' notes on
// bitwise reproducibility ask for a fixed reduction order).
//
// The backward main kernel stores every (token, slot, head block)
// contribution row dS^T Q + P^T [dO | 0] (fp32, dim_qk wide) once, into a
// workspace indexed by (token * topk + slot) * head_blocks + head_block,
// instead of adding it into dKV.  Here the index lists are inverted into a
// CSR by key row, each row's entries in ascending token order:
//   count  per (token block, key row) the slots that name the row
//   scan   down the token blocks per key row (block bases and totals), then
//          across key rows (row offsets)
//   fill   each token block walks its tokens in order and appends (t, slot)
//          at its row's running position
// and one CTA per key row sums its contribution rows in a fixed tree (eight
// contiguous segments of the ordered list, each summed in order by a warp,
// then the segment sums in segment order) and writes the bf16 dKV row.  The
// result is bitwise reproducible; it differs from the atomic path only in the
// order of the fp32 additions.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

namespace {

constexpr int kDqk = 576;
constexpr int kCsrThreads = 512;

__global__ void __launch_bounds__(kCsrThreads) csr_count_kernel(const int32_t* __restrict__ idx,
                                                                int T, int K, int tb,
                                                                int32_t* __restrict__ table) {
  const int b = blockIdx.x;
  const int t_end = min(T, (b + 1) * tb);
  int32_t* row = table + static_cast<size_t>(b) * T;
  for (int t = b * tb; t < t_end; ++t) {
    const int32_t* it = idx + static_cast<size_t>(t) * K;
    for (int s = threadIdx.x; s < K; s += blockDim.x) {
      const int j = __ldg(it + s);
      if (j >= 0 && j < T) atomicAdd(row + j, 1);
    }
  }
}

// Per key row j: exclusive prefix over the token blocks (in place), total.
__global__ void __launch_bounds__(256) csr_colscan_kernel(int32_t* __restrict__ table, int T,
                                                          int nblk, int32_t* __restrict__ total) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= T) return;
  int run = 0;
  for (int b = 0; b < nblk; ++b) {
    int32_t* c = table + static_cast<size_t>(b) * T + j;
    const int v = *c;
    *c = run;
    run += v;
  }
  total[j] = run;
}

// Exclusive prefix of total[0..T) into off[0..T], one block.
__global__ void __launch_bounds__(1024) csr_rowscan_kernel(const int32_t* __restrict__ total,
                                                           int T, int32_t* __restrict__ off) {
  __shared__ int part[1024];
  const int n = blockDim.x, tid = threadIdx.x;
  const int per = (T + n - 1) / n;
  const int lo = min(T, tid * per), hi = min(T, lo + per);
  int sum = 0;
  for (int j = lo; j < hi; ++j) sum += total[j];
  part[tid] = sum;
  __syncthreads();
  // Hillis-Steele inclusive scan of the per-thread sums
  for (int d = 1; d < n; d <<= 1) {
    const int v = tid >= d ? part[tid - d] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - sum;
  for (int j = lo; j < hi; ++j) {
    off[j] = run;
    run += total[j];
  }
  if (tid == n - 1) off[T] = part[n - 1];
}

__global__ void __launch_bounds__(kCsrThreads) csr_fill_kernel(const int32_t* __restrict__ idx,
                                                               int T, int K, int tb,
                                                               int32_t* __restrict__ table,
                                                               const int32_t* __restrict__ off,
                                                               int32_t* __restrict__ entries) {
  const int b = blockIdx.x;
  const int t_end = min(T, (b + 1) * tb);
  int32_t* row = table + static_cast<size_t>(b) * T;
  for (int t = b * tb; t < t_end; ++t) {
    const int32_t* it = idx + static_cast<size_t>(t) * K;
    for (int s = threadIdx.x; s < K; s += blockDim.x) {
      const int j = __ldg(it + s);
      // a token names a row at most once, so within a token the running
      // positions do not collide; the atomic only keeps the positions
      // distinct for lists that break that contract
      if (j >= 0 && j < T) entries[off[j] + atomicAdd(row + j, 1)] = t * K + s;
    }
    __syncthreads();   // tokens append in ascending order
  }
}

// One CTA of kRedWarps warps per key row.  The row's contribution rows (in
// entry order) are cut into kRedWarps contiguous segments of equal count;
// warp w sums segment w in order, lane l owning dims 2l + 64k, k = 0..8
// (float2 each), and the partial sums are added in warp order.  The tree
// depends only on the entry list, so the result is bitwise repeatable, and
// the rows named by many tokens (the first rows under a causal selection)
// are spread over eight warps instead of setting the kernel's length.
constexpr int kRedWarps = 8;

__global__ void __launch_bounds__(32 * kRedWarps) dkv_reduce_kernel(
    const float* __restrict__ contrib, const int32_t* __restrict__ entries,
    const int32_t* __restrict__ off, int T, int nhb, __nv_bfloat16* __restrict__ dkv) {
  __shared__ float2 part[kRedWarps][kDqk / 2];
  const int j = blockIdx.x;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[18];
#pragma unroll
  for (int i = 0; i < 18; ++i) acc[i] = 0.f;
  const int e0 = off[j], e1 = off[j + 1];
  const long long nrow = static_cast<long long>(e1 - e0) * nhb;   // contribution rows of key row j
  const int i_end = static_cast<int>(nrow * (w + 1) / kRedWarps);
  auto row_of = [&](int i) -> const float2* {
    const int e = e0 + i / nhb, h = i - (i / nhb) * nhb;
    const size_t base = (static_cast<size_t>(__ldg(entries + e)) * nhb + h) * kDqk;
    return reinterpret_cast<const float2*>(contrib + base) + lane;
  };
  int i = static_cast<int>(nrow * w / kRedWarps);
  // four rows in flight per warp (the loads of a row are independent of the
  // sums, so they overlap; the additions stay in row order)
  for (; i + 4 <= i_end; i += 4) {
    float2 v[4][9];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2* r = row_of(i + u);
#pragma unroll
      for (int k = 0; k < 9; ++k) v[u][k] = __ldcs(r + 32 * k);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        acc[2 * k] += v[u][k].x;
        acc[2 * k + 1] += v[u][k].y;
      }
  }
  for (; i < i_end; ++i) {
    const float2* r = row_of(i);
    float2 v[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) v[k] = __ldcs(r + 32 * k);
#pragma unroll
    for (int k = 0; k < 9; ++k) {
      acc[2 * k] += v[k].x;
      acc[2 * k + 1] += v[k].y;
    }
  }
#pragma unroll
  for (int k = 0; k < 9; ++k) part[w][lane + 32 * k] = make_float2(acc[2 * k], acc[2 * k + 1]);
  __syncthreads();
  uint32_t* out = reinterpret_cast<uint32_t*>(dkv + static_cast<size_t>(j) * kDqk);
  for (int d = threadIdx.x; d < kDqk / 2; d += 32 * kRedWarps) {
    float2 sum = part[0][d];
#pragma unroll
    for (int u = 1; u < kRedWarps; ++u) {
      sum.x += part[u][d].x;
      sum.y += part[u][d].y;
    }
    out[d] = pack_bf16(sum.x, sum.y);
  }
}

}  // namespace

SparseCsrLayout sparse_csr_layout(int T, int K) {
  SparseCsrLayout l{};
  const int nblk_max = 128;
  l.nblk = T < nblk_max ? T : nblk_max;
  if (l.nblk < 1) l.nblk = 1;
  l.tb = (T + l.nblk - 1) / l.nblk;
  l.nblk = (T + l.tb - 1) / l.tb;
  l.table_elems = static_cast<size_t>(l.nblk) * T;
  l.total_elems = static_cast<size_t>(T);
  l.off_elems = static_cast<size_t>(T) + 1;
  l.entry_elems = static_cast<size_t>(T) * K;
  return l;
}

cudaError_t launch_sparse_csr(const int32_t* idx, int T, int K, const SparseCsrLayout& l,
                              int32_t* table, int32_t* total, int32_t* off, int32_t* entries,
                              cudaStream_t st) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(table, 0, l.table_elems * sizeof(int32_t), st)) != cudaSuccess) return e;
  csr_count_kernel<<<l.nblk, kCsrThreads, 0, st>>>(idx, T, K, l.tb, table);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  csr_colscan_kernel<<<(T + 255) / 256, 256, 0, st>>>(table, T, l.nblk, total);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  csr_rowscan_kernel<<<1, 1024, 0, st>>>(total, T, off);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  csr_fill_kernel<<<l.nblk, kCsrThreads, 0, st>>>(idx, T, K, l.tb, table, off, entries);
  return cudaGetLastError();
}

cudaError_t launch_sparse_dkv_reduce(const float* contrib, const int32_t* entries,
                                     const int32_t* off, int T, int nhb, __nv_bfloat16* dkv,
                                     cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  dkv_reduce_kernel<<<T, 32 * kRedWarps, 0, st>>>(contrib, entries, off, T, nhb, dkv);
  return cudaGetLastError();
}

}  // namespace attn
