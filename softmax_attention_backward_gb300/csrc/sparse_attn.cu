// Top-k sparse attention over one shared KV head (SparseMLA style, "[2/2] Add
// TileLang fused DSA kernels support with THD and CP", Megatron-LM #5049:
// sparse MLA forward/backward with preprocess/postprocess, dim 576 =
// 512 latent + 64 rope, v_channels 512, -1 for empty top-k slots).
//
// The forward and the backward main kernel run on tcgen05 (sparse_fwd_tc.cu,
// sparse_bwd_tc.cu).  This file holds the backward's streaming passes around
// the main kernel: Delta = rowsum(dO * O) with the clearing of the fp32 dKV
// accumulator before it, and the cast of the accumulator to bf16 after it.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

constexpr int SP_DQK = 576;
constexpr int SP_DV = 512;

// Delta[t, h] = <dO, O> (fp32) and clearing of the fp32 dKV accumulator.
__global__ void __launch_bounds__(256) sparse_bwd_preprocess_kernel(const SparseArgs a,
                                                                    float* delta) {
  const size_t rows = static_cast<size_t>(a.T) * a.H;
  const size_t gw = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const size_t nw = (static_cast<size_t>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (size_t r = gw; r < rows; r += nw) {
    const __nv_bfloat16* o = a.o + r * SP_DV;
    const __nv_bfloat16* d = a.dout + r * SP_DV;
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < SP_DV / 256; ++i) {
      const uint4 ov = *reinterpret_cast<const uint4*>(o + i * 256 + lane * 8);
      const uint4 dv = *reinterpret_cast<const uint4*>(d + i * 256 + lane * 8);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(o2[e]);
        const float2 y = __bfloat1622float2(d2[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) delta[r] = acc;
  }
  float4* z = reinterpret_cast<float4*>(a.dkv_acc);
  const size_t n4 = a.dkv_acc ? static_cast<size_t>(a.T) * SP_DQK / 4 : 0;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) sparse_dkv_cast_kernel(const float* acc,
                                                              __nv_bfloat16* dkv, size_t n8) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a0 = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 a1 = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a0.x, a0.y);
    o.y = pack_bf16(a0.z, a0.w);
    o.z = pack_bf16(a1.x, a1.y);
    o.w = pack_bf16(a1.z, a1.w);
    reinterpret_cast<uint4*>(dkv)[i] = o;
  }
}

cudaError_t launch_sparse_bwd(const SparseArgs& a, float* delta, __nv_bfloat16* dkv,
                              cudaStream_t st) {
  cudaError_t e;
  const size_t rows = static_cast<size_t>(a.T) * a.H;
  const int g = resident_grid(sparse_bwd_preprocess_kernel, rows * 32, 256);
  SparseArgs pa = a;
  sparse_bwd_preprocess_kernel<<<g, 256, 0, st>>>(pa, delta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  pa.delta = delta;
  if ((e = launch_sparse_bwd_main(pa, st)) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(a.T) * SP_DQK / 8;
  const int gc = resident_grid(sparse_dkv_cast_kernel, n8, 256);
  sparse_dkv_cast_kernel<<<gc, 256, 0, st>>>(a.dkv_acc, dkv, n8);
  return cudaGetLastError();
}

cudaError_t launch_sparse_bwd_ordered(const SparseArgs& a, float* delta, int32_t* table,
                                      int32_t* total, int32_t* off, int32_t* entries,
                                      __nv_bfloat16* dkv, cudaStream_t st) {
  cudaError_t e;
  const size_t rows = static_cast<size_t>(a.T) * a.H;
  const int g = resident_grid(sparse_bwd_preprocess_kernel, rows * 32, 256);
  SparseArgs pa = a;
  pa.dkv_acc = nullptr;   // Delta only: there is no accumulator to clear
  sparse_bwd_preprocess_kernel<<<g, 256, 0, st>>>(pa, delta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const SparseCsrLayout l = sparse_csr_layout(a.T, a.K);
  if ((e = launch_sparse_csr(a.idx, a.T, a.K, l, table, total, off, entries, st)) != cudaSuccess)
    return e;
  pa.delta = delta;
  if ((e = launch_sparse_bwd_main(pa, st)) != cudaSuccess) return e;
  const int nhb = (a.H + 63) / 64;
  return launch_sparse_dkv_reduce(a.contrib, entries, off, a.T, nhb, dkv, st);
}

}  // namespace attn
