// Top-k sparse attention over one shared KV head (SparseMLA style, "[2/2] Add
// TileLang fused DSA kernels support with THD and CP", Megatron-LM #5049:
// sparse MLA forward/backward with preprocess/postprocess, dim 576 =
// 512 latent + 64 rope, v_channels 512, -1 for empty top-k slots).
//
// The forward and the backward main kernel run on tcgen05 (sparse_fwd_tc.cu,
// sparse_bwd_tc.cu).  This file holds the backward's streaming passes around
// the main kernel: Delta = rowsum(dO * O), the chunk count of every token and
// the clearing of the fp32 dKV accumulator (or of the private slabs) before
// it; after it, the cast of the accumulator to bf16, or the sum of the slabs
// in slab order and its cast.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

constexpr int SP_DQK = 576;
constexpr int SP_DV = 512;

// Delta[t, h] = <dO, O> (fp32); nch[t] = chunks of kSparseChunk slots up to
// token t's last valid slot (0 when it has none); clearing of the fp32 dKV
// accumulator (max(slabs, 1) x [T, 576]).
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
  for (size_t t = gw; t < static_cast<size_t>(a.T); t += nw) {
    const int32_t* ir = a.idx + t * a.K;
    int last = -1;
    for (int s = lane; s < a.K; s += 32) {
      const int j = __ldg(ir + s);
      if (j >= 0 && j < a.T) last = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    if (lane == 0) a.nch[t] = (last + kSparseChunk) / kSparseChunk;
  }
  float4* z = reinterpret_cast<float4*>(a.dkv_acc);
  const size_t n4 = static_cast<size_t>(a.slabs > 0 ? a.slabs : 1) * a.T * (SP_DQK / 4);
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

// dkv = bf16(slab 0 + slab 1 + ... + slab nslab-1), added in that order (n4
// float4 per slab); eight slabs' loads in flight per thread.
__global__ void __launch_bounds__(256) sparse_dkv_slab_sum_kernel(const float* __restrict__ slabs,
                                                                  int nslab, size_t n4,
                                                                  __nv_bfloat16* __restrict__ dkv) {
  const float4* s4 = reinterpret_cast<const float4*>(slabs);
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float4 s = __ldcs(s4 + i);
    int b = 1;
    for (; b + 8 <= nslab; b += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcs(s4 + static_cast<size_t>(b + u) * n4 + i);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s.x += v[u].x;
        s.y += v[u].y;
        s.z += v[u].z;
        s.w += v[u].w;
      }
    }
    for (; b < nslab; ++b) {
      const float4 v = __ldcs(s4 + static_cast<size_t>(b) * n4 + i);
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    reinterpret_cast<uint2*>(dkv)[i] = make_uint2(pack_bf16(s.x, s.y), pack_bf16(s.z, s.w));
  }
}

cudaError_t launch_sparse_bwd(const SparseArgs& a, float* delta, __nv_bfloat16* dkv,
                              cudaStream_t st) {
  cudaError_t e;
  const size_t rows = static_cast<size_t>(a.T) * a.H;
  const int g = resident_grid(sparse_bwd_preprocess_kernel, rows * 32, 256);
  sparse_bwd_preprocess_kernel<<<g, 256, 0, st>>>(a, delta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  SparseArgs pa = a;
  pa.delta = delta;
  if ((e = launch_sparse_bwd_main(pa, st)) != cudaSuccess) return e;
  if (a.slabs > 0) {
    const size_t n4 = static_cast<size_t>(a.T) * SP_DQK / 4;
    const int gs = resident_grid(sparse_dkv_slab_sum_kernel, n4, 256);
    sparse_dkv_slab_sum_kernel<<<gs, 256, 0, st>>>(a.dkv_acc, a.slabs, n4, dkv);
    return cudaGetLastError();
  }
  const size_t n8 = static_cast<size_t>(a.T) * SP_DQK / 8;
  const int gc = resident_grid(sparse_dkv_cast_kernel, n8, 256);
  sparse_dkv_cast_kernel<<<gc, 256, 0, st>>>(a.dkv_acc, dkv, n8);
  return cudaGetLastError();
}

}  // namespace attn
