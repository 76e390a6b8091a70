// Memory-bound stages around the dense backward:
//   * preprocess: Delta = rowsum(dO o O) in fp32 (the `flashattn_bwd_preprocess`
//     stage of tile-ai/tilelang #940) and, for the atomic dQ mode, clearing of
//     the fp32 dQ accumulator;
//   * finalize: dQ = bf16(scale * accumulator) for the atomic mode, or
//     bf16(scale * sum of the per-KV-tile partials in ascending tile order) for
//     the split mode (the `flashattn_bwd_postprocess` stage of #940 and its
//     split+sum template); THD padding rows of dQ, dK and dV are written as
//     exact zeros here (the padding contract of cudnn-frontend #427, backward
//     zero-write commit, tokens beyond cu_seqlens[-1]).
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

// One group of D/8 threads per (row, head); 16-byte loads of O and dO.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(Problem p,
                                                                  const __nv_bfloat16* o,
                                                                  const __nv_bfloat16* dout,
                                                                  float* delta, float* dq_acc,
                                                                  size_t acc_elems) {
  constexpr int TPR = D / 8;   // threads per row
  const int end = valid_end(p);
  const size_t nrows = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q;
  const size_t gtid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  const int sub = threadIdx.x % TPR;
  // each warp takes 32 / TPR consecutive rows per step, so the loop trip count
  // is warp-uniform and the full-warp shuffles below stay converged
  const size_t step = nthreads / TPR;
  for (size_t base = (gtid / 32) * (32 / TPR); base < nrows; base += step) {
    const size_t rr = base + (threadIdx.x % 32) / TPR;
    const bool live = rr < nrows;
    float acc = 0.f;
    int h = 0, srow = 0, b = 0;
    if (live) {
      h = static_cast<int>(rr % p.heads_q);
      const size_t bs = rr / p.heads_q;
      srow = static_cast<int>(bs % p.rows_total);
      b = static_cast<int>(bs / p.rows_total);
      const uint4 ov = *reinterpret_cast<const uint4*>(o + rr * D + sub * 8);
      const uint4 dv = *reinterpret_cast<const uint4*>(dout + rr * D + sub * 8);
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
      const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(o2[i]);
        const float2 c = __bfloat1622float2(d2[i]);
        acc = fmaf(a.x, c.x, acc);
        acc = fmaf(a.y, c.y, acc);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && sub == 0) {
      size_t li;
      if (p.cu_seqlens)
        li = static_cast<size_t>(h) * p.rows_total + srow;
      else
        li = (static_cast<size_t>(b) * p.heads_q + h) * p.rows_total + srow;
      delta[li] = (srow < end) ? acc : 0.f;
    }
  }
  if (dq_acc) {
    float4* z = reinterpret_cast<float4*>(dq_acc);
    const size_t n4 = acc_elems / 4;
    for (size_t i = gtid; i < n4; i += nthreads) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Finalize dQ.  Each thread handles 8 consecutive head dims of one (row, head).
template <int D>
__global__ void __launch_bounds__(256) attn_dq_finalize_kernel(Problem p, const float* acc,
                                                               size_t slab_elems, int split,
                                                               int n_split, int kv_tile,
                                                               __nv_bfloat16* dq,
                                                               __nv_bfloat16* dk,
                                                               __nv_bfloat16* dv) {
  constexpr int CPR = D / 8;   // chunks per (row, head)
  const int end = valid_end(p);
  const size_t nchunks = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q * CPR;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  const float sc = p.scale;
  for (size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks;
       c += nthreads) {
    const size_t rh = c / CPR;
    const int sub = static_cast<int>(c % CPR);
    const size_t bs = rh / p.heads_q;
    const int hh = static_cast<int>(rh % p.heads_q);
    const int srow = static_cast<int>(bs % p.rows_total);
    const size_t bb = bs / p.rows_total;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (srow < end) {
      // accumulator / slabs are head-major: [batch, head, row, dim]
      const size_t e0 = ((bb * p.heads_q + hh) * p.rows_total + srow) * D + sub * 8;
      if (!split) {
        const float4 a0 = *reinterpret_cast<const float4*>(acc + e0);
        const float4 a1 = *reinterpret_cast<const float4*>(acc + e0 + 4);
        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
        v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
      } else {
        // sequence-local row index and length
        int local = srow, len = p.rows_total;
        if (p.cu_seqlens) {
          int lo = 0, hi = p.num_seqs - 1;
          while (lo < hi) {   // last sequence whose start <= srow
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu_seqlens + mid) <= srow) lo = mid; else hi = mid - 1;
          }
          const int s0 = __ldg(p.cu_seqlens + lo);
          local = srow - s0;
          len = __ldg(p.cu_seqlens + lo + 1) - s0;
        }
        const int ntile = (len + kv_tile - 1) / kv_tile;
        int nsum = p.causal ? local / kv_tile + 1 : ntile;
        if (nsum > n_split) nsum = n_split;   // sequence longer than max_seqlen (flagged)
        for (int j = 0; j < nsum; ++j) {
          const float* s = acc + j * slab_elems + e0;
          const float4 a0 = *reinterpret_cast<const float4*>(s);
          const float4 a1 = *reinterpret_cast<const float4*>(s + 4);
          v[0] += a0.x; v[1] += a0.y; v[2] += a0.z; v[3] += a0.w;
          v[4] += a1.x; v[5] += a1.y; v[6] += a1.z; v[7] += a1.w;
        }
      }
    }
    uint4 out;
    out.x = pack_bf16(v[0] * sc, v[1] * sc);
    out.y = pack_bf16(v[2] * sc, v[3] * sc);
    out.z = pack_bf16(v[4] * sc, v[5] * sc);
    out.w = pack_bf16(v[6] * sc, v[7] * sc);
    *reinterpret_cast<uint4*>(dq + rh * D + sub * 8) = out;
  }
  // THD: zero dK / dV rows past the last sequence
  if (p.cu_seqlens) {
    const size_t n = static_cast<size_t>(p.rows_total - end) * p.heads_kv * D / 8;
    const size_t off = static_cast<size_t>(end) * p.heads_kv * D / 8;
    uint4* k4 = reinterpret_cast<uint4*>(dk) + off;
    uint4* v4 = reinterpret_cast<uint4*>(dv) + off;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += nthreads) {
      k4[i] = make_uint4(0, 0, 0, 0);
      v4[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

static int grid_for(size_t work, int per_block) {
  size_t g = (work + per_block - 1) / per_block;
  const size_t cap = 152 * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

template <int D>
cudaError_t launch_bwd_preprocess(const Problem& p, const __nv_bfloat16* o,
                                  const __nv_bfloat16* dout, float* delta, float* dq_acc,
                                  size_t acc_elems, cudaStream_t st) {
  const size_t rows = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q;
  const int g = grid_for(rows * (D / 8), 256);
  attn_bwd_preprocess_kernel<D><<<g, 256, 0, st>>>(p, o, dout, delta, dq_acc, acc_elems);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_finalize(const Problem& p, const float* acc, size_t slab_elems, int split,
                               int n_split, __nv_bfloat16* dq, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t st) {
  const size_t chunks = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q * (D / 8);
  const int g = grid_for(chunks, 256);
  attn_dq_finalize_kernel<D><<<g, 256, 0, st>>>(p, acc, slab_elems, split, n_split, 128, dq,
                                                        dk, dv);
  return cudaGetLastError();
}

template cudaError_t launch_bwd_preprocess<64>(const Problem&, const __nv_bfloat16*,
                                               const __nv_bfloat16*, float*, float*, size_t,
                                               cudaStream_t);
template cudaError_t launch_bwd_preprocess<128>(const Problem&, const __nv_bfloat16*,
                                                const __nv_bfloat16*, float*, float*, size_t,
                                                cudaStream_t);
template cudaError_t launch_dq_finalize<64>(const Problem&, const float*, size_t, int, int,
                                            __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*,
                                            cudaStream_t);
template cudaError_t launch_dq_finalize<128>(const Problem&, const float*, size_t, int, int,
                                             __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*,
                                             cudaStream_t);

}  // namespace attn
