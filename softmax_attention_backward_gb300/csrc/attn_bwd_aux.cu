// Memory-bound stages around the dense backward:
//   * preprocess: Delta = rowsum(dO o O) in fp32 (the `flashattn_bwd_preprocess`
//     stage of tile-ai/tilelang #940) and, for the atomic dQ mode, clearing of
//     the fp32 dQ accumulator (for the split mode at head_dim 128, of its order
//     tickets);
//   * finalize: dQ = bf16(scale * accumulator) for the atomic mode and the
//     split mode at head_dim 128, or bf16(scale * sum of the per-KV-tile
//     partials in ascending tile order) for the split mode at head_dim 64
//     (the `flashattn_bwd_postprocess` stage of #940 and its
//     split+sum template); THD padding rows of dQ, dK and dV are written as
//     exact zeros here (the padding contract of cudnn-frontend #427, backward
//     zero-write commit, tokens beyond cu_seqlens[-1]).
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

// Index math of the two kernels runs in 32 bits: the host checks that one
// batch entry holds fewer than 2^31 elements, and the launchers below fall
// back to a grid that covers 2^31 rows x heads at most per launch offset.

// One group of D/8 threads per (row, head); 16-byte loads of O and dO.  Each
// group handles two (row, head) pairs per iteration so that four 16-byte
// loads per thread are in flight.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(Problem p,
                                                                  const __nv_bfloat16* __restrict__ o,
                                                                  const __nv_bfloat16* __restrict__ dout,
                                                                  float* __restrict__ delta,
                                                                  float* __restrict__ dq_acc,
                                                                  size_t acc_elems,
                                                                  float* __restrict__ clear,
                                                                  size_t n_clear) {
  constexpr int TPR = D / 8;   // threads per row
  constexpr int RPW = 32 / TPR;   // rows per warp step
  const int end = valid_end(p);
  // THD (batch 1): the rows before the end of the last sequence here, the
  // padding rows' exact zeros by the contiguous fill below
  const uint32_t nrows = p.cu_seqlens ? static_cast<uint32_t>(end) * p.heads_q
                                      : static_cast<uint32_t>(p.batch) * p.rows_total * p.heads_q;
  const uint32_t nthreads = gridDim.x * blockDim.x;
  const uint32_t gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int sub = threadIdx.x % TPR;
  const uint32_t hq = p.heads_q, rt = p.rows_total;
  // each warp takes 2 * RPW consecutive rows per step, so the loop trip count
  // is warp-uniform and the full-warp shuffles below stay converged
  const uint32_t step = (nthreads / 32) * 2 * RPW;
  for (uint32_t base = (gtid / 32) * 2 * RPW; base < nrows; base += step) {
    uint32_t rr[2];
    float acc[2] = {0.f, 0.f};
    uint4 ov[2], dv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rr[u] = base + u * RPW + (threadIdx.x % 32) / TPR;
      ov[u] = dv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (rr[u] < nrows) {
        ov[u] = *reinterpret_cast<const uint4*>(o + static_cast<size_t>(rr[u]) * D + sub * 8);
        dv[u] = *reinterpret_cast<const uint4*>(dout + static_cast<size_t>(rr[u]) * D + sub * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (rr[u] < nrows) {
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[u]);
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 a = __bfloat1622float2(o2[i]);
          const float2 c = __bfloat1622float2(d2[i]);
          acc[u] = fmaf(a.x, c.x, acc[u]);
          acc[u] = fmaf(a.y, c.y, acc[u]);
        }
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) {
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], off);
      acc[1] += __shfl_xor_sync(0xffffffffu, acc[1], off);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (rr[u] < nrows && sub == 0) {
        const uint32_t h = rr[u] % hq;
        const uint32_t bs = rr[u] / hq;
        const uint32_t srow = bs % rt;
        const uint32_t b = bs / rt;
        size_t li;
        if (p.cu_seqlens)
          li = static_cast<size_t>(h) * rt + srow;
        else
          li = (static_cast<size_t>(b) * hq + h) * rt + srow;
        delta[li] = acc[u];
      }
    }
  }
  if (p.cu_seqlens) {
    // Delta of the THD padding rows (end .. rows_total of every head): exact zeros
    const uint32_t pad = rt - static_cast<uint32_t>(end);
    for (uint32_t i = gtid; i < pad * hq; i += nthreads) {
      const uint32_t h = i / pad;
      delta[static_cast<size_t>(h) * rt + end + (i - h * pad)] = 0.f;
    }
  }
  if (clear) {
    float4* z = reinterpret_cast<float4*>(clear);
    for (size_t i = gtid; i < n_clear / 4; i += nthreads) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (dq_acc) {
    // the accumulator is [batch, head, row, dim]: clear the first `end` rows of
    // every (batch, head) segment (all rows for dense; the finalize writes
    // zeros for THD rows past the last sequence without reading them)
    float4* z = reinterpret_cast<float4*>(dq_acc);
    if (p.cu_seqlens == nullptr) {
      const size_t n4 = acc_elems / 4;
      for (size_t i = gtid; i < n4; i += nthreads) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      // THD (batch 1): rows [0, end) of each head's segment
      const uint32_t seg4 = static_cast<uint32_t>(end) * (D / 4);
      const size_t stride4 = static_cast<size_t>(rt) * (D / 4);
      const uint32_t n4 = seg4 * hq;
      for (uint32_t i = gtid; i < n4; i += nthreads) {
        const uint32_t sgm = i / seg4;
        z[sgm * stride4 + (i - sgm * seg4)] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// Finalize dQ.  Each thread handles 8 consecutive head dims of one (row,
// head); in the atomic mode it converts two such chunks per iteration.
template <int D>
__global__ void __launch_bounds__(256) attn_dq_finalize_kernel(Problem p,
                                                               const float* __restrict__ acc,
                                                               size_t slab_elems, int split,
                                                               int n_split, int kv_tile,
                                                               __nv_bfloat16* __restrict__ dq,
                                                               __nv_bfloat16* __restrict__ dk,
                                                               __nv_bfloat16* __restrict__ dv) {
  constexpr int CPR = D / 8;   // chunks per (row, head)
  const int end = valid_end(p);
  const uint32_t hq = p.heads_q, rt = p.rows_total;
  const uint32_t nchunks = static_cast<uint32_t>(p.batch) * rt * hq * CPR;
  const uint32_t nthreads = gridDim.x * blockDim.x;
  const float sc = p.scale;
  // Chunk c (8 dims) walks the head-major accumulator / slabs [batch, head,
  // row, dim] in memory order, so a warp reads one contiguous kilobyte; its dQ
  // destination [batch, row, head, dim] is a whole 128-byte line per (row,
  // head) for D = 64.  Returns the dQ element offset and the row.
  auto dq_index = [&](uint32_t c, int& srow) -> size_t {
    const uint32_t sub = c % CPR;
    const uint32_t rh = c / CPR;             // (batch, head, row)
    srow = static_cast<int>(rh % rt);
    const uint32_t bh = rh / rt;
    const uint32_t hh = bh % hq;
    const uint32_t bb = bh / hq;
    return ((static_cast<size_t>(bb) * rt + srow) * hq + hh) * D + sub * 8;
  };
  auto store = [&](size_t di, const float (&v)[8]) {
    uint4 out;
    out.x = pack_bf16(v[0] * sc, v[1] * sc);
    out.y = pack_bf16(v[2] * sc, v[3] * sc);
    out.z = pack_bf16(v[4] * sc, v[5] * sc);
    out.w = pack_bf16(v[6] * sc, v[7] * sc);
    *reinterpret_cast<uint4*>(dq + di) = out;
  };
  const uint32_t c_first = blockIdx.x * blockDim.x + threadIdx.x;
  if (!split) {
    // four chunks (128 bytes of the accumulator) in flight per thread
    constexpr int U = 4;
    for (uint32_t c0 = c_first; c0 < nchunks; c0 += U * nthreads) {
      float4 a[U][2];
      bool live[U];
      size_t di[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t cu = c0 + u * nthreads;
        int srow = 0;
        live[u] = false;
        di[u] = 0;
        a[u][0] = a[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (cu < nchunks) {
          di[u] = dq_index(cu, srow);
          live[u] = true;
          if (srow < end) {
            const float4* src = reinterpret_cast<const float4*>(acc + static_cast<size_t>(cu) * 8);
            a[u][0] = __ldcs(src);
            a[u][1] = __ldcs(src + 1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!live[u]) continue;
        const float v[8] = {a[u][0].x, a[u][0].y, a[u][0].z, a[u][0].w,
                            a[u][1].x, a[u][1].y, a[u][1].z, a[u][1].w};
        store(di[u], v);
      }
    }
  } else {
    for (uint32_t c = c_first; c < nchunks; c += nthreads) {
      int srow = 0;
      const size_t di = dq_index(c, srow);
      const size_t e0 = static_cast<size_t>(c) * 8;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (srow < end) {
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
      store(di, v);
    }
  }
  // THD: zero dK / dV rows past the last sequence (when dk is not null; the
  // backward main kernels write them and pass null here)
  if (p.cu_seqlens && dk) {
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

template <int D>
cudaError_t launch_bwd_preprocess(const Problem& p, const __nv_bfloat16* o,
                                  const __nv_bfloat16* dout, float* delta, float* dq_acc,
                                  size_t acc_elems, float* clear, size_t n_clear,
                                  cudaStream_t st) {
  const size_t rows = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q;
  const int g = resident_grid(attn_bwd_preprocess_kernel<D>, rows * (D / 8), 256);
  attn_bwd_preprocess_kernel<D><<<g, 256, 0, st>>>(p, o, dout, delta, dq_acc, acc_elems, clear,
                                                   n_clear);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_finalize(const Problem& p, const float* acc, size_t slab_elems, int split,
                               int n_split, __nv_bfloat16* dq, __nv_bfloat16* dk,
                               __nv_bfloat16* dv, cudaStream_t st) {
  const size_t chunks = static_cast<size_t>(p.batch) * p.rows_total * p.heads_q * (D / 8);
  // two waves measured faster than one for the dense finalize (causal B 8, H 32, S 1024,
  // D 64: 20.0 vs 21.1 us)
  const int g = resident_grid(attn_dq_finalize_kernel<D>, chunks, 256, 2);
  attn_dq_finalize_kernel<D><<<g, 256, 0, st>>>(p, acc, slab_elems, split, n_split, 128, dq,
                                                        dk, dv);
  return cudaGetLastError();
}

template cudaError_t launch_bwd_preprocess<64>(const Problem&, const __nv_bfloat16*,
                                               const __nv_bfloat16*, float*, float*, size_t,
                                               float*, size_t, cudaStream_t);
template cudaError_t launch_bwd_preprocess<128>(const Problem&, const __nv_bfloat16*,
                                                const __nv_bfloat16*, float*, float*, size_t,
                                                float*, size_t, cudaStream_t);
template cudaError_t launch_dq_finalize<64>(const Problem&, const float*, size_t, int, int,
                                            __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*,
                                            cudaStream_t);
template cudaError_t launch_dq_finalize<128>(const Problem&, const float*, size_t, int, int,
                                             __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*,
                                             cudaStream_t);

}  // namespace attn
