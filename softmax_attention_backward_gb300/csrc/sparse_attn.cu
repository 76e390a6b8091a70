// Top-k sparse attention over one shared KV head (SparseMLA style, "[2/2] Add
// TileLang fused DSA kernels support with THD and CP", Megatron-LM #5049:
// sparse MLA forward/backward with preprocess/postprocess, dim 576 =
// 512 latent + 64 rope, v_channels 512, -1 for empty top-k slots).
//
// Backward (the forward runs on tcgen05, sparse_fwd_tc.cu).  One CTA per
// (token, block of 64 query heads).  The token's key rows are gathered 32 at
// a time with 16-byte cp.async into a double-buffered, XOR-swizzled shared
// tile, so all heads share one gather.  The contractions are warp-level
// tensor-core tiles (m16n8k16, bf16 in, fp32 out):
//   backward: P = exp(S - LSE), dP = dO V^T, dS = P (dP - Delta) * scale,
//             dQ += dS K (registers, stored once per token),
//             dKV[idx] += dS^T Q (576 dims) + P^T dO (first 512 dims) with
//             fp32 vector atomics; a final pass casts dKV to bf16.
#include <cuda_runtime.h>

#include "launch.h"
#include "mma_sm80.cuh"

namespace attn {

constexpr int SP_DQK = 576;
constexpr int SP_DV = 512;
constexpr int SP_HB = 64;   // heads per CTA
constexpr int SP_BN = 32;   // key rows per gathered chunk
constexpr int SP_PSTR = 40; // padded row (elements) of the P / dS tiles

// Loads the slot indices of chunk `c` and gathers the selected rows.
template <int NTHREADS>
__device__ __forceinline__ void sparse_gather(const SparseArgs& a, int t, int c, uint8_t* dst,
                                              int* s_idx) {
  const int tid = threadIdx.x;
  const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
  const uint32_t dbase = smem_u32(dst);
  for (int id = tid; id < SP_BN * (SP_DQK / 8); id += NTHREADS) {
    const int row = id / (SP_DQK / 8);
    const int ch = id % (SP_DQK / 8);
    const int slot = c * SP_BN + row;
    int j = (slot < a.K) ? __ldg(irow + slot) : -1;
    const bool valid = j >= 0 && j < a.T;
    const void* src = valid ? static_cast<const void*>(a.kv + static_cast<size_t>(j) * SP_DQK + ch * 8)
                            : static_cast<const void*>(a.kv);
    cp_async16(dbase + swz<SP_DQK>(row, ch * 8), src, valid ? 16u : 0u);
    if (ch == 0) {
      if (!valid && j != -1 && a.err) atomicOr(a.err, ATTN_DEVERR_INDEX_RANGE);
      s_idx[row] = valid ? j : -1;
    }
  }
}

// Index of the last chunk holding a valid slot, plus one (block-wide).
template <int NTHREADS>
__device__ __forceinline__ int sparse_chunk_count(const SparseArgs& a, int t, int* s_red) {
  const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
  int last = -1;
  for (int s = threadIdx.x; s < a.K; s += NTHREADS) {
    const int j = __ldg(irow + s);
    if (j >= 0 && j < a.T) last = s;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = last;
  __syncthreads();
  int m = -1;
  for (int w = 0; w < NTHREADS / 32; ++w) m = max(m, s_red[w]);
  __syncthreads();
  return (m + SP_BN) / SP_BN;
}

// Loads `rows` x `cols` bf16 rows of a [*, ld] tensor into a swizzled tile;
// rows >= nvalid are zero-filled.
template <int COLS, int NTHREADS>
__device__ __forceinline__ void load_rows(const __nv_bfloat16* src, size_t ld, int rows,
                                          int nvalid, uint8_t* dst) {
  const uint32_t dbase = smem_u32(dst);
  for (int id = threadIdx.x; id < rows * (COLS / 8); id += NTHREADS) {
    const int r = id / (COLS / 8), ch = id % (COLS / 8);
    const bool v = r < nvalid;
    const void* s = v ? static_cast<const void*>(src + r * ld + ch * 8) : static_cast<const void*>(src);
    cp_async16(dbase + swz<COLS>(r, ch * 8), s, v ? 16u : 0u);
  }
}

// ============================================================================
// Backward
// ============================================================================
constexpr int SPB_THREADS = 512;
constexpr int SPB_SMEM = SP_HB * SP_DQK * 2 + SP_HB * SP_DV * 2 + 2 * SP_BN * SP_DQK * 2 +
                         2 * SP_HB * SP_PSTR * 2 + 128;

__global__ void __launch_bounds__(SPB_THREADS, 1) sparse_bwd_kernel(const SparseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + SP_HB * SP_DQK * 2;
  uint8_t* sKV = sdO + SP_HB * SP_DV * 2;                 // 2 buffers
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(sKV + 2 * SP_BN * SP_DQK * 2);
  __nv_bfloat16* sdS = sP + SP_HB * SP_PSTR;
  __shared__ int s_idx[2][SP_BN];
  __shared__ float s_lse[SP_HB], s_delta[SP_HB];
  __shared__ int s_red[SPB_THREADS / 32];

  const int t = blockIdx.x;
  const int hb = blockIdx.y * SP_HB;
  const int nh = min(SP_HB, a.H - hb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const float sl2 = a.scale_log2;
  const float scale = a.scale;

  const int nchunks = sparse_chunk_count<SPB_THREADS>(a, t, s_red);

  if (threadIdx.x < SP_HB) {
    const int h = threadIdx.x;
    float l = INFINITY, d = 0.f;
    if (h < nh) {
      const float lv = __ldg(a.lse_in + static_cast<size_t>(t) * a.H + hb + h);
      l = (lv == -INFINITY) ? INFINITY : lv * kLog2e;
      d = __ldg(a.delta + static_cast<size_t>(t) * a.H + hb + h);
    }
    s_lse[threadIdx.x] = l;
    s_delta[threadIdx.x] = d;
  }
  load_rows<SP_DQK, SPB_THREADS>(a.q + (static_cast<size_t>(t) * a.H + hb) * SP_DQK, SP_DQK,
                                 SP_HB, nh, sQ);
  load_rows<SP_DV, SPB_THREADS>(a.dout + (static_cast<size_t>(t) * a.H + hb) * SP_DV, SP_DV,
                                SP_HB, nh, sdO);
  if (nchunks > 0) sparse_gather<SPB_THREADS>(a, t, 0, sKV, s_idx[0]);
  cp_async_commit();

  // dQ accumulators: heads 16*(warp&3).., columns 144*(warp>>2).. (18 n8 tiles)
  const int qg = warp & 3, qc = warp >> 2;
  float dq[18][4];
#pragma unroll
  for (int n = 0; n < 18; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;

  const uint32_t aQ = smem_u32(sQ), adO = smem_u32(sdO), aP = smem_u32(sP), adS = smem_u32(sdS);
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) {
      sparse_gather<SPB_THREADS>(a, t, c + 1, sKV + (buf ^ 1) * SP_BN * SP_DQK * 2, s_idx[buf ^ 1]);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t aK = smem_u32(sKV + buf * SP_BN * SP_DQK * 2);
    // ---- phase A: S and dP for heads 16*(warp&3).., keys 8*(warp>>2).. ----
    {
      const int hg = warp & 3, kq = warp >> 2;
      float s[4] = {0.f, 0.f, 0.f, 0.f}, dp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int k = 0; k < SP_DQK / 16; k += 2) {
        uint32_t bb[4];
        {
          const int n = 8 * kq + (lane & 7);
          const int kk = 16 * k + 8 * (lane >> 3);
          ldsm_x4(aK + swz<SP_DQK>(n, kk), bb[0], bb[1], bb[2], bb[3]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ks = k + u;
          uint32_t af[4];
          const int r = 16 * hg + (lane & 7) + 8 * ((lane >> 3) & 1);
          const int cc = 16 * ks + 8 * (lane >> 4);
          ldsm_x4(aQ + swz<SP_DQK>(r, cc), af[0], af[1], af[2], af[3]);
          const uint32_t b[2] = {bb[2 * u], bb[2 * u + 1]};
          mma_bf16_16816(s, af, b);
          if (ks < SP_DV / 16) {
            uint32_t of[4];
            ldsm_x4(adO + swz<SP_DV>(r, cc), of[0], of[1], of[2], of[3]);
            mma_bf16_16816(dp, of, b);
          }
        }
      }
      float pv[4], dsv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * hg + g + 8 * (e >> 1);
        const int col = 8 * kq + 2 * tq + (e & 1);
        float pe = ex2(fmaf(s[e], sl2, -s_lse[row]));
        if (s_idx[buf][col] < 0) pe = 0.f;
        pv[e] = pe;
        dsv[e] = pe * (dp[e] - s_delta[row]) * scale;
      }
      const int col = 8 * kq + 2 * tq;
      *reinterpret_cast<uint32_t*>(sP + (16 * hg + g) * SP_PSTR + col) = pack_bf16(pv[0], pv[1]);
      *reinterpret_cast<uint32_t*>(sP + (16 * hg + g + 8) * SP_PSTR + col) = pack_bf16(pv[2], pv[3]);
      *reinterpret_cast<uint32_t*>(sdS + (16 * hg + g) * SP_PSTR + col) = pack_bf16(dsv[0], dsv[1]);
      *reinterpret_cast<uint32_t*>(sdS + (16 * hg + g + 8) * SP_PSTR + col) =
          pack_bf16(dsv[2], dsv[3]);
    }
    __syncthreads();
    // ---- phase B1: dQ += dS K ----
#pragma unroll
    for (int kk = 0; kk < SP_BN / 16; ++kk) {
      uint32_t af[4];
      {
        const int r = 16 * qg + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int cc = 16 * kk + 8 * (lane >> 4);
        ldsm_x4(adS + (r * SP_PSTR + cc) * 2, af[0], af[1], af[2], af[3]);
      }
#pragma unroll
      for (int np = 0; np < 9; ++np) {
        uint32_t b0[2], b1[2];
        const int kr = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int n = 144 * qc + 16 * np + 8 * (lane >> 4);
        ldsm_x4_t(aK + swz<SP_DQK>(kr, n), b0[0], b0[1], b1[0], b1[1]);
        mma_bf16_16816(dq[2 * np], af, b0);
        mma_bf16_16816(dq[2 * np + 1], af, b1);
      }
    }
    // ---- phase B2: dKV rows = dS^T Q (+ P^T dO for the first 512 columns) ----
    {
      const int mg = warp & 1;          // 16 key rows
      const int ng = warp >> 1;         // 72 columns
      uint32_t aS[4][4], aPt[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {     // 16 heads per step
        const int sr = 16 * k + (lane & 7) + 8 * (lane >> 4);
        const int sc = 16 * mg + 8 * ((lane >> 3) & 1);
        ldsm_x4_t(adS + (sr * SP_PSTR + sc) * 2, aS[k][0], aS[k][1], aS[k][2], aS[k][3]);
        ldsm_x4_t(aP + (sr * SP_PSTR + sc) * 2, aPt[k][0], aPt[k][1], aPt[k][2], aPt[k][3]);
      }
      const int slot0 = 16 * mg + g;
      const int j0 = s_idx[buf][slot0], j1 = s_idx[buf][slot0 + 8];
#pragma unroll 1
      for (int nt = 0; nt < 9; ++nt) {
        const int n0 = 72 * ng + 8 * nt;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t b[2];
          const int kr = 16 * k + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x2_t(aQ + swz<SP_DQK>(kr, n0), b[0], b[1]);
          mma_bf16_16816(d, aS[k], b);
          if (n0 < SP_DV) {
            ldsm_x2_t(adO + swz<SP_DV>(kr, n0), b[0], b[1]);
            mma_bf16_16816(d, aPt[k], b);
          }
        }
        if (j0 >= 0) red_add_v2(a.dkv_acc + static_cast<size_t>(j0) * SP_DQK + n0 + 2 * tq, d[0], d[1]);
        if (j1 >= 0) red_add_v2(a.dkv_acc + static_cast<size_t>(j1) * SP_DQK + n0 + 2 * tq, d[2], d[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // ---- dQ rows (scale already folded into dS) ----
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = 16 * qg + g + 8 * r;
    if (row >= nh) continue;
    __nv_bfloat16* qrow = a.dq + (static_cast<size_t>(t) * a.H + hb + row) * SP_DQK + 144 * qc;
#pragma unroll
    for (int n = 0; n < 18; ++n)
      *reinterpret_cast<uint32_t*>(qrow + 8 * n + 2 * tq) = pack_bf16(dq[n][2 * r], dq[n][2 * r + 1]);
  }
}

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
  const size_t n4 = static_cast<size_t>(a.T) * SP_DQK / 4;
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
  cudaError_t e = cudaFuncSetAttribute(sparse_bwd_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SPB_SMEM);
  if (e != cudaSuccess) return e;
  const size_t rows = static_cast<size_t>(a.T) * a.H;
  int g = static_cast<int>((rows * 32 + 255) / 256);
  if (g > 152 * 8) g = 152 * 8;
  SparseArgs pa = a;
  sparse_bwd_preprocess_kernel<<<g, 256, 0, st>>>(pa, delta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  pa.delta = delta;
  dim3 grid(a.T, (a.H + SP_HB - 1) / SP_HB);
  sparse_bwd_kernel<<<grid, SPB_THREADS, SPB_SMEM, st>>>(pa);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(a.T) * SP_DQK / 8;
  int gc = static_cast<int>((n8 + 255) / 256);
  if (gc > 152 * 8) gc = 152 * 8;
  sparse_dkv_cast_kernel<<<gc, 256, 0, st>>>(a.dkv_acc, dkv, n8);
  return cudaGetLastError();
}

}  // namespace attn
