// Sparse KL loss of the DSA indexer (the streaming sparse-KL hook of "[2/2] Add
// TileLang fused DSA kernels support with THD and CP & Clean up", Megatron-LM
// #5049).  Formulas and layouts: dsa.h (dsa_sparse_kl).
//
// One CTA per token.  The token's query heads load once per 64-head block; its
// key rows are gathered 64 slots at a time (16-byte cp.async into the SW128
// K-major layout, as in the sparse attention kernels) into two chunk buffers,
// so the gather of one chunk overlaps the MMA of the other, and S = Q K^T runs
// on tcgen05 (M = 64 heads, N = 64 slots, K = 576) into two TMEM buffers.  Four
// warps turn S into the attention probabilities P = exp(scale S - lse) with the
// forward's lse and sum each slot's column over their heads with a
// reduce-scatter of warp shuffles; the four warps' sums meet in shared memory
// and the per-slot total (summed over the head blocks) is kept in the token's
// row of `grad` until the end.  Nothing of size heads x slots leaves the chip.
// After the last chunk the whole CTA forms the softmax of the scores over the
// valid slots, the loss and its gradient (which replaces the kept sums).
#include <cuda_runtime.h>

#include "dsa.h"
#include "launch.h"

namespace attn {
namespace {

constexpr int KL_HB = 64;                       // heads per block
constexpr int KL_NK = 64;                       // slots per chunk
constexpr int KL_DQK = 576;
constexpr int KL_Q_BYTES = KL_HB * KL_DQK * 2;  // 72 KB
constexpr int KL_KV_BYTES = KL_NK * KL_DQK * 2; // 72 KB per chunk buffer
constexpr int KL_SMEM = KL_Q_BYTES + 2 * KL_KV_BYTES + 1024;
constexpr int KL_THREADS = 224;                 // 0..3 softmax / target, 4..5 gather, 6 MMA
constexpr uint32_t KL_TMEM_COLS = 128;          // two S buffers of 64 columns

struct KlArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const float* lse;
  const int32_t* idx;
  const float* scores;
  float* loss;
  float* grad;
  float* target;
  int T, H, K;
  float scale_log2;
  int32_t* err;
};

__device__ __forceinline__ uint32_t kl_off(int row, int ch, int rows) {
  return (ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ float block_reduce(float v, float* s_red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, y) : v + y;
  }
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float r = is_max ? -INFINITY : 0.f;
  for (int w = 0; w < KL_THREADS / 32; ++w) r = is_max ? fmaxf(r, s_red[w]) : r + s_red[w];
  __syncthreads();
  return r;
}

// Sum of v over the 32 lanes of the warp, per column, spread over the lanes:
// five halving rounds (each lane keeps one half of its columns and adds the
// partner's copy of that half), after which lane l holds the sums of columns
// col0(l) and col0(l) + 1.
__device__ __forceinline__ void column_sums(float (&v)[64], int lane) {
#pragma unroll
  for (int o = 16, hs = 32; o >= 1; o >>= 1, hs >>= 1) {
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < hs; ++i) {
      const float send = up ? v[i] : v[i + hs];
      const float keep = up ? v[i + hs] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}
__device__ __forceinline__ int col0_of_lane(int lane) {
  return ((lane >> 4) & 1) * 32 + ((lane >> 3) & 1) * 16 + ((lane >> 2) & 1) * 8 +
         ((lane >> 1) & 1) * 4 + (lane & 1) * 2;
}

__global__ void __launch_bounds__(KL_THREADS, 1) dsa_sparse_kl_kernel(const KlArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + KL_Q_BYTES;               // two chunk buffers
  __shared__ uint64_t bar_kv_full[2], bar_kv_empty[2], bar_s_full[2], bar_s_free[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float s_col[4][KL_NK];             // per softmax warp: column sums of its rows
  __shared__ float s_red[KL_THREADS / 32];
  __shared__ int s_last[KL_THREADS / 32];

  const int t = blockIdx.x;
  const int warp = warp_id(), lane = lane_id();
  AbortCtx ac{&abort_flag, a.err};
  const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
  float* grow = a.grad + static_cast<size_t>(t) * a.K;   // holds the head sums until the end
  const int nhb = (a.H + KL_HB - 1) / KL_HB;

  int nchunks;
  {
    int last = -1;
    for (int s = threadIdx.x; s < a.K; s += KL_THREADS) {
      const int j = __ldg(irow + s);
      if (j >= 0 && j < a.T) last = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    if (lane == 0) s_last[warp] = last;
    if (threadIdx.x == 0) {
      abort_flag = 0;
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bar_kv_full[b], 64);
        mbar_init(&bar_kv_empty[b], 1);
        mbar_init(&bar_s_full[b], 1);
        mbar_init(&bar_s_free[b], 128);
      }
      fence_mbar_init();
    }
    if (warp == 6) tmem_alloc(&tmem_base_sh, KL_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int m = -1;
    for (int w = 0; w < KL_THREADS / 32; ++w) m = max(m, s_last[w]);
    nchunks = (m + KL_NK) / KL_NK;
  }
  const uint32_t tmem = tmem_base_sh;
  const int steps = nchunks * nhb;              // (head block, chunk) steps, head block outer

  if (warp == 4 || warp == 5) {
    // ---------------- producers: a head block's queries, then the chunks ----------------
    const int pt = threadIdx.x - 128;            // 0..63
    for (int st = 0; st < steps; ++st) {
      const int hb = st / nchunks, c = st % nchunks, b = st & 1;
      // buffer b was last read by the S of step st - 2
      if (!mbar_wait_w(&bar_kv_empty[b], ((st >> 1) & 1) ^ 1, ac)) break;
      if (c == 0) {
        // a new head block replaces Q: the S of step st - 1 must be done too
        if (st > 0 && !mbar_wait_w(&bar_kv_empty[(st - 1) & 1], ((st - 1) >> 1) & 1, ac)) break;
        const int h0 = hb * KL_HB, nh = min(KL_HB, a.H - h0);
        const __nv_bfloat16* qb = a.q + (static_cast<size_t>(t) * a.H + h0) * KL_DQK;
        for (int id = pt; id < KL_HB * (KL_DQK / 8); id += 64) {
          const int r = id / (KL_DQK / 8), ch = id % (KL_DQK / 8);
          const bool v = r < nh;
          cp_async16(smem_u32(sQ) + kl_off(r, ch, KL_HB),
                     v ? static_cast<const void*>(qb + r * KL_DQK + ch * 8) : static_cast<const void*>(a.q),
                     v ? 16u : 0u);
        }
      }
      const int slot = c * KL_NK + pt;
      const int j = slot < a.K ? __ldg(irow + slot) : -1;
      const bool valid = j >= 0 && j < a.T;
      if (hb == 0 && !valid && j != -1 && a.err) atomicOr(a.err, ATTN_DEVERR_INDEX_RANGE);
      const int jr = valid ? j : -1;
      const uint32_t base = smem_u32(sKV + b * KL_KV_BYTES);
      const int rw = pt & ~31;
#pragma unroll
      for (int k = 0; k < KL_DQK / 8; ++k) {   // 32 rows x 72 columns / 32 lanes
        const int e = 32 * k + lane;
        const int rl = e / (KL_DQK / 8), ch = e - rl * (KL_DQK / 8);
        const int jj = __shfl_sync(0xffffffffu, jr, rl);
        cp_async16(base + kl_off(rw + rl, ch, KL_NK),
                   jj >= 0 ? static_cast<const void*>(a.kv + static_cast<size_t>(jj) * KL_DQK + ch * 8)
                           : static_cast<const void*>(a.kv),
                   jj >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&bar_kv_full[b]);
    }
    cp_async_wait<0>();
  } else if (warp == 6) {
    // ---------------- MMA issuer: S = Q K^T per step, two TMEM buffers ----------------
    const uint32_t idS = idesc_bf16(64, KL_NK, false, false);
    const uint64_t dQk = desc_kmajor_base(smem_u32(sQ));
    bool ok = true;
    for (int st = 0; ok && st < steps; ++st) {
      const int b = st & 1;
      if (!mbar_wait_w(&bar_kv_full[b], (st >> 1) & 1, ac)) { ok = false; break; }
      if (!mbar_wait_w(&bar_s_free[b], ((st >> 1) & 1) ^ 1, ac)) { ok = false; break; }
      tc_fence_after();
      const uint64_t dKk = desc_kmajor_base(smem_u32(sKV + b * KL_KV_BYTES));
#pragma unroll 4
      for (int kk = 0; kk < KL_DQK / 16; ++kk)
        umma_ss_w(tmem + b * KL_NK, desc_advance(dQk, kmajor_step_bytes(KL_HB, kk)),
                  desc_advance(dKk, kmajor_step_bytes(KL_NK, kk)), idS, kk > 0 ? 1u : 0u);
      umma_commit_w(&bar_s_full[b]);
      umma_commit_w(&bar_kv_empty[b]);
    }
  } else if (warp < 4) {
    // ---------------- P and the per-slot sums over the heads ----------------
    const int qq = warp;
    const bool active = lane < 16;
    const int row = 16 * qq + (lane & 15);       // head row of the block held by this lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * qq) << 16;
    const int col0 = col0_of_lane(lane);
    bool ok = true;
    for (int st = 0; ok && st < steps; ++st) {
      const int hb = st / nchunks, c = st % nchunks, b = st & 1;
      const int h = hb * KL_HB + row;
      const float lse2 = (active && h < a.H) ? __ldg(a.lse + static_cast<size_t>(t) * a.H + h) * kLog2e
                                            : INFINITY;
      // valid slots of the chunk, read by each warp itself (the producer may
      // already be gathering the next chunk)
      const int sl0 = c * KL_NK + lane, sl1 = sl0 + 32;
      const int j0 = sl0 < a.K ? __ldg(irow + sl0) : -1, j1 = sl1 < a.K ? __ldg(irow + sl1) : -1;
      const unsigned long long vm =
          static_cast<unsigned long long>(__ballot_sync(0xffffffffu, j0 >= 0 && j0 < a.T)) |
          (static_cast<unsigned long long>(__ballot_sync(0xffffffffu, j1 >= 0 && j1 < a.T)) << 32);
      if (!mbar_wait(&bar_s_full[b], (st >> 1) & 1, ac)) { ok = false; break; }
      tc_fence_after();
      uint32_t us[64];
      tmem_ld32_nowait(tmem + lane_base + b * KL_NK, us);
      tmem_ld32_nowait(tmem + lane_base + b * KL_NK + 32, us + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_s_free[b]);
      float pv[64];
#pragma unroll
      for (int cc = 0; cc < 64; ++cc) {
        const float p = ex2(fmaf(__uint_as_float(us[cc]), a.scale_log2, -lse2));
        pv[cc] = (active && ((vm >> cc) & 1ull) && lse2 < INFINITY) ? p : 0.f;
      }
      column_sums(pv, lane);
      s_col[qq][col0] = pv[0];
      s_col[qq][col0 + 1] = pv[1];
      named_bar_sync(1, 128);
      if (threadIdx.x < KL_NK) {
        const float sum = s_col[0][threadIdx.x] + s_col[1][threadIdx.x] + s_col[2][threadIdx.x] +
                          s_col[3][threadIdx.x];
        const int slot = c * KL_NK + threadIdx.x;
        if (slot < a.K) grow[slot] = hb == 0 ? sum : grow[slot] + sum;
      }
      named_bar_sync(1, 128);
    }
  }

  // ---------------- loss and gradient over the token's slots (all threads) ----------------
  tc_fence_before();
  __syncthreads();
  const bool ok = *reinterpret_cast<volatile int*>(&abort_flag) == 0;
  const float inv_h = 1.f / static_cast<float>(a.H);
  const float* srow = a.scores + static_cast<size_t>(t) * a.K;
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < a.K; s += KL_THREADS) {
    const int j = __ldg(irow + s);
    if (j >= 0 && j < a.T) mx = fmaxf(mx, __ldg(srow + s));
  }
  mx = block_reduce(mx, s_red, true);
  float z = 0.f;
  for (int s = threadIdx.x; s < a.K; s += KL_THREADS) {
    const int j = __ldg(irow + s);
    if (j >= 0 && j < a.T) z += expf(__ldg(srow + s) - mx);
  }
  z = block_reduce(z, s_red, false);
  const float lnz = mx + logf(z);
  float part = 0.f;
  float* trow = a.target ? a.target + static_cast<size_t>(t) * a.K : nullptr;
  for (int s = threadIdx.x; s < a.K; s += KL_THREADS) {
    const int j = __ldg(irow + s);
    float g = 0.f, p = 0.f;
    if (ok && j >= 0 && j < a.T && s < nchunks * KL_NK) {
      p = grow[s] * inv_h;
      const float lr = __ldg(srow + s) - lnz;
      g = expf(lr) - p;
      if (p > 0.f) part += p * (logf(p) - lr);
    }
    grow[s] = g;
    if (trow) trow[s] = p;
  }
  part = block_reduce(part, s_red, false);
  if (threadIdx.x == 0) a.loss[t] = (ok && nchunks > 0) ? part : 0.f;

  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, KL_TMEM_COLS);
    tmem_relinquish();
  }
}

bool aligned(const void* p, unsigned m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t dsa_sparse_kl(const sparse_attn_problem_t* p, const void* q,
                                       const void* kv, const float* lse, const int32_t* idx,
                                       const float* scores, float* loss, float* grad,
                                       float* target, attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->tokens < 0 || p->heads <= 0 || p->topk <= 0 || !(p->scale == p->scale))
    return ATTN_ERR_INVALID_ARG;
  if (p->dim_qk != KL_DQK || p->dim_v != 512) return ATTN_ERR_UNSUPPORTED;
  if (p->heads != 16 && p->heads != 32 && p->heads != 64 && p->heads != 128)
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->tokens) * p->heads * KL_DQK >= (int64_t(1) << 31) ||
      static_cast<int64_t>(p->tokens) * p->topk >= (int64_t(1) << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (p->tokens == 0) return ATTN_OK;
  if (!q || !kv || !lse || !idx || !scores || !loss || !grad) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(lse, 16) || !aligned(idx, 16) ||
      !aligned(scores, 16) || !aligned(loss, 16) || !aligned(grad, 16) ||
      (target && !aligned(target, 16)))
    return ATTN_ERR_ALIGNMENT;
  KlArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.lse = lse;
  a.idx = idx;
  a.scores = scores;
  a.loss = loss;
  a.grad = grad;
  a.target = target;
  a.T = p->tokens;
  a.H = p->heads;
  a.K = p->topk;
  a.scale_log2 = p->scale * kLog2e;
  a.err = p->error_word;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(dsa_sparse_kl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           KL_SMEM) != cudaSuccess)
    return ATTN_ERR_CUDA;
  dsa_sparse_kl_kernel<<<p->tokens, KL_THREADS, KL_SMEM, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
