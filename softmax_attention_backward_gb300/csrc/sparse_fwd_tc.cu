// Top-k sparse attention forward on tcgen05 (SparseMLA style, "[2/2] Add
// TileLang fused DSA kernels support with THD and CP", Megatron-LM #5049:
// one shared KV head, dim 576 = 512 latent + 64 rope, v_channels 512, -1 for
// empty top-k slots).
//
// Work item = one token t and a block of 64 query heads (H = 16 / 32 use the
// block with zero query rows; H = 128 takes two blocks).  The token's key rows
// are gathered 64 slots at a time with 16-byte cp.async into the 128-byte
// swizzled K-major layout the MMA reads, double-buffered, and every chunk
// feeds two GEMMs:
//   S   = Q K^T     M = 64 heads, N = 64 slots, K = 576   (TMEM, two buffers)
//   O^T += V^T P^T  M = 128 value dims (four tiles), N = 64 heads, K = 64 slots
// The second GEMM keeps the 512 x 64 fp32 output in 256 TMEM columns (as O
// with 64 rows it would need all 512 columns); V^T is the gathered chunk read
// as an MN-major operand and P^T comes from a bf16 tile the softmax warps
// write to shared memory.  The softmax runs online in the log2 domain with a
// stale-max threshold of 2^8: when a head's running max grows by more, the
// softmax warps rescale that head's column of the four O^T tiles in TMEM.
// An M = 64 accumulator keeps row r in TMEM lane 32 (r / 16) + r % 16.
//
// Warp roles (256 threads): 0..3 softmax and epilogue (lanes 0..15 of each
// warp own one head row of S; all 32 lanes own one value dim per O^T tile),
// 4, 5 and 7 gather producers, 6 MMA issuer.  Every wait is a bounded
// mbarrier wait; the softmax warps exchange rescale factors through an
// mbarrier as well, not a hardware barrier.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

namespace {

constexpr int SF_HB = 64;                      // heads per item (M of the S GEMM)
constexpr int SF_NK = 64;                      // key slots per chunk
constexpr int SF_DQK = 576, SF_DV = 512;
constexpr int SF_Q_BYTES = SF_HB * SF_DQK * 2;
constexpr int SF_KV_BYTES = SF_NK * SF_DQK * 2;
constexpr int SF_P_BYTES = SF_HB * SF_NK * 2;
constexpr int SF_SMEM = SF_Q_BYTES + 2 * SF_KV_BYTES + SF_P_BYTES + 1024;
constexpr int SF_THREADS = 256;
constexpr int SF_PRODUCERS = 96;               // threads of warps 4, 5 and 7
constexpr int SF_GATHER_PER_WARP = SF_NK * (SF_DQK / 8) / 3;   // 16-byte copies per chunk and warp
constexpr int SF_GATHER_ROWS = 22;             // key rows one warp's copies touch
static_assert(SF_GATHER_PER_WARP % 32 == 0, "whole warp iterations");
// first row and number of rows of producer warp w's copies
constexpr int sf_gather_row0(int w) { return SF_GATHER_PER_WARP * w / (SF_DQK / 8); }
constexpr int sf_gather_rows(int w) {
  return (SF_GATHER_PER_WARP * (w + 1) - 1) / (SF_DQK / 8) - sf_gather_row0(w) + 1;
}
static_assert(sf_gather_rows(0) <= SF_GATHER_ROWS && sf_gather_rows(1) <= SF_GATHER_ROWS &&
                  sf_gather_rows(2) <= SF_GATHER_ROWS && sf_gather_row0(2) + SF_GATHER_ROWS <= SF_NK,
              "each warp's copies stay within the rows its lanes hold");
constexpr uint32_t SF_TMEM_COLS = 512;
constexpr uint32_t SF_COL_S = 0;               // two S buffers of 64 columns
constexpr uint32_t SF_COL_O = 128;             // four O^T tiles of 64 columns

// Byte offset of 16-byte chunk `ch` (0..71) of row `row` in a tile of `rows`
// rows stored as 64-column SW128 panels.
__device__ __forceinline__ uint32_t sf_off(int row, int ch, int rows) {
  return (ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

}  // namespace

__global__ void __launch_bounds__(SF_THREADS, 1) sparse_fwd_tc_kernel(const SparseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = sQ + SF_Q_BYTES;                // 2 chunk buffers
  uint8_t* sP = sKV + 2 * SF_KV_BYTES;           // P tile, [head][slot] bf16, K-major

  __shared__ uint64_t bar_q, bar_kv_full[2], bar_kv_empty[2], bar_s_full[2], bar_s_free[2];
  __shared__ uint64_t bar_p_full, bar_o_done, bar_alpha;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ uint32_t s_valid[2][2];             // valid-slot mask of each chunk buffer
  __shared__ float s_alpha[2][SF_HB];
  __shared__ int s_grow[2];
  __shared__ float s_l[SF_HB];
  __shared__ int s_red[SF_THREADS / 32];

  const int t = blockIdx.x;
  const int hb = blockIdx.y * SF_HB;
  const int nh = min(SF_HB, a.H - hb);
  const int warp = warp_id(), lane = lane_id();
  AbortCtx ac{&abort_flag, a.err};

  // chunks up to the last valid slot of this token (all-empty tail chunks are skipped)
  int nchunks;
  {
    const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
    int last = -1;
    for (int s = threadIdx.x; s < a.K; s += SF_THREADS) {
      const int j = __ldg(irow + s);
      if (j >= 0 && j < a.T) last = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    if (lane == 0) s_red[warp] = last;
    if (threadIdx.x == 0) {
      abort_flag = 0;
      mbar_init(&bar_q, SF_PRODUCERS);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bar_kv_full[b], SF_PRODUCERS);
        mbar_init(&bar_kv_empty[b], 1);
        mbar_init(&bar_s_full[b], 1);
        mbar_init(&bar_s_free[b], 128);
      }
      mbar_init(&bar_p_full, 128);
      mbar_init(&bar_o_done, 1);
      mbar_init(&bar_alpha, 128);
      s_grow[0] = s_grow[1] = 0;
      fence_mbar_init();
    }
    if (warp == 6) tmem_alloc(&tmem_base_sh, SF_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int m = -1;
    for (int w = 0; w < SF_THREADS / 32; ++w) m = max(m, s_red[w]);
    nchunks = (m + SF_NK) / SF_NK;
  }
  const uint32_t tmem = tmem_base_sh;

  if (warp == 4 || warp == 5 || warp == 7) {
    // ---------------- gather producers ----------------
    const int pt = (warp == 7) ? 64 + lane : threadIdx.x - 128;   // 0..95
    const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
    // the query block (rows past H are zero)
    {
      const __nv_bfloat16* qb = a.q + (static_cast<size_t>(t) * a.H + hb) * SF_DQK;
      const uint32_t base = smem_u32(sQ);
      for (int id = pt; id < SF_HB * (SF_DQK / 8); id += SF_PRODUCERS) {
        const int r = id / (SF_DQK / 8), ch = id % (SF_DQK / 8);
        const bool v = r < nh;
        const void* src = v ? static_cast<const void*>(qb + r * SF_DQK + ch * 8)
                            : static_cast<const void*>(a.q);
        cp_async16(base + sf_off(r, ch, SF_HB), src, v ? 16u : 0u);
      }
      cp_async_commit();
    }
    bool ok = true;
    auto issue_chunk = [&](int c) -> bool {
      const int b = c & 1;
      // buffer b was last read by the O^T GEMM of chunk c - 2 (warp-uniform
      // answer: the lanes exchange indices below)
      if (!mbar_wait_w(&bar_kv_empty[b], ((c >> 1) & 1) ^ 1, ac)) return false;
      if (pt < SF_NK) {
        // slot pt of the chunk: range check, and one word of the valid mask per warp
        const int slot = c * SF_NK + pt;
        const int j = (slot < a.K) ? __ldg(irow + slot) : -1;
        const bool valid = j >= 0 && j < a.T;
        if (!valid && j != -1 && a.err) atomicOr(a.err, ATTN_DEVERR_INDEX_RANGE);
        const uint32_t m32 = __ballot_sync(0xffffffffu, valid);
        if ((pt & 31) == 0) s_valid[b][pt >> 5] = m32;
      }
      // Producer warp pw takes copies [SF_GATHER_PER_WARP * pw, + SF_GATHER_PER_WARP) of
      // the chunk in (row, 16-byte column) order.  Its lanes first load the key
      // row indices of the (at most SF_GATHER_ROWS) rows those copies touch, once;
      // each copy then takes its row's index by a shuffle.  The 48 copies of a
      // lane are fully unrolled: the gather is issue-bound, and it runs faster
      // the more copies go out back to back.
      const uint32_t base = smem_u32(sKV + b * SF_KV_BYTES);
      const int pw = pt >> 5;
      const int e0 = pw * SF_GATHER_PER_WARP, r0 = e0 / (SF_DQK / 8);
      int jl = -1;
      if (lane < SF_GATHER_ROWS) {
        const int slot = c * SF_NK + r0 + lane;
        jl = (slot < a.K) ? __ldg(irow + slot) : -1;
        if (jl >= a.T) jl = -1;
      }
#pragma unroll
      for (int k = 0; k < SF_GATHER_PER_WARP / 32; ++k) {
        const int id = e0 + 32 * k + lane;
        const int r = id / (SF_DQK / 8), ch = id - r * (SF_DQK / 8);
        const int j = __shfl_sync(0xffffffffu, jl, r - r0);
        const void* src = (j >= 0) ? static_cast<const void*>(a.kv + static_cast<size_t>(j) * SF_DQK + ch * 8)
                                   : static_cast<const void*>(a.kv);
        cp_async16(base + sf_off(r, ch, SF_NK), src, (j >= 0) ? 16u : 0u);
      }
      cp_async_commit();
      return true;
    };
    // a chunk (and the query block with chunk 0) is published as soon as its
    // copies landed; the next chunk's copies start right after, while the
    // MMAs and the softmax work on the published one.  (Issuing chunk c + 1
    // before publishing chunk c would wait for the O^T GEMM of chunk c - 1,
    // which the issuer only starts after S of chunk c.)
    for (int c = 0; ok && c < nchunks; ++c) {
      if (!issue_chunk(c)) { ok = false; break; }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      if (c == 0) mbar_arrive(&bar_q);
      mbar_arrive(&bar_kv_full[c & 1]);
    }
    cp_async_wait<0>();
  } else if (warp == 6) {
    // ---------------- MMA issuer ----------------
    if (nchunks > 0) {   // warp-uniform: one elected lane issues
      const uint32_t idS = idesc_bf16(64, SF_NK, false, false);
      const uint32_t idO = idesc_bf16(128, SF_HB, true, false);
      const uint64_t dQ = desc_kmajor_base(smem_u32(sQ));
      const uint64_t dP = desc_kmajor_base(smem_u32(sP));
      auto issue_o = [&](int c) {
        // O^T(m) += V^T(dims 128m..) P^T, P of chunk c from shared memory
        tc_fence_after();
        const int b = c & 1;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint64_t dV = desc_mnmajor_base(smem_u32(sKV + b * SF_KV_BYTES + 2 * m * SF_NK * 128), SF_NK);
#pragma unroll
          for (int kk = 0; kk < SF_NK / 16; ++kk)
            umma_ss_w(tmem + SF_COL_O + 64 * m, desc_advance(dV, mnmajor_step_bytes(kk)),
                    desc_advance(dP, kmajor_step_bytes(SF_HB, kk)), idO, (c > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_w(&bar_o_done);
        umma_commit_w(&bar_kv_empty[b]);
      };
      auto issue_s = [&](int c) {
        tc_fence_after();
        const int b = c & 1;
        const uint64_t dK = desc_kmajor_base(smem_u32(sKV + b * SF_KV_BYTES));
#pragma unroll 4
        for (int kk = 0; kk < SF_DQK / 16; ++kk)
          umma_ss_w(tmem + SF_COL_S + 64 * b, desc_advance(dQ, kmajor_step_bytes(SF_HB, kk)),
                  desc_advance(dK, kmajor_step_bytes(SF_NK, kk)), idS, kk > 0);
        umma_commit_w(&bar_s_full[b]);
      };
      // Issue in readiness order: O^T of chunk `no` as soon as its P is
      // written (that frees its buffer for the gather two chunks ahead), S of
      // chunk `ns` as soon as the chunk landed and its TMEM buffer was read,
      // so S of the next chunk overlaps the softmax of the current one.
      bool ok = mbar_wait_w(&bar_q, 0, ac);
      int ns = 0, no = 0;
      uint64_t t0 = 0;
      while (ok && no < nchunks) {
        bool did = false;
        if (no < ns && mbar_test_wait_w(smem_u32(&bar_p_full), no & 1)) {
          issue_o(no++);
          did = true;
        } else if (ns < nchunks &&
                   mbar_test_wait_w(smem_u32(&bar_kv_full[ns & 1]), (ns >> 1) & 1) &&
                   mbar_test_wait_w(smem_u32(&bar_s_free[ns & 1]), ((ns >> 1) & 1) ^ 1)) {
          issue_s(ns++);
          did = true;
        }
        if (did) {
          t0 = 0;
        } else {
          // lane 0 decides for the warp, which stays converged
          if (t0 == 0) t0 = globaltimer();
          if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&abort_flag), 0)) {
            ok = false;
            break;
          }
          if (__shfl_sync(0xffffffffu, (globaltimer() - t0 > kWaitLimitNs) ? 1 : 0, 0)) {
            raise_error(ac, ATTN_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
        }
      }
    }
  } else if (warp < 4) {
    // ---------------- softmax and epilogue ----------------
    const int q = warp;
    const bool active = lane < 16;
    const int row = 16 * q + (lane & 15);          // head row of S held by this lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      if (!mbar_wait(&bar_s_full[b], (c >> 1) & 1, ac)) { ok = false; break; }
      // (the gather of this chunk, and so its valid-slot mask, is complete)
      if (!mbar_wait(&bar_kv_full[b], (c >> 1) & 1, ac)) { ok = false; break; }
      tc_fence_after();
      uint32_t u[64];
      tmem_ld32_nowait(tmem + lane_base + SF_COL_S + 64 * b, u);
      tmem_ld32_nowait(tmem + lane_base + SF_COL_S + 64 * b + 32, u + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_s_free[b]);
      const unsigned long long vm =
          static_cast<unsigned long long>(s_valid[b][0]) | (static_cast<unsigned long long>(s_valid[b][1]) << 32);
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 64; ++cc) {
        if (!((vm >> cc) & 1ull)) u[cc] = 0xff800000u;   // empty slot: -inf
        mx = fmaxf(mx, __uint_as_float(u[cc]));
      }
      const float mt = mx * sl2;
      const float m_new = fmaxf(m_run, mt);
      const bool grow = active && m_new > m_run + 8.0f;  // also true on the first finite max
      const float m_use = grow ? m_new : m_run;
      const float alpha = grow ? ex2(m_run - m_use) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      // P = 2^(S c - m) as bf16 pairs, row sum
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t nm2 = f2_pack(-msub, -msub);
      uint64_t rs2[2] = {0ull, 0ull};
      uint32_t pk[32];
#pragma unroll
      for (int cc = 0; cc < 64; cc += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(u[cc]), __uint_as_float(u[cc + 1])), sl2x2, nm2),
                  x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        rs2[(cc >> 1) & 1] = f2_add(rs2[(cc >> 1) & 1], f2_pack(p0, p1));
        pk[cc / 2] = pack_bf16(p0, p1);
      }
      float r0, r1, r2, r3;
      f2_unpack(rs2[0], r0, r1);
      f2_unpack(rs2[1], r2, r3);
      // O^T(c-1) must be done before P is overwritten and before O^T is rescaled
      if (c > 0) {
        if (!mbar_wait(&bar_o_done, (c - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
      }
      // exchange the per-head rescale factors of this chunk through shared
      // memory (double-buffered by chunk parity) and a bounded mbarrier wait;
      // the O^T columns of heads whose max grew are rescaled by all 128 threads
      if (active) s_alpha[b][row] = alpha;
      if (c > 0 && grow) s_grow[b] = c + 1;
      mbar_arrive(&bar_alpha);
      if (!mbar_wait(&bar_alpha, c & 1, ac)) { ok = false; break; }
      if (s_grow[b] == c + 1) {
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
#pragma unroll
          for (int h0 = 0; h0 < SF_HB; h0 += 32) {
            uint32_t o[32];
            tmem_ld32_nowait(tmem + lane_base + SF_COL_O + 64 * m + h0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * s_alpha[b][h0 + i]);
            tmem_st32(tmem + lane_base + SF_COL_O + 64 * m + h0, o);
          }
        }
        tmem_wait_st();
      }
      if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint4*>(sP + row * 128 + ((i ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        l_run = l_run * alpha + ((r0 + r1) + (r2 + r3));
        m_run = m_use;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full);
    }
    // ---- epilogue: O = O^T / l (transposed back), LSE ----
    if (ok) {
      if (active) s_l[row] = l_run;
      if (active && row < nh)
        a.lse[static_cast<size_t>(t) * a.H + hb + row] =
            l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      mbar_arrive(&bar_alpha);
      const bool synced = mbar_wait(&bar_alpha, nchunks & 1, ac);
      const bool have_o = synced && nchunks > 0 && mbar_wait(&bar_o_done, (nchunks - 1) & 1, ac);
      tc_fence_after();
      __nv_bfloat16* obase = a.o + (static_cast<size_t>(t) * a.H + hb) * SF_DV;
#pragma unroll 1
      for (int m = 0; synced && m < 4; ++m) {
        const int d = 128 * m + 32 * q + lane;          // value dim of this lane
#pragma unroll
        for (int h0 = 0; h0 < SF_HB; h0 += 32) {
          uint32_t o[32];
          if (have_o) {
            tmem_ld32_nowait(tmem + lane_base + SF_COL_O + 64 * m + h0, o);
            tmem_wait_ld();
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int h = h0 + i;
            if (h < nh) {
              const float l = s_l[h];
              const float v = (have_o && l > 0.f) ? __uint_as_float(o[i]) / l : 0.f;
              obase[static_cast<size_t>(h) * SF_DV + d] = __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, SF_TMEM_COLS);
    tmem_relinquish();
  }
}

cudaError_t launch_sparse_fwd(const SparseArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(sparse_fwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SF_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.T, (a.H + SF_HB - 1) / SF_HB);
  sparse_fwd_tc_kernel<<<grid, SF_THREADS, SF_SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
