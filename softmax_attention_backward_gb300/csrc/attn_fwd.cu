// Dense / GQA / THD attention forward with the row log-sum-exp saved for the
// backward (the `flashattn_fwd` stage of "[Example] Introduce split+sum
// template, and optimize atomic_add performance for bwd examples",
// tile-ai/tilelang #940, code-graph section).
//
// One CTA owns two 128-row query tiles of one (batch, query head) and streams
// 128-row K/V tiles through a TMA ring:
//   warp 8        TMA producer (Q once, then K_j, V_j into the ring)
//   warps 9, 10   MMA issuers, one per query tile w: S_w = Q_w K_j^T (both
//                 operands in shared memory) and O_w += P_w V_j with P_w read
//                 from TMEM (it overwrites the first 64 columns of S_w as
//                 packed bf16 pairs); accumulators S0, S1, O0, O1 in TMEM
//                 (512 columns for D = 128)
//   warps 0..3    softmax for query tile 0, warps 4..7 for query tile 1: each
//                 thread owns one row (TMEM lane), runs the online softmax in
//                 the log2 domain, rescales its O row in TMEM when the running
//                 max grew by more than 2^8, and stores P back into TMEM.
// A single issuing thread needs ~100 cycles per tcgen05.mma, so each query
// tile has its own issuer; the two tiles alternate on the tensor core, one
// tile's softmax overlapping the other tile's MMAs.  Each issuer runs
// S_w(j), [P_w(j) ready] PV_w(j), S_w(j+1), ...: MMAs from one thread execute
// in order, so S_w(j+1) never overwrites P_w(j) before PV_w(j) has read it,
// and a completed S_w(j+1) also means O_w holds every PV_w up to j.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                   // rows per query tile
  static constexpr int BN = 128;                   // rows per key/value tile
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int NSLOT = (D == 128) ? 4 : 6; // K/V ring slots
  static constexpr int SMEM = 2 * Q_BYTES + NSLOT * KV_BYTES + 1024;
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
};

template <int D>
__global__ void __launch_bounds__(352, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int PANELS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // 2 tiles
  uint8_t* sRing = sQ + 2 * C::Q_BYTES;                 // NSLOT tiles

  __shared__ uint64_t bar_q, bar_full[C::NSLOT], bar_empty[C::NSLOT];
  __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const Problem& p = a.p;
  const int warp = warp_id();
  AbortCtx ac{&abort_flag, p.err};

  // ---- work decode ---------------------------------------------------------
  SeqRef seq;
  int pair;
  const int h = blockIdx.y;
  if (!decode_tile(p, blockIdx.x, blockIdx.z, 2 * C::BM, seq, pair)) return;
  {
    // heaviest (last) pairs first under causal masking
    const int npairs = (seq.len + 2 * C::BM - 1) / (2 * C::BM);
    if (p.causal) pair = npairs - 1 - pair;
  }
  const int hk = h / (p.heads_q / p.heads_kv);
  const int m0 = pair * 2 * C::BM;
  int n_w[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const int r0 = m0 + w * C::BM;
    if (r0 >= seq.len) {
      n_w[w] = 0;
    } else {
      const int kv_end = p.causal ? min(seq.len, r0 + C::BM) : seq.len;
      n_w[w] = (kv_end + C::BN - 1) / C::BN;
    }
  }
  const int n_kv = max(n_w[0], n_w[1]);

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 2);       // released by both issuers
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bar_s[w], 1);
      mbar_init(&bar_p[w], 128);
      mbar_init(&bar_o[w], 1);
    }
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane_id() == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int row_base = seq.row0;
      mbar_arrive_expect_tx(&bar_q, 2 * C::Q_BYTES);
      for (int w = 0; w < 2; ++w)
        for (int pn = 0; pn < PANELS; ++pn)
          tma_load_4d(&tmQ, &bar_q, sQ + w * C::Q_BYTES + pn * C::BM * 128, pn * 64, h,
                      row_base + m0 + w * C::BM, seq.b);
      for (int i = 0; i < 2 * n_kv; ++i) {
        const int slot = i % C::NSLOT;
        const int use = i / C::NSLOT;
        if (!mbar_wait(&bar_empty[slot], (use & 1) ^ 1, ac)) break;
        const CUtensorMap* m = (i & 1) ? &tmV : &tmK;
        uint8_t* dst = sRing + slot * C::KV_BYTES;
        mbar_arrive_expect_tx(&bar_full[slot], C::KV_BYTES);
        for (int pn = 0; pn < PANELS; ++pn)
          tma_load_4d(m, &bar_full[slot], dst + pn * C::BN * 128, pn * 64, hk,
                      row_base + (i >> 1) * C::BN, seq.b);
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ---------------- MMA issuer of query tile w ----------------
    const int w = warp - 9;
    if (lane_id() == 0) {
      const uint32_t idS = idesc_bf16(C::BM, C::BN, false, false);
      const uint32_t idO = idesc_bf16(C::BM, D, false, true);
      const uint64_t dQw = desc_kmajor_base(smem_u32(sQ + w * C::Q_BYTES));
      const uint64_t dR_k0 = desc_kmajor_base(smem_u32(sRing));
      const uint64_t dR_mn0 = desc_mnmajor_base(smem_u32(sRing), C::BN);
      const uint32_t tS = tmem + (w ? C::COL_S1 : C::COL_S0);
      const uint32_t tO = tmem + (w ? C::COL_O1 : C::COL_O0);
      const int nt = n_w[w];
      bool ok = mbar_wait(&bar_q, 0, ac);
      // this tile stops after nt key tiles, but every ring slot up to n_kv must
      // still be released twice
      for (int j = 0; ok && j < n_kv; ++j) {
        const int ik = 2 * j, iv = 2 * j + 1;
        const int sk = ik % C::NSLOT, sv = iv % C::NSLOT;
        if (j >= nt) {                      // release without using
          if (!mbar_wait(&bar_full[sk], (ik / C::NSLOT) & 1, ac)) break;
          mbar_arrive(&bar_empty[sk]);
          if (!mbar_wait(&bar_full[sv], (iv / C::NSLOT) & 1, ac)) break;
          mbar_arrive(&bar_empty[sv]);
          continue;
        }
        if (!mbar_wait(&bar_full[sk], (ik / C::NSLOT) & 1, ac)) break;
        tc_fence_after();
        const uint64_t kd = desc_advance(dR_k0, sk * C::KV_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tS, desc_advance(dQw, kmajor_step_bytes(C::BM, k)),
                  desc_advance(kd, kmajor_step_bytes(C::BN, k)), idS, k > 0);
        umma_commit(&bar_s[w]);
        umma_commit(&bar_empty[sk]);
        if (!mbar_wait(&bar_full[sv], (iv / C::NSLOT) & 1, ac)) break;
        if (!mbar_wait(&bar_p[w], j & 1, ac)) break;
        tc_fence_after();
        const uint64_t vd = desc_advance(dR_mn0, sv * C::KV_BYTES);
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k)   // P: 8 packed columns per 16 keys
          umma_ts(tO, tS + 8 * k, desc_advance(vd, mnmajor_step_bytes(k)), idO,
                  (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_o[w]);
        umma_commit(&bar_empty[sv]);
      }
    }
  } else {
    // ---------------- softmax warpgroups ----------------
    const int w = warp >> 2;                 // query tile of this warpgroup
    const int t = threadIdx.x & 127;         // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_base + (w ? C::COL_O1 : C::COL_O0);
    const int row = m0 + w * C::BM + t;      // row inside the sequence
    const int nt = n_w[w];
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // S_w(j) complete also means PV_w(j-1) is complete (same issuer, in order)
      if (!mbar_wait(&bar_s[w], j & 1, ac)) { ok = false; break; }
      tc_fence_after();
      float s[C::BN];
      {
        uint32_t u[C::BN];
#pragma unroll
        for (int c = 0; c < C::BN; c += 32) tmem_ld32_nowait(tS + c, u + c);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < C::BN; ++c) s[c] = __uint_as_float(u[c]);
      }
      const int kv0 = j * C::BN;
      const bool need_mask =
          (kv0 + C::BN > seq.len) || (p.causal && kv0 + C::BN - 1 > m0 + w * C::BM);
      if (need_mask) {
        const int lim = p.causal ? min(seq.len - 1, row) : seq.len - 1;
#pragma unroll
        for (int c = 0; c < C::BN; ++c)
          if (kv0 + c > lim) s[c] = -INFINITY;
      }
      // row max with independent partial maxima (short dependency chains)
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
      for (int c = 8; c < C::BN; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      const float m_new = fmaxf(m_run, mt);
      const bool grow = m_new > m_run + 8.0f;          // also true on the first finite max
      const float m_use = grow ? m_new : m_run;
      const float alpha = grow ? ex2(m_run - m_use) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      const bool warp_rescale = j > 0 && __any_sync(0xffffffffu, grow);
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[C::BN / 2];
#pragma unroll
      for (int c = 0; c < C::BN; c += 2) {
        const float p0 = ex2(fmaf(s[c], sl2, -msub));
        const float p1 = ex2(fmaf(s[c + 1], sl2, -msub));
        rsum[(c >> 1) & 3] += p0 + p1;
        pk[c / 2] = pack_bf16(p0, p1);
      }
      l_run = l_run * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
      m_run = m_use;
      if (warp_rescale) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t r[32];
          tmem_ld32_nowait(tO + c, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + c, r);
        }
      }
      // P (bf16 pairs) into the first 64 columns of this row's S
      tmem_st32(tS, pk);
      tmem_st32(tS + 32, pk + 32);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_p[w]);
    }
    // ---- epilogue: O / l, LSE ----
    if (ok && nt > 0 && mbar_wait(&bar_o[w], (nt - 1) & 1, ac)) {
      tc_fence_after();
      const bool valid = row < seq.len;
      const float inv_l = (l_run > 0.f) ? 1.0f / l_run : 0.f;
      const size_t grow_idx = (static_cast<size_t>(seq.b) * p.rows_total + seq.row0 + row);
      __nv_bfloat16* orow = a.o + (grow_idx * p.heads_q + h) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32_nowait(tO + c, r);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[i + 0]) * inv_l, __uint_as_float(r[i + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(r[i + 2]) * inv_l, __uint_as_float(r[i + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(r[i + 4]) * inv_l, __uint_as_float(r[i + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(r[i + 6]) * inv_l, __uint_as_float(r[i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c + i) = v;
          }
        }
      }
      if (valid) {
        const float lse = (l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
        size_t li;
        if (p.cu_seqlens)
          li = static_cast<size_t>(h) * p.rows_total + seq.row0 + row;
        else
          li = (static_cast<size_t>(seq.b) * p.heads_q + h) * p.rows_total + row;
        a.lse[li] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
}

// THD padding rows [cu_seqlens[num_seqs], capacity): O = 0, LSE = -inf.
__global__ void thd_fwd_pad_kernel(Problem p, __nv_bfloat16* o, float* lse, int head_dim) {
  const int end = valid_end(p);
  const int rows = p.rows_total - end;
  if (rows <= 0) return;
  const size_t n_o = static_cast<size_t>(rows) * p.heads_q * head_dim / 8;  // uint4 chunks
  uint4* o4 = reinterpret_cast<uint4*>(o + static_cast<size_t>(end) * p.heads_q * head_dim);
  for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_o; i += gridDim.x * blockDim.x)
    o4[i] = make_uint4(0, 0, 0, 0);
  const size_t n_l = static_cast<size_t>(rows) * p.heads_q;
  for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_l; i += gridDim.x * blockDim.x) {
    const size_t hh = i / rows, r = i % rows;
    lse[hh * p.rows_total + end + r] = -INFINITY;
  }
}

template <int D>
cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x, cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = attn_fwd_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(grid_x, a.p.heads_q, a.p.batch);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(q, k, v, a);
  return cudaGetLastError();
}

template cudaError_t launch_attn_fwd<64>(const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const FwdArgs&, int, cudaStream_t);
template cudaError_t launch_attn_fwd<128>(const CUtensorMap&, const CUtensorMap&,
                                          const CUtensorMap&, const FwdArgs&, int, cudaStream_t);

cudaError_t launch_thd_fwd_pad(const Problem& p, __nv_bfloat16* o, float* lse, int head_dim,
                               cudaStream_t st) {
  thd_fwd_pad_kernel<<<304, 256, 0, st>>>(p, o, lse, head_dim);
  return cudaGetLastError();
}

}  // namespace attn
