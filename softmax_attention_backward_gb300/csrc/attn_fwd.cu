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
//                 from TMEM as packed bf16 pairs (64 columns of its own for
//                 D = 64, the first 64 columns of S_w for D = 128, where S0,
//                 S1, O0, O1 already fill the 512 columns)
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
  static constexpr int NSLOT = (D == 128) ? 5 : 6; // K/V ring slots
  static constexpr int SMEM = 2 * Q_BYTES + NSLOT * KV_BYTES + 1024;
  static constexpr int THREADS = 352;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
  // With D = 64 each tile also gets its own P region (64 packed columns), so
  // S_w(j+1) can be computed while the softmax of tile j runs; with D = 128 P
  // overwrites the first 64 columns of S_w.
  static constexpr bool SEP_P = (256 + 2 * D + 2 * 64 <= 512);
  static constexpr uint32_t COL_P0 = SEP_P ? 256 + 2 * D : COL_S0;
  static constexpr uint32_t COL_P1 = SEP_P ? 256 + 2 * D + 64 : COL_S1;
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
  __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2], bar_sfree[2], bar_stagger;
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
      mbar_init(&bar_sfree[w], 128);
    }
    mbar_init(&bar_stagger, 1);
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
      const uint32_t tP = tmem + (w ? C::COL_P1 : C::COL_P0);
      const int nt = n_w[w];
      bool ok = mbar_wait(&bar_q, 0, ac);
      // Tile 1 starts one softmax phase after tile 0 (when P_0(0) is ready), so
      // that one tile's softmax overlaps the other tile's MMAs instead of both
      // running in lockstep.  bar_stagger completes exactly once.
      if (w == 1 && ok) ok = mbar_wait(&bar_stagger, 0, ac);
      auto issue_s = [&](int j) -> bool {
        const int ik = 2 * j, sk = ik % C::NSLOT;
        if (!mbar_wait(&bar_full[sk], (ik / C::NSLOT) & 1, ac)) return false;
        tc_fence_after();
        const uint64_t kd = desc_advance(dR_k0, sk * C::KV_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tS, desc_advance(dQw, kmajor_step_bytes(C::BM, k)),
                  desc_advance(kd, kmajor_step_bytes(C::BN, k)), idS, k > 0);
        umma_commit(&bar_s[w]);
        umma_commit(&bar_empty[sk]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int iv = 2 * j + 1, sv = iv % C::NSLOT;
        if (!mbar_wait(&bar_full[sv], (iv / C::NSLOT) & 1, ac)) return false;
        if (!mbar_wait(&bar_p[w], j & 1, ac)) return false;
        if (w == 0 && j == 0) mbar_arrive(&bar_stagger);
        tc_fence_after();
        const uint64_t vd = desc_advance(dR_mn0, sv * C::KV_BYTES);
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k)   // P: 8 packed columns per 16 keys
          umma_ts(tO, tP + 8 * k, desc_advance(vd, mnmajor_step_bytes(k)), idO,
                  (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_o[w]);
        umma_commit(&bar_empty[sv]);
        return true;
      };
      // release a ring slot this tile does not use (both issuers release each)
      auto skip = [&](int i) -> bool {
        if (!mbar_wait(&bar_full[i % C::NSLOT], (i / C::NSLOT) & 1, ac)) return false;
        mbar_arrive(&bar_empty[i % C::NSLOT]);
        return true;
      };
      if (C::SEP_P) {
        // S(j+1) as soon as the softmax has read S(j); PV(j) once P(j) is ready
        if (ok && nt > 0) ok = issue_s(0);
        for (int j = 0; ok && j < nt; ++j) {
          if (j + 1 < nt) {
            if (!mbar_wait(&bar_sfree[w], j & 1, ac) || !issue_s(j + 1)) break;
          }
          if (!issue_pv(j)) break;
        }
      } else {
        // S(j), PV(j), S(j+1), ...: MMAs of one thread execute in order, so
        // S(j+1) cannot overwrite P(j) (stored over S) before PV(j) read it
        for (int j = 0; ok && j < nt; ++j)
          if (!issue_s(j) || !issue_pv(j)) ok = false;
      }
      for (int j = nt; ok && j < n_kv; ++j)
        if (!skip(2 * j) || !skip(2 * j + 1)) ok = false;
    }
  } else {
    // ---------------- softmax warpgroups ----------------
    const int w = warp >> 2;                 // query tile of this warpgroup
    const int t = threadIdx.x & 127;         // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_base + (w ? C::COL_O1 : C::COL_O0);
    const uint32_t tP = tmem + lane_base + (w ? C::COL_P1 : C::COL_P0);
    const int row = m0 + w * C::BM + t;      // row inside the sequence
    const int nt = n_w[w];
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // without a separate P region, S_w(j) complete also means PV_w(j-1) is
      // complete (same issuer, in order)
      if (!mbar_wait(&bar_s[w], j & 1, ac)) { ok = false; break; }
      tc_fence_after();
      float s[C::BN];
      {
        uint32_t u[C::BN];
#pragma unroll
        for (int c = 0; c < C::BN; c += 32) tmem_ld32_nowait(tS + c, u + c);
        tmem_wait_ld();
        if (C::SEP_P) {
          tc_fence_before();
          mbar_arrive(&bar_sfree[w]);
        }
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
      // row max: eight independent partial maxima over 3-input max steps
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx[i] = s[i];
#pragma unroll
        for (int b = 1; b + 1 < C::BN / 8; b += 2) mx[i] = fmax3(mx[i], s[8 * b + i], s[8 * b + 8 + i]);
        if constexpr ((C::BN / 8) % 2 == 0) mx[i] = fmaxf(mx[i], s[C::BN - 8 + i]);
      }
      const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * sl2;
      const float m_new = fmaxf(m_run, mt);
      const bool grow = m_new > m_run + 8.0f;          // also true on the first finite max
      const float m_use = grow ? m_new : m_run;
      const float alpha = grow ? ex2(m_run - m_use) : 1.0f;
      const float msub = (m_use == -INFINITY) ? 0.f : m_use;
      const bool warp_rescale = j > 0 && __any_sync(0xffffffffu, grow);
      // P = 2^(S * scale * log2 e - m): packed fp32x2 argument, row sum in four
      // packed partial sums, bf16 pairs for the PV MMA
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t nm2 = f2_pack(-msub, -msub);
      uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[C::BN / 2];
#pragma unroll
      for (int c = 0; c < C::BN; c += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, nm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        rs2[(c >> 1) & 3] = f2_add(rs2[(c >> 1) & 3], f2_pack(p0, p1));
        pk[c / 2] = pack_bf16(p0, p1);
      }
      float r0, r1, r2, r3, r4, r5, r6, r7;
      f2_unpack(rs2[0], r0, r1);
      f2_unpack(rs2[1], r2, r3);
      f2_unpack(rs2[2], r4, r5);
      f2_unpack(rs2[3], r6, r7);
      l_run = l_run * alpha + (((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7)));
      m_run = m_use;
      if (C::SEP_P && j > 0) {
        // PV(j-1) must be done before O is rescaled and P(j) overwrites P(j-1)
        if (!mbar_wait(&bar_o[w], (j - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
      }
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
      // P (bf16 pairs): 64 packed columns
      tmem_st32(tP, pk);
      tmem_st32(tP + 32, pk + 32);
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
