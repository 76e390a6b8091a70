// Dense / GQA / THD attention backward (the `flash_bwd` stage of "[Example]
// Introduce split+sum template, and optimize atomic_add performance for bwd
// examples", tile-ai/tilelang #940: atomic and split variants).
//
// KV-tile-major: one CTA owns a 128-row K/V tile of one kv head and walks the
// query tiles of every query head of its GQA group, so dK and dV stay in TMEM
// for the whole CTA and are stored once (the group reduction of the #940 GQA
// backward, where dK is indexed by head // groups, happens on chip, without
// atomics).  Per query tile i of head h (KV rows j, query rows q):
//   S^T  = K Q_i^T   (TMEM)     P^T  = exp2(S^T * c - LSE_q * log2 e)
//   dP^T = V dO_i^T  (TMEM)     dS^T = P^T o (dP^T - Delta_q)
//   dV  += P^T dO_i             dK  += dS^T Q_i
// with P^T and dS^T written back into TMEM as packed bf16 over the S^T / dP^T
// columns they came from and used as the TMEM A operand of the dV / dK MMAs, and
//   dQ_i  = dS K  (D = 64, 128-row query tiles)  or
//   dQ_i^T = K^T dS^T (D = 128, 64-row query tiles) from a bf16 dS tile in
// shared memory, streamed out of TMEM through a shared-memory tile and either
// added into one fp32 accumulator with a bulk reduce-add (ATOMIC) or
// bulk-stored into the partial slab of this KV tile (SPLIT, summed in order
// later).  The accumulator and slabs are head-major, [batch, head, row, dim],
// so a query tile of one head is one contiguous block.
// The scale factor of dK is applied in the epilogue and that of dQ in the
// postprocess pass.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

template <int D>
struct BwdCfg {
  static constexpr int BN = 128;                      // KV rows per CTA
  static constexpr int BM = (D == 64) ? 128 : 64;     // query rows per step
  static constexpr int HALF = BM / 2;                 // query columns per P/dS thread
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;        // bf16 dS tile (for dQ)
  static constexpr int DQ_BYTES = BM * D * 4;         // fp32 dQ staging tile
  static constexpr int NST = 3;                       // Q/dO stages
  static constexpr int SMEM = 2 * KV_BYTES + 2 * NST * QT_BYTES + DS_BYTES + DQ_BYTES + 1024;
  static constexpr int THREADS = 512;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;                // S^T (fp32)
  static constexpr uint32_t COL_DP = BM;              // dP^T (fp32)
  static constexpr uint32_t COL_DV = 2 * BM;
  static constexpr uint32_t COL_DK = 2 * BM + D;
  static constexpr uint32_t COL_DQ = 2 * BM + 2 * D;  // one 64-column dQ tile
  static constexpr uint32_t COL_PT = COL_DQ + 64;     // P^T, packed bf16 (BM/2 columns)
  // D = 128 also has room for dS^T (packed) of its own; D = 64 writes dS^T
  // over the dP^T columns it came from (each thread over its own columns).
  static constexpr bool DS_ALIAS = (COL_PT + BM / 2 + BM / 2 > TMEM_COLS);
  static constexpr uint32_t COL_DST = DS_ALIAS ? COL_DP : COL_PT + BM / 2;
  // TMEM column (relative to COL_DST) of the packed dS^T columns of K-step kk.
  // Dedicated region: 8 per step.  Aliased: warpgroup w = 16 kk / HALF keeps
  // its HALF/2 packed columns at the start of its own HALF-column range.
  __host__ __device__ static constexpr uint32_t dst_col(int kk) {
    return DS_ALIAS ? 8 * kk + (16 * kk / HALF) * (HALF / 2) : 8 * kk;
  }
};

// Warp roles (512 threads): 0..7 P/dS (two warpgroups, each owns half of the
// query columns of every KV row), 8..11 dQ drain, 12 TMA, 13..15 MMA issuers
// (S^T and dP^T; dV and dK; dQ).  One issuing thread needs ~100 cycles per
// tcgen05.mma, so the five GEMMs of a step are spread over three issuers that
// run independently, synchronized only through the data they exchange.
template <int D>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, HALF = C::HALF;
  constexpr int PANELS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::KV_BYTES;
  uint8_t* sQ = sV + C::KV_BYTES;                 // NST stages
  uint8_t* sdO = sQ + C::NST * C::QT_BYTES;       // NST stages
  uint8_t* sdS = sdO + C::NST * C::QT_BYTES;
  float* sDQ = reinterpret_cast<float*>(sdS + C::DS_BYTES);

  __shared__ uint64_t bar_kv, bar_qfull[C::NST], bar_qempty[C::NST];
  __shared__ uint64_t bar_s, bar_dp, bar_p, bar_ds, bar_pt_done, bar_dst_done, bar_dss_free;
  __shared__ uint64_t bar_s_free, bar_dp_free, bar_done, bar_dq_full, bar_dq_empty;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ __align__(16) float s_nlse[2][BM];   // -LSE * log2(e) per query column
  __shared__ __align__(16) float s_delta[2][BM];

  const Problem& p = a.p;
  const int warp = warp_id();
  AbortCtx ac{&abort_flag, p.err};

  SeqRef seq;
  int jt;
  const int hk = blockIdx.y;
  if (!decode_tile(p, blockIdx.x, blockIdx.z, BN, seq, jt)) return;
  if (p.causal) jt = (seq.len + BN - 1) / BN - 1 - jt;   // longest work first
  const int G = p.heads_q / p.heads_kv;
  const int kv0 = jt * BN;
  const int i_start = p.causal ? kv0 / BM : 0;
  const int i_end = (seq.len + BM - 1) / BM;
  const int n_i = i_end - i_start;
  const int n_it = G * n_i;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 2);     // S/dP issuer and dV/dK issuer
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, 256);
    mbar_init(&bar_ds, 256);
    mbar_init(&bar_pt_done, 1);
    mbar_init(&bar_dst_done, 1);
    mbar_init(&bar_dss_free, 1);
    mbar_init(&bar_s_free, 256);
    mbar_init(&bar_dp_free, 256);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_empty, 128);
    fence_mbar_init();
  }
  if (warp == 13) tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 12) {
    // ---------------- TMA producer ----------------
    if (lane_id() == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(&bar_kv, 2 * C::KV_BYTES);
      for (int pn = 0; pn < PANELS; ++pn) {
        tma_load_4d(&tmK, &bar_kv, sK + pn * BN * 128, pn * 64, hk, seq.row0 + kv0, seq.b);
        tma_load_4d(&tmV, &bar_kv, sV + pn * BN * 128, pn * 64, hk, seq.row0 + kv0, seq.b);
      }
      for (int it = 0; it < n_it; ++it) {
        const int st = it % C::NST, use = it / C::NST;
        if (!mbar_wait(&bar_qempty[st], (use & 1) ^ 1, ac)) break;
        const int h = hk * G + it / n_i;
        const int q0 = (i_start + it % n_i) * BM;
        mbar_arrive_expect_tx(&bar_qfull[st], 2 * C::QT_BYTES);
        for (int pn = 0; pn < PANELS; ++pn) {
          tma_load_4d(&tmQ, &bar_qfull[st], sQ + st * C::QT_BYTES + pn * BM * 128, pn * 64, h,
                      seq.row0 + q0, seq.b);
          tma_load_4d(&tmdO, &bar_qfull[st], sdO + st * C::QT_BYTES + pn * BM * 128, pn * 64, h,
                      seq.row0 + q0, seq.b);
        }
      }
    }
  } else if (warp == 13) {
    // ---------------- issuer 1: S^T = K Q_i^T, dP^T = V dO_i^T ----------------
    if (lane_id() == 0) {
      const uint32_t idSD = idesc_bf16(128, BM, false, false);
      const uint64_t dK_k = desc_kmajor_base(smem_u32(sK));
      const uint64_t dV_k = desc_kmajor_base(smem_u32(sV));
      const uint64_t dQ_k0 = desc_kmajor_base(smem_u32(sQ));
      const uint64_t ddO_k0 = desc_kmajor_base(smem_u32(sdO));
      bool ok = mbar_wait(&bar_kv, 0, ac);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % C::NST;
        if (!mbar_wait(&bar_qfull[st], (it / C::NST) & 1, ac)) break;
        // S^T region is free once the P/dS warps have read S^T(it-1)
        if (it > 0 && !mbar_wait(&bar_s_free, (it - 1) & 1, ac)) break;
        tc_fence_after();
        const uint64_t qd = desc_advance(dQ_k0, st * C::QT_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tmem + C::COL_S, desc_advance(dK_k, kmajor_step_bytes(BN, k)),
                  desc_advance(qd, kmajor_step_bytes(BM, k)), idSD, k > 0);
        umma_commit(&bar_s);
        // dP^T region is free once dP^T(it-1) has been read and, when dS^T is
        // stored over it, once dK(it-1) has consumed dS^T(it-1)
        if (it > 0 && !mbar_wait(C::DS_ALIAS ? &bar_dst_done : &bar_dp_free, (it - 1) & 1, ac))
          break;
        tc_fence_after();
        const uint64_t od = desc_advance(ddO_k0, st * C::QT_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tmem + C::COL_DP, desc_advance(dV_k, kmajor_step_bytes(BN, k)),
                  desc_advance(od, kmajor_step_bytes(BM, k)), idSD, k > 0);
        umma_commit(&bar_dp);
        umma_commit(&bar_qempty[st]);
      }
    }
  } else if (warp == 14) {
    // ---------------- issuer 2: dV += P^T dO_i, dK += dS^T Q_i (A from TMEM) ----
    if (lane_id() == 0) {
      const uint32_t idKV = idesc_bf16(128, D, false, true);
      const uint64_t dQ_mn0 = desc_mnmajor_base(smem_u32(sQ), BM);
      const uint64_t ddO_mn0 = desc_mnmajor_base(smem_u32(sdO), BM);
      bool ok = true;
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % C::NST;
        if (!mbar_wait(&bar_qfull[st], (it / C::NST) & 1, ac)) break;
        if (!mbar_wait(&bar_p, it & 1, ac)) break;
        tc_fence_after();
        const uint64_t omn = desc_advance(ddO_mn0, st * C::QT_BYTES);
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          umma_ts(tmem + C::COL_DV, tmem + C::COL_PT + 8 * k,
                  desc_advance(omn, mnmajor_step_bytes(k)), idKV, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_pt_done);
        if (!mbar_wait(&bar_ds, it & 1, ac)) break;
        tc_fence_after();
        const uint64_t qmn = desc_advance(dQ_mn0, st * C::QT_BYTES);
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          umma_ts(tmem + C::COL_DK, tmem + C::COL_DST + C::dst_col(k),
                  desc_advance(qmn, mnmajor_step_bytes(k)), idKV, (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_dst_done);
        umma_commit(&bar_qempty[st]);
      }
      umma_commit(&bar_done);
    }
  } else if (warp == 15) {
    // ---------------- issuer 3: dQ (both operands in shared memory) ----------
    if (lane_id() == 0) {
      const uint32_t idQ = idesc_bf16(128, 64, true, true);
      const uint64_t dK_mn = desc_mnmajor_base(smem_u32(sK), BN);
      const uint64_t ddS_mn = desc_mnmajor_base(smem_u32(sdS), BN);
      bool ok = mbar_wait(&bar_kv, 0, ac);
      for (int it = 0; ok && it < n_it; ++it) {
        if (!mbar_wait(&bar_ds, it & 1, ac)) break;
        if (!mbar_wait(&bar_dq_empty, (it & 1) ^ 1, ac)) break;
        tc_fence_after();
        const uint32_t tDQ = tmem + C::COL_DQ;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          if (D == 64)   // dQ[q, d] = dS[q, kv] K[kv, d]
            umma_ss(tDQ, desc_advance(ddS_mn, mnmajor_step_bytes(k)),
                    desc_advance(dK_mn, mnmajor_step_bytes(k)), idQ, k > 0);
          else           // dQ^T[d, q] = K^T[d, kv] dS^T[kv, q]
            umma_ss(tDQ, desc_advance(dK_mn, mnmajor_step_bytes(k)),
                    desc_advance(ddS_mn, mnmajor_step_bytes(k)), idQ, k > 0);
        }
        umma_commit(&bar_dq_full);
        umma_commit(&bar_dss_free);
      }
    }
  } else if (warp < 8) {
    // ---------------- P / dS warpgroups ----------------
    const int tid = threadIdx.x;                       // 0..255
    const int wg = warp >> 2;                          // column half
    const int r = (warp & 3) * 32 + lane_id();         // KV row in tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int c0 = wg * HALF;
    const int kv = kv0 + r;                            // KV row inside the sequence
    const bool kv_ok = kv < seq.len;
    const float sl2 = a.scale_log2;
    // LSE or Delta of one query column, loaded one step ahead; the loaded value
    // is not touched until the next step, so the load latency stays hidden
    auto fetch = [&](int it) -> float {
      if (tid >= 2 * BM) return 0.f;
      const bool is_lse = tid < BM;
      const int c = is_lse ? tid : tid - BM;
      const int h = hk * G + it / n_i;
      const int q = (i_start + it % n_i) * BM + c;
      if (q >= seq.len) return is_lse ? INFINITY : 0.f;
      size_t li;
      if (p.cu_seqlens)
        li = static_cast<size_t>(h) * p.rows_total + seq.row0 + q;
      else
        li = (static_cast<size_t>(seq.b) * p.heads_q + h) * p.rows_total + q;
      return __ldg((is_lse ? a.lse : a.delta) + li);
    };
    float pf = (n_it > 0) ? fetch(0) : 0.f;
    bool ok = true;
    const uint32_t tSme = tmem + lane_base + C::COL_S + c0;      // this thread's S columns
    const uint32_t tDPme = tmem + lane_base + C::COL_DP + c0;    // this thread's dP columns
    const uint32_t tPTme = tmem + lane_base + C::COL_PT + c0 / 2;
    const uint32_t tDSTme = tmem + lane_base + C::COL_DST + (C::DS_ALIAS ? c0 : c0 / 2);
    for (int it = 0; it < n_it; ++it) {
      const int q0 = (i_start + it % n_i) * BM;
      const int buf = it & 1;
      if (tid < BM) s_nlse[buf][tid] = -pf * kLog2e;   // LSE in the log2 domain, negated
      else if (tid < 2 * BM) s_delta[buf][tid - BM] = pf;
      if (it + 1 < n_it) pf = fetch(it + 1);
      named_bar_sync(1, 256);
      // ---- P^T (KV row r, query columns c0 .. c0 + HALF) ----
      if (!mbar_wait(&bar_s, it & 1, ac)) { ok = false; break; }
      tc_fence_after();
      // P^T in fp32 pairs: p2[i] = (P[2i], P[2i+1]) of this thread's columns
      uint64_t p2[HALF / 2];
      {
        uint32_t u[HALF];
#pragma unroll
        for (int c = 0; c < HALF; c += 32) tmem_ld32_nowait(tSme + c, u + c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_s_free);
        // masking on S: the whole row past the sequence end, the causal
        // triangle on diagonal tiles (columns c < lim hold earlier queries)
        int lim = 0;
        if (!kv_ok) lim = HALF;
        else if (p.causal && q0 < kv0 + BN) lim = kv - q0 - c0;
        if (lim > 0) {
#pragma unroll
          for (int c = 0; c < HALF; ++c)
            if (c < lim) u[c] = 0xff800000u;   // -inf
        }
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int c = 0; c < HALF; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(&s_nlse[buf][c0 + c]);
          float a0, a1, a2, a3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2x2,
                           f2_pack(l4.x, l4.y)), a0, a1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sl2x2,
                           f2_pack(l4.z, l4.w)), a2, a3);
          p2[c / 2] = f2_pack(ex2(a0), ex2(a1));
          p2[c / 2 + 1] = f2_pack(ex2(a2), ex2(a3));
        }
      }
      {
        uint32_t pk[HALF / 2];
#pragma unroll
        for (int i = 0; i < HALF / 2; ++i) pk[i] = f2_to_bf16x2(p2[i]);
        // P^T(it-1) must have been consumed by dV(it-1)
        if (it > 0 && !mbar_wait(&bar_pt_done, (it - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
        if constexpr (HALF / 2 == 32) tmem_st32(tPTme, pk);
        else tmem_st16p(tPTme, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_p);
      // ---- dS^T = P^T o (dP^T - Delta) ----
      if (!mbar_wait(&bar_dp, it & 1, ac)) { ok = false; break; }
      tc_fence_after();
      uint32_t pk[HALF / 2];
      {
        uint32_t u[HALF];
#pragma unroll
        for (int c = 0; c < HALF; c += 32) tmem_ld32_nowait(tDPme + c, u + c);
        tmem_wait_ld();
        if constexpr (!C::DS_ALIAS) {
          tc_fence_before();
          mbar_arrive(&bar_dp_free);
        }
#pragma unroll
        for (int c = 0; c < HALF; c += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(&s_delta[buf][c0 + c]);
          const uint64_t ds01 = f2_mul(
              f2_sub(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), f2_pack(d4.x, d4.y)),
              p2[c / 2]);
          const uint64_t ds23 = f2_mul(
              f2_sub(f2_pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])),
                     f2_pack(d4.z, d4.w)),
              p2[c / 2 + 1]);
          pk[c / 2] = f2_to_bf16x2(ds01);
          pk[c / 2 + 1] = f2_to_bf16x2(ds23);
        }
      }
      if constexpr (!C::DS_ALIAS) {
        // dS^T(it-1) must have been consumed by dK(it-1)
        if (it > 0 && !mbar_wait(&bar_dst_done, (it - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
      }
      if constexpr (HALF / 2 == 32) tmem_st32(tDSTme, pk);
      else tmem_st16p(tDSTme, pk);
      // dS (bf16) also to shared memory for the dQ GEMM
      if (it > 0 && !mbar_wait(&bar_dss_free, (it - 1) & 1, ac)) { ok = false; break; }
#pragma unroll
      for (int i = 0; i < HALF / 8; ++i) {
        const int ch = c0 / 8 + i;
        const uint32_t off = (ch >> 3) * BN * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sdS + off) =
            make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_ds);
    }
    // ---- epilogue: dK (x scale) and dV, this thread's half of the head dims ----
    if (ok && mbar_wait(&bar_done, 0, ac)) {
      tc_fence_after();
      constexpr int DH = D / 2;
      const int d0 = wg * DH;
      const size_t grow = static_cast<size_t>(seq.b) * p.rows_total + seq.row0 + kv;
      __nv_bfloat16* dkrow = a.dk + (grow * p.heads_kv + hk) * D + d0;
      __nv_bfloat16* dvrow = a.dv + (grow * p.heads_kv + hk) * D + d0;
      const float sc = p.scale;
#pragma unroll
      for (int c0d = 0; c0d < DH; c0d += 32) {
        uint32_t u[32], w[32];
        tmem_ld32_nowait(tmem + lane_base + C::COL_DK + d0 + c0d, u);
        tmem_ld32_nowait(tmem + lane_base + C::COL_DV + d0 + c0d, w);
        tmem_wait_ld();
        if (kv_ok) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 kk, vv;
            kk.x = pack_bf16(__uint_as_float(u[c + 0]) * sc, __uint_as_float(u[c + 1]) * sc);
            kk.y = pack_bf16(__uint_as_float(u[c + 2]) * sc, __uint_as_float(u[c + 3]) * sc);
            kk.z = pack_bf16(__uint_as_float(u[c + 4]) * sc, __uint_as_float(u[c + 5]) * sc);
            kk.w = pack_bf16(__uint_as_float(u[c + 6]) * sc, __uint_as_float(u[c + 7]) * sc);
            vv.x = pack_bf16(__uint_as_float(w[c + 0]), __uint_as_float(w[c + 1]));
            vv.y = pack_bf16(__uint_as_float(w[c + 2]), __uint_as_float(w[c + 3]));
            vv.z = pack_bf16(__uint_as_float(w[c + 4]), __uint_as_float(w[c + 5]));
            vv.w = pack_bf16(__uint_as_float(w[c + 6]), __uint_as_float(w[c + 7]));
            *reinterpret_cast<uint4*>(dkrow + c0d + c) = kk;
            *reinterpret_cast<uint4*>(dvrow + c0d + c) = vv;
          }
        }
      }
    }
  } else {
    // ---------------- dQ drain (warps 8..11) ----------------
    // TMEM -> fp32 staging tile in shared memory (row-major [query][dim], the
    // layout of one head's rows in the head-major accumulator) -> one bulk
    // reduce-add (ATOMIC) or bulk store into this KV tile's slab (SPLIT).
    const int t = threadIdx.x - 256;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* base = a.dq_acc;
    bool slab_ok = true;
    if (a.split) {
      if (jt >= a.n_split) {
        slab_ok = false;
        if (t == 0 && p.err) atomicOr(p.err, ATTN_DEVERR_SEQLEN);
      } else {
        base += static_cast<size_t>(jt) * a.slab_elems;
      }
    }
    for (int it = 0; it < n_it; ++it) {
      const int h = hk * G + it / n_i;
      const int q0 = (i_start + it % n_i) * BM;
      if (!mbar_wait(&bar_dq_full, it & 1, ac)) break;
      tc_fence_after();
      // free the TMEM tile first, then wait for the staging tile
      uint32_t u[64];
      tmem_ld32_nowait(tmem + lane_base + C::COL_DQ, u);
      tmem_ld32_nowait(tmem + lane_base + C::COL_DQ + 32, u + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_dq_empty);
      if (t == 0) bulk_wait_read<0>();   // previous bulk copy finished reading the tile
      named_bar_sync(2, 128);
      if (D == 64) {
        // lane = query row, 64 columns = head dims
        float4* row = reinterpret_cast<float4*>(sDQ + t * D);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          row[c] = make_float4(__uint_as_float(u[4 * c]), __uint_as_float(u[4 * c + 1]),
                               __uint_as_float(u[4 * c + 2]), __uint_as_float(u[4 * c + 3]));
      } else {
        // lane = head dim, 64 columns = query rows
#pragma unroll
        for (int c = 0; c < 64; ++c) sDQ[c * D + t] = __uint_as_float(u[c]);
      }
      fence_proxy_async_smem();
      named_bar_sync(2, 128);
      if (t == 0 && slab_ok) {
        const int nq = min(BM, seq.len - q0);
        float* dst = base + ((static_cast<size_t>(seq.b) * p.heads_q + h) * p.rows_total +
                             seq.row0 + q0) * D;
        if (a.split)
          bulk_store(dst, sDQ, static_cast<uint32_t>(nq) * D * 4);
        else
          bulk_reduce_add_f32(dst, sDQ, static_cast<uint32_t>(nq) * D * 4);
        bulk_commit();
      }
    }
    if (t == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
}

template <int D>
cudaError_t launch_attn_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dO, const BwdArgs& a, int grid_x, cudaStream_t st) {
  using C = BwdCfg<D>;
  auto kern = attn_bwd_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(grid_x, a.p.heads_kv, a.p.batch);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(q, k, v, dO, a);
  return cudaGetLastError();
}

template cudaError_t launch_attn_bwd<64>(const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const CUtensorMap&, const BwdArgs&,
                                         int, cudaStream_t);
template cudaError_t launch_attn_bwd<128>(const CUtensorMap&, const CUtensorMap&,
                                          const CUtensorMap&, const CUtensorMap&, const BwdArgs&,
                                          int, cudaStream_t);

}  // namespace attn
