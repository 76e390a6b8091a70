// Dense / GQA / THD attention backward at head_dim 64 (the `flash_bwd` stage
// of "[Example] Introduce split+sum template, and optimize atomic_add
// performance for bwd examples", tile-ai/tilelang #940: atomic and split
// variants).  head_dim 128 has a kernel of its own (attn_bwd_d128.cu).
//
// Work item = one 128-row K/V tile of one kv head.  The CTA owning an item
// walks the query tiles of every query head of its GQA group, so dK and dV stay
// in TMEM for the whole item and are stored once (the group reduction of the
// #940 GQA backward, where dK is indexed by head // groups, happens on chip,
// without atomics).  Per 128-row query tile i of head h (KV rows j, query rows q):
//   S^T  = K Q_i^T   (TMEM)     P^T  = exp2(S^T * c - LSE_q * log2 e)
//   dP^T = V dO_i^T  (TMEM)     dS^T = P^T o (dP^T - Delta_q)
//   dV  += P^T dO_i             dK  += dS^T Q_i
// with P^T and dS^T written back into TMEM as packed bf16 and used as the TMEM
// A operand of the dV / dK MMAs, and dQ_i = dS K from a bf16 dS tile in shared
// memory, streamed out of TMEM through a shared-memory tile and either added
// into one fp32 accumulator (ATOMIC) or stored into the partial slab of this
// KV tile (SPLIT, summed in order later).  The accumulator and slabs are
// head-major, [batch, head, row, dim], so a query tile of one head is one
// contiguous block.
// The kernel is persistent: one CTA per SM walks a static list of items
// (longest first under causal masking, dealt to the CTAs in snake order), and
// every role runs ahead into the next item while the previous one finishes:
// K/V of the next item are loaded into a second buffer while the current one
// runs, and dK / dV leave TMEM through the dQ-drain warps, overlapped with the
// next item's first steps.
// The scale factor of dK is applied on the way out and that of dQ in the
// postprocess pass.
#include <cuda_runtime.h>

#include "bwd_items.cuh"
#include "launch.h"

namespace attn {

template <int D>
struct BwdCfg {
  static_assert(D == 64, "head_dim 64 only (head_dim 128: attn_bwd_d128.cu)");
  static constexpr int BN = 128;                      // KV rows per item
  static constexpr int BM = 128;                      // query rows per step
  static constexpr int HALF = BM / 2;                 // query columns per P/dS thread
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;        // bf16 dS tile (for dQ)
  // staging tile for dQ (fp32) and dK/dV (bf16) on their way out: half of the
  // 128 x 64 dQ tile, which leaves in two halves, so that three Q/dO stages fit
  // next to two K/V buffers
  static constexpr int STG_BYTES = BM * D * 2;
  static constexpr int KV_BUFS = 2;                   // K/V buffers (next item prefetch)
  static constexpr int NST = 3;                       // Q/dO stages
  static constexpr int SMEM =
      KV_BUFS * 2 * KV_BYTES + 2 * NST * QT_BYTES + DS_BYTES + STG_BYTES + 1024;
  static constexpr int THREADS = 448;
  static constexpr int THREADS_PAD = 480;   // with the padding warp (THD)
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns.  S^T and dP^T are BM fp32 columns each; P^T and dS^T are
  // packed bf16 pairs (BM / 2 columns each), P^T in columns of its own so that
  // S^T of the next step can be issued as soon as S^T of this one has been read.
  // That leaves no room for dS^T: each thread writes its packed dS^T over the
  // dP^T columns it has just read (the first half of its own HALF-column
  // range), and the next dP^T is issued after dK has read them.
  //   S^T 0..127, dP^T|dS^T 128..255, dV 256, dK 320, dQ 384, P^T 448
  static constexpr uint32_t COL_S = 0;                // S^T (fp32)
  static constexpr uint32_t COL_DP = BM;              // dP^T (fp32)
  static constexpr uint32_t COL_DV = 2 * BM;
  static constexpr uint32_t COL_DK = COL_DV + D;
  static constexpr uint32_t COL_DQ = COL_DK + D;      // one 64-column dQ tile
  static constexpr uint32_t COL_PT = COL_DQ + 64;
  static_assert(COL_PT + BM / 2 <= TMEM_COLS, "TMEM budget");
  // TMEM column of the packed dS^T columns of K-step kk (16 queries)
  __host__ __device__ static constexpr uint32_t ds_col(int kk) {
    return COL_DP + (16 * kk / HALF) * HALF + (16 * kk % HALF) / 2;
  }
  // dK and dV leave one after the other through the staging tile
  static_assert(BN * D * 2 <= STG_BYTES, "dK/dV staging");
  static_assert(SMEM <= 227 * 1024 - 4096, "shared memory budget");
};

// Warp roles: 0..7 P/dS (two warpgroups, each owns half of the query columns
// of every KV row), 8..11 dQ drain and dK/dV epilogue, 12 TMA, 13 the MMA
// issuer, which interleaves independent GEMMs.
// kThd: the instantiation for numbering 3; kPad: THD, with warp 14 writing the
// padding rows of dK and dV during the computation.  The others carry none of
// their code.
template <int D, bool kThd, bool kPad>
__global__ void __launch_bounds__(kPad ? BwdCfg<D>::THREADS_PAD : BwdCfg<D>::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmdK,
                    const __grid_constant__ CUtensorMap tmdV, const BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN, HALF = C::HALF;
  constexpr int PANELS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sKV = smem;                                  // KV_BUFS x (K, V)
  uint8_t* sQ = sKV + C::KV_BUFS * 2 * C::KV_BYTES;     // NST stages
  uint8_t* sdO = sQ + C::NST * C::QT_BYTES;             // NST stages
  uint8_t* sdS = sdO + C::NST * C::QT_BYTES;
  float* sDQ = reinterpret_cast<float*>(sdS + C::DS_BYTES);
  auto sK = [&](int b) { return sKV + b * 2 * C::KV_BYTES; };
  auto sV = [&](int b) { return sKV + b * 2 * C::KV_BYTES + C::KV_BYTES; };

  __shared__ uint64_t bar_kv_full[C::KV_BUFS], bar_kv_empty[C::KV_BUFS];
  __shared__ uint64_t bar_qfull[C::NST], bar_qempty[C::NST];
  __shared__ uint64_t bar_s, bar_dp, bar_p, bar_ds;
  __shared__ uint64_t bar_done, bar_dq_full, bar_dq_empty;
  __shared__ uint64_t bar_dv_empty, bar_dk_empty;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int s_mma_done;   // the MMA issuer has left its item loop
  __shared__ ThdOrder s_thd;   // the item list of numbering 3
  __shared__ __align__(16) float s_nlse[2][BM];   // -LSE * log2(e) per query column
  __shared__ __align__(16) float s_delta[2][BM];

  const Problem& p = a.p;
  const int warp = warp_id();
  const int total = a.total_items;
  const int G = static_cast<int>(p.fd_grp.d);   // query heads per kv head
  AbortCtx ac{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    s_mma_done = 0;
    for (int b = 0; b < C::KV_BUFS; ++b) {
      mbar_init(&bar_kv_full[b], 1);
      mbar_init(&bar_kv_empty[b], 1);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, 256);
    mbar_init(&bar_ds, 256);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_empty, 128);
    mbar_init(&bar_dv_empty, 128);
    mbar_init(&bar_dk_empty, 128);
    fence_mbar_init();
  }
  if constexpr (kThd)
    if (warp == 1) thd_order_build(p, BN, p.heads_kv * p.batch, s_thd);
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
      BwdItem w;
      int k = 0, ic = 0, gs = 0;
      ThdCursor cur;
      bool ok = true;
      while (ok && next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
        const int kb = ic % C::KV_BUFS, ku = ic / C::KV_BUFS;
        if (!mbar_wait(&bar_kv_empty[kb], (ku & 1) ^ 1, ac)) break;
        mbar_arrive_expect_tx(&bar_kv_full[kb], 2 * C::KV_BYTES);
        for (int pn = 0; pn < PANELS; ++pn) {
          tma_load_4d(&tmK, &bar_kv_full[kb], sK(kb) + pn * BN * 128, pn * 64, w.hk,
                      w.seq.row0 + w.kv0, w.seq.b);
          tma_load_4d(&tmV, &bar_kv_full[kb], sV(kb) + pn * BN * 128, pn * 64, w.hk,
                      w.seq.row0 + w.kv0, w.seq.b);
        }
        // step it = ih * n_i + ii: query head hk * G + ih, query tile i_start + ii
        int ih = 0, ii = -1;
        for (int it = 0; it < w.n_it; ++it) {
          if (++ii == w.n_i) { ii = 0; ++ih; }
          const int g = gs + it;
          const int st = g % C::NST, use = g / C::NST;
          if (!mbar_wait(&bar_qempty[st], (use & 1) ^ 1, ac)) { ok = false; break; }
          const int h = w.hk * G + ih;
          const int q0 = (w.i_start + ii) * BM;
          mbar_arrive_expect_tx(&bar_qfull[st], 2 * C::QT_BYTES);
          for (int pn = 0; pn < PANELS; ++pn) {
            tma_load_4d(&tmQ, &bar_qfull[st], sQ + st * C::QT_BYTES + pn * BM * 128, pn * 64, h,
                        w.seq.row0 + q0, w.seq.b);
            tma_load_4d(&tmdO, &bar_qfull[st], sdO + st * C::QT_BYTES + pn * BM * 128, pn * 64,
                        h, w.seq.row0 + q0, w.seq.b);
          }
        }
        gs += w.n_it;
        ++ic;
      }
    }
  } else if (warp == 13) {
    // ---------------- D = 64: one MMA issuer ----------------
    // The GEMMs go out in two phases per step g, each as soon as the P/dS
    // warps have produced its operand:
    //   after P(g):  S^T(g+1), then dV(g)
    //   after dS(g): dK(g), dQ(g), then dP^T(g+1)
    // each GEMM as one run of K-steps (measured faster than interleaving the
    // K-steps of independent GEMMs).
    // Step g+1's S^T/dP^T are issued here when its K/V tile is resident
    // (same item, or a second K/V buffer); otherwise at the start of its item.
    {   // warp-uniform: one elected lane issues
      constexpr int KS = D / 16;     // K-steps of S^T and dP^T
      constexpr int KV = BM / 16;    // K-steps of dV and dK
      constexpr int KQ = BN / 16;    // K-steps of dQ
      const uint32_t idSD = idesc_bf16(128, BM, false, false);
      const uint32_t idKV = idesc_bf16(128, D, false, true);
      const uint32_t idQ = idesc_bf16(128, 64, true, true);
      const uint64_t dQ_k0 = desc_kmajor_base(smem_u32(sQ));
      const uint64_t ddO_k0 = desc_kmajor_base(smem_u32(sdO));
      const uint64_t dQ_mn0 = desc_mnmajor_base(smem_u32(sQ), BM);
      const uint64_t ddO_mn0 = desc_mnmajor_base(smem_u32(sdO), BM);
      const uint64_t ddS_mn = desc_mnmajor_base(smem_u32(sdS), BN);
      auto issue_s = [&](int kb, int st, int kk) {
        umma_ss_w(tmem + C::COL_S, desc_advance(desc_kmajor_base(smem_u32(sK(kb))), kmajor_step_bytes(BN, kk)),
                desc_advance(dQ_k0, st * C::QT_BYTES + kmajor_step_bytes(BM, kk)), idSD, kk > 0);
      };
      auto issue_dp = [&](int kb, int st, int kk) {
        umma_ss_w(tmem + C::COL_DP, desc_advance(desc_kmajor_base(smem_u32(sV(kb))), kmajor_step_bytes(BN, kk)),
                desc_advance(ddO_k0, st * C::QT_BYTES + kmajor_step_bytes(BM, kk)), idSD, kk > 0);
      };
      // S^T and dP^T of one step, interleaved (both operands resident)
      auto issue_sdp = [&](int kb, int st) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          issue_s(kb, st, kk);
          issue_dp(kb, st, kk);
        }
        umma_commit_w(&bar_s);
        umma_commit_w(&bar_dp);
      };
      BwdItem w, wn;
      int k = 0, ic = 0, gs = 0;
      ThdCursor cur;
      bool ok = true;
      bool have = next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w);
      bool sdp_done = false;   // S^T/dP^T of the next step already issued
      while (ok && have) {
        const int kb = ic % C::KV_BUFS, ku = ic / C::KV_BUFS;
        const bool have_next = next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, wn);
        const int kbn = (ic + 1) % C::KV_BUFS, kun = (ic + 1) / C::KV_BUFS;
        if (!mbar_wait_w(&bar_kv_full[kb], ku & 1, ac)) break;
        const uint64_t dK_mn = desc_mnmajor_base(smem_u32(sK(kb)), BN);
        for (int it = 0; it < w.n_it; ++it) {
          const int g = gs + it;
          const int st = g % C::NST;
          if (!sdp_done) {
            if (!mbar_wait_w(&bar_qfull[st], (g / C::NST) & 1, ac)) { ok = false; break; }
            tc_fence_after();
            issue_sdp(kb, st);
          }
          // step g+1: its K/V buffer and whether its S^T/dP^T go out now
          const bool last = it + 1 == w.n_it;
          const bool nx = !last || (have_next && C::KV_BUFS > 1);
          const int kb1 = last ? kbn : kb;
          const int st1 = (g + 1) % C::NST;
          // ---- phase A: [S^T(g+1)], dV(g) ----
          if (!mbar_wait_w(&bar_p, g & 1, ac)) { ok = false; break; }
          if (it == 0 && ic > 0 && !mbar_wait_w(&bar_dv_empty, (ic - 1) & 1, ac)) { ok = false; break; }
          if (nx && last && !mbar_wait_w(&bar_kv_full[kbn], kun & 1, ac)) { ok = false; break; }
          if (nx && !mbar_wait_w(&bar_qfull[st1], ((g + 1) / C::NST) & 1, ac)) { ok = false; break; }
          tc_fence_after();
          const uint64_t omn = desc_advance(ddO_mn0, st * C::QT_BYTES);
          if (nx) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) issue_s(kb1, st1, kk);
            umma_commit_w(&bar_s);
          }
#pragma unroll
          for (int kk = 0; kk < KV; ++kk)
            umma_ts_w(tmem + C::COL_DV, tmem + C::COL_PT + 8 * kk,
                      desc_advance(omn, mnmajor_step_bytes(kk)), idKV, (it > 0 || kk > 0) ? 1u : 0u);
          // ---- phase B: dK(g), dQ(g) [, dP^T(g+1)] ----
          if (!mbar_wait_w(&bar_ds, g & 1, ac)) { ok = false; break; }
          if (!mbar_wait_w(&bar_dq_empty, (g & 1) ^ 1, ac)) { ok = false; break; }
          if (it == 0 && ic > 0 && !mbar_wait_w(&bar_dk_empty, (ic - 1) & 1, ac)) { ok = false; break; }
          tc_fence_after();
          const uint64_t qmn = desc_advance(dQ_mn0, st * C::QT_BYTES);
          // dK reads dS^T from the dP^T columns, so the next dP^T goes out
          // after it (MMAs of one thread execute in order)
#pragma unroll
          for (int kk = 0; kk < KV; ++kk)
            umma_ts_w(tmem + C::COL_DK, tmem + C::ds_col(kk), desc_advance(qmn, mnmajor_step_bytes(kk)),
                      idKV, (it > 0 || kk > 0) ? 1u : 0u);
          // dQ[q, d] = dS[q, kv] K[kv, d]
#pragma unroll
          for (int kk = 0; kk < KQ; ++kk)
            umma_ss_w(tmem + C::COL_DQ, desc_advance(ddS_mn, mnmajor_step_bytes(kk)),
                      desc_advance(dK_mn, mnmajor_step_bytes(kk)), idQ, kk > 0);
          if (nx) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) issue_dp(kb1, st1, kk);
            umma_commit_w(&bar_dp);
          }
          umma_commit_w(&bar_dq_full);
          umma_commit_w(&bar_qempty[st]);
          sdp_done = nx;
        }
        if (!ok) break;
        umma_commit_w(&bar_done);   // dV and dK of this item are final
        umma_commit_w(&bar_kv_empty[kb]);
        gs += w.n_it;
        ++ic;
        w = wn;
        have = have_next;
      }
    }
    if constexpr (kPad) *reinterpret_cast<volatile int*>(&s_mma_done) = 1;
  } else if (warp < 8) {
    // ---------------- P / dS warpgroups ----------------
    const int tid = threadIdx.x;                       // 0..255
    const int wg = warp >> 2;                          // column half
    const int r = (warp & 3) * 32 + lane_id();         // KV row in tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int c0 = wg * HALF;
    const float sl2 = a.scale_log2;
    // LSE or Delta of one query column, loaded one step ahead; the loaded value
    // is not touched until the next step, so the load latency stays hidden
    auto fetch = [&](const BwdItem& w, int ih, int ii) -> float {
      if (tid >= 2 * BM) return 0.f;
      const bool is_lse = tid < BM;
      const int c = is_lse ? tid : tid - BM;
      const int h = w.hk * G + ih;
      const int q = (w.i_start + ii) * BM + c;
      if (q >= w.seq.len) return is_lse ? INFINITY : 0.f;
      size_t li;
      if (p.cu_seqlens)
        li = static_cast<size_t>(h) * p.rows_total + w.seq.row0 + q;
      else
        li = (static_cast<size_t>(w.seq.b) * p.heads_q + h) * p.rows_total + q;
      return __ldg((is_lse ? a.lse : a.delta) + li);
    };
    const uint32_t tSme = tmem + lane_base + C::COL_S + c0;      // this thread's S columns
    const uint32_t tDPme = tmem + lane_base + C::COL_DP + c0;    // this thread's dP columns
    const uint32_t tPTme = tmem + lane_base + C::COL_PT + c0 / 2;
    const uint32_t tDSme = tmem + lane_base + C::COL_DP + c0;    // dS^T over dP^T
    BwdItem w;
    int k = 0, gs = 0;
    ThdCursor cur;
    bool have = next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w);
    float pf = have ? fetch(w, 0, 0) : 0.f;
    bool ok = true;
    while (ok && have) {
      const int kv = w.kv0 + r;                        // KV row inside the sequence
      const bool kv_ok = kv < w.seq.len;
      int ih = 0, ii = -1;   // step it = ih * n_i + ii
      for (int it = 0; it < w.n_it; ++it) {
        if (++ii == w.n_i) { ii = 0; ++ih; }
        const int g = gs + it;
        const int q0 = (w.i_start + ii) * BM;
        const int buf = g & 1;
        if (tid < BM) s_nlse[buf][tid] = -pf * kLog2e;   // LSE in the log2 domain, negated
        else if (tid < 2 * BM) s_delta[buf][tid - BM] = pf;
        if (it + 1 < w.n_it) {
          const bool wrap = ii + 1 == w.n_i;
          pf = fetch(w, wrap ? ih + 1 : ih, wrap ? 0 : ii + 1);
        } else {
          // last step of the item: look up the next one for the prefetch
          BwdItem wn;
          int kn = k;
          ThdCursor cn = cur;
          if (next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cn, kn, wn)) pf = fetch(wn, 0, 0);
        }
        named_bar_sync(1, 256);
        // ---- P^T (KV row r, query columns c0 .. c0 + HALF) ----
        if (!mbar_wait(&bar_s, g & 1, ac)) { ok = false; break; }
        tc_fence_after();
        {
          // Both passes run as rolled loops over 32-column chunks.  The
          // smaller loop body keeps the hot code of the eight P/dS warps, the
          // drain warps and the issuer small enough to stay in the
          // instruction cache (measured ~15% faster per step than the fully
          // unrolled 64-column body), and frees registers.  P comes back from
          // the P^T columns in the dS pass.
          const int lim_all = !kv_ok ? HALF : ((p.causal && q0 < w.kv0 + BN) ? kv - q0 - c0 : 0);
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
          // dV(g-1) has read P^T(g-1), and dK(g-1) / dQ(g-1) the dS tile,
          // once dP^T(g) has completed: the issuer sends dP^T(g) after them,
          // and its commit arrives only when every earlier MMA has completed.
          // So one wait on dP^T(g), before the first P^T store, covers both
          // (separate waits on those phases, long complete, still cost ~300
          // and ~500 cycles per step on the critical path).
#pragma unroll 1
          for (int c1 = 0; c1 < HALF; c1 += 32) {
            uint32_t u[32];
            tmem_ld32_nowait(tSme + c1, u);
            tmem_wait_ld();
            const int lim = lim_all - c1;
            if (lim > 0) {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (c < lim) u[c] = 0xff800000u;
            }
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(&s_nlse[buf][c0 + c1 + c]);
              float a0, a1, a2, a3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2x2,
                               f2_pack(l4.x, l4.y)), a0, a1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])),
                               sl2x2, f2_pack(l4.z, l4.w)), a2, a3);
              pk[c / 2] = f2_to_bf16x2(f2_pack(ex2(a0), ex2(a1)));
              pk[c / 2 + 1] = f2_to_bf16x2(f2_pack(ex2(a2), ex2(a3)));
            }
            if (c1 == 0) {
              if (!mbar_wait(&bar_dp, g & 1, ac)) { ok = false; break; }
              tc_fence_after();
            }
            tmem_st16p(tPTme + c1 / 2, pk);
          }
          if (!ok) break;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bar_p);
#pragma unroll 1
          for (int c1 = 0; c1 < HALF; c1 += 32) {
            uint32_t u[32], pp[16];
            tmem_ld32_nowait(tDPme + c1, u);
            tmem_ld16_nowait(tPTme + c1 / 2, pp);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const uint64_t pa = f2_pack(__uint_as_float(pp[c / 2] << 16),
                                          __uint_as_float(pp[c / 2] & 0xffff0000u));
              const uint64_t pb = f2_pack(__uint_as_float(pp[c / 2 + 1] << 16),
                                          __uint_as_float(pp[c / 2 + 1] & 0xffff0000u));
              const float4 d4 = *reinterpret_cast<const float4*>(&s_delta[buf][c0 + c1 + c]);
              pk[c / 2] = f2_to_bf16x2(f2_mul(f2_sub(f2_pack(__uint_as_float(u[c]),
                                                             __uint_as_float(u[c + 1])),
                                                     f2_pack(d4.x, d4.y)), pa));
              pk[c / 2 + 1] = f2_to_bf16x2(f2_mul(f2_sub(f2_pack(__uint_as_float(u[c + 2]),
                                                                 __uint_as_float(u[c + 3])),
                                                         f2_pack(d4.z, d4.w)), pb));
            }
            tmem_st16p(tDSme + c1 / 2, pk);   // dS^T over the dP^T columns just read
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int ch = (c0 + c1) / 8 + i;
              const uint32_t off = (ch >> 3) * BN * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(sdS + off) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bar_ds);
      }
      gs += w.n_it;
      have = next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w);
    }
  } else if (kPad ? warp < 12 : true) {
    // ---------------- dQ drain and dK/dV epilogue (warps 8..11) ----------------
    // dQ: TMEM -> fp32 staging tile in shared memory -> reduce-add into the
    // accumulator (ATOMIC) or store into this KV tile's slab (SPLIT), in two
    // halves: with dq_tma each 32-column box is staged in the 128-byte
    // swizzled layout of the accumulator's tensor map (one query row per
    // thread, conflict-free) and leaves through one TMA tensor copy, clipped
    // at the end of the rows by the map; otherwise 64 query rows at a time are
    // staged row-major [query][dim] (the layout of one head's rows in the
    // head-major accumulator) and leave through one bulk copy of the valid
    // rows.
    // dK / dV: at the end of every item, TMEM -> bf16 (dK x scale) -> the same
    // staging tile in the 128-byte swizzled layout of the dK/dV tensor maps ->
    // TMA stores; a THD tile that ends past its sequence is written row by row
    // with plain stores instead, so rows of the next sequence stay untouched.
    const int t = threadIdx.x - 256;                   // == TMEM lane == KV row / query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    if (t == 0) {
      if (a.dq_tma) tma_prefetch_desc(&tmDQ);
      tma_prefetch_desc(&tmdK);
      tma_prefetch_desc(&tmdV);
    }
    uint8_t* stg = reinterpret_cast<uint8_t*>(sDQ);
    BwdItem w;
    int k = 0, ic = 0, gs = 0;
    ThdCursor cur;
    bool ok = true;
    while (ok && next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
      float* base = a.dq_acc;
      bool slab_ok = true;
      if (a.split) {
        if (w.jt >= a.n_split) {
          slab_ok = false;
          if (t == 0 && p.err) atomicOr(p.err, ATTN_DEVERR_SEQLEN);
        } else {
          base += static_cast<size_t>(w.jt) * a.slab_elems;
        }
      }
      int ih = 0, ii = -1;   // step it = ih * n_i + ii
      for (int it = 0; it < w.n_it; ++it) {
        if (++ii == w.n_i) { ii = 0; ++ih; }
        const int g = gs + it;
        const int h = w.hk * G + ih;
        const int q0 = (w.i_start + ii) * BM;
        if (!mbar_wait(&bar_dq_full, g & 1, ac)) { ok = false; break; }
        tc_fence_after();
        // free the TMEM tile first, then wait for the staging tile
        uint32_t u[64];
        tmem_ld32_nowait(tmem + lane_base + C::COL_DQ, u);
        tmem_ld32_nowait(tmem + lane_base + C::COL_DQ + 32, u + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_dq_empty);
        {
          // two halves through the staging tile: the two 32-dim boxes of the
          // accumulator's map (dq_tma), else query rows 0..63 and 64..127
#pragma unroll
          for (int hx = 0; hx < 2; ++hx) {
            if (t == 0) bulk_wait_read<0>();   // previous copy finished reading the tile
            named_bar_sync(2, 128);
            if (a.dq_tma) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const int cc = 8 * hx + c;
                const uint32_t off = t * 128 + ((c ^ (t & 7)) << 4);
                *reinterpret_cast<float4*>(stg + off) =
                    make_float4(__uint_as_float(u[4 * cc]), __uint_as_float(u[4 * cc + 1]),
                                __uint_as_float(u[4 * cc + 2]), __uint_as_float(u[4 * cc + 3]));
              }
            } else if ((t >> 6) == hx) {
              // lane = query row, 64 columns = head dims
              float4* row = reinterpret_cast<float4*>(sDQ + (t & 63) * D);
#pragma unroll
              for (int c = 0; c < 16; ++c)
                row[c] = make_float4(__uint_as_float(u[4 * c]), __uint_as_float(u[4 * c + 1]),
                                     __uint_as_float(u[4 * c + 2]), __uint_as_float(u[4 * c + 3]));
            }
            fence_proxy_async_smem();
            named_bar_sync(2, 128);
            if (t == 0 && slab_ok) {
              if (a.dq_tma) {
                if (a.split)
                  tma_store_5d(&tmDQ, stg, hx * 32, w.seq.row0 + q0, h, w.seq.b, w.jt);
                else
                  tma_reduce_add_4d(&tmDQ, stg, hx * 32, w.seq.row0 + q0, h, w.seq.b);
              } else {
                const int nq = min(64, w.seq.len - q0 - 64 * hx);
                if (nq > 0) {
                  float* dst = base + ((static_cast<size_t>(w.seq.b) * p.heads_q + h) *
                                           p.rows_total + w.seq.row0 + q0 + 64 * hx) * D;
                  if (a.split)
                    bulk_store(dst, sDQ, static_cast<uint32_t>(nq) * D * 4);
                  else
                    bulk_reduce_add_f32(dst, sDQ, static_cast<uint32_t>(nq) * D * 4);
                }
              }
              bulk_commit();
            }
          }
        }
      }
      if (!ok) break;
      // ---- dV and dK (x scale) of this item ----
      if (!mbar_wait(&bar_done, ic & 1, ac)) break;
      tc_fence_after();
      const int kv = w.kv0 + t;
      const bool rows_exact = p.cu_seqlens != nullptr && w.kv0 + BN > w.seq.len;
      const size_t grow = static_cast<size_t>(w.seq.b) * p.rows_total + w.seq.row0 + kv;
      // dV first (the next item's first MMA overwrites it first), then dK,
      // each in panels of 64 dims staged at panel * BN * 128 of the tile
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::COL_DV : C::COL_DK;
        const float mul = which == 0 ? 1.0f : p.scale;
        uint8_t* tile = stg;
        __nv_bfloat16* gdst = (which == 0 ? a.dv : a.dk) + (grow * p.heads_kv + w.hk) * D;
        if (t == 0) bulk_wait_read<0>();   // the staging tile is free again
        named_bar_sync(2, 128);
#pragma unroll
        for (int pn = 0; pn < PANELS; ++pn) {
          uint32_t x[64];
          tmem_ld32_nowait(tmem + lane_base + col + pn * 64, x);
          tmem_ld32_nowait(tmem + lane_base + col + pn * 64 + 32, x + 32);
          tmem_wait_ld();
          if (pn == PANELS - 1) {
            tc_fence_before();
            mbar_arrive(which == 0 ? &bar_dv_empty : &bar_dk_empty);
          }
          uint32_t pkx[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pkx[c] = pack_bf16(__uint_as_float(x[2 * c]) * mul, __uint_as_float(x[2 * c + 1]) * mul);
          if (rows_exact) {
            if (kv < w.seq.len) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(gdst + pn * 64 + 8 * c) =
                    make_uint4(pkx[4 * c], pkx[4 * c + 1], pkx[4 * c + 2], pkx[4 * c + 3]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t off = pn * (BN * 128) + t * 128 + ((c ^ (t & 7)) << 4);
              *reinterpret_cast<uint4*>(tile + off) =
                  make_uint4(pkx[4 * c], pkx[4 * c + 1], pkx[4 * c + 2], pkx[4 * c + 3]);
            }
          }
        }
        if (!rows_exact) {
          fence_proxy_async_smem();
          named_bar_sync(2, 128);
          if (t == 0) {
            const CUtensorMap* m = which == 0 ? &tmdV : &tmdK;
            for (int pn = 0; pn < PANELS; ++pn)
              tma_store_4d(m, tile + pn * (BN * 128), pn * 64, w.hk, w.seq.row0 + w.kv0, w.seq.b);
            bulk_commit();
          }
        }
      }
      gs += w.n_it;
      ++ic;
    }
    if (t == 0) bulk_wait<0>();
  } else if constexpr (kPad) {
    // ---------------- warp 14: THD padding rows of dK and dV ----------------
    // Exact zeros for the rows at or past cu_seqlens[num_seqs] (this CTA's
    // slice of both tensors), 4 KB at a time with a 1 us pause while the MMA
    // issuer still has items.
    const int lane = lane_id();
    const int end = valid_end(p);
    const size_t per_row = static_cast<size_t>(p.heads_kv) * D / 8;   // 16-byte words
    const size_t n = static_cast<size_t>(p.rows_total - end) * per_row;
    const size_t lo = n * blockIdx.x / gridDim.x, hi = n * (blockIdx.x + 1) / gridDim.x;
    uint4* k4 = reinterpret_cast<uint4*>(a.dk) + static_cast<size_t>(end) * per_row;
    uint4* v4 = reinterpret_cast<uint4*>(a.dv) + static_cast<size_t>(end) * per_row;
    int it = 0;
    for (size_t i = lo + lane; i < hi; i += 32) {
      k4[i] = make_uint4(0u, 0u, 0u, 0u);
      v4[i] = make_uint4(0u, 0u, 0u, 0u);
      if ((++it & 3) == 0 && !*reinterpret_cast<volatile int*>(&s_mma_done)) __nanosleep(1000);
    }
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
                            const CUtensorMap& dO, const CUtensorMap& dq, const CUtensorMap& dk,
                            const CUtensorMap& dv, const BwdArgs& a, int grid, cudaStream_t st) {
  using C = BwdCfg<D>;
  const bool pad = a.pad_zero != 0;
  auto kern = a.x_major == 3 ? attn_bwd_kernel<D, true, true>
              : (pad ? attn_bwd_kernel<D, false, true> : attn_bwd_kernel<D, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, pad ? C::THREADS_PAD : C::THREADS, C::SMEM, st>>>(q, k, v, dO, dq, dk, dv, a);
  return cudaGetLastError();
}

template cudaError_t launch_attn_bwd<64>(const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const CUtensorMap&, const BwdArgs&,
                                         int, cudaStream_t);

}  // namespace attn
