// Dense / GQA / THD attention backward at head_dim 128 (the `flash_bwd` stage of
// "[Example] Introduce split+sum template, and optimize atomic_add performance
// for bwd examples", tile-ai/tilelang #940: atomic and split variants).
//
// Work item = one 128-row K/V tile of one kv head, as in the D = 64 kernel: the
// CTA owning an item walks the 128-row query tiles of every query head of its
// GQA group, so dK and dV stay in TMEM for the whole item and are stored once.
// One step is a 128 x 128 (K/V rows x query rows) tile:
//   S^T  = K Q^T    ->  P^T  = exp2(S^T c - LSE log2 e)
//   dP^T = V dO^T   ->  dS^T = P^T o (dP^T - Delta)
//   dV  += P^T dO,  dK += dS^T Q     (P^T, dS^T: packed bf16, TMEM A operand)
//   dQ^T = K^T dS^T                  (dS: bf16 tile in shared memory)
// Every GEMM has N = 128.  An SS MMA of N = 64 reads 6 KB of operands per
// 16-deep K-step for 2^18 FLOPs, one of N = 128 reads 8 KB for 2^19, so the
// 128-query step halves the operand traffic per FLOP that bounds the shared
// memory, and each synchronisation covers twice the work.
// TMEM (512 columns; lanes = K/V rows, except dQ^T whose lanes are head dims):
//   0..127    S^T(g).  Each P/dS warpgroup owns 64 of these columns; its P pass
//             leaves P^T in the first 32 of them and its dS pass dS^T in the
//             last 32, both over S^T values that thread has already read.
//   128..255  dP^T(g), then dQ^T(g) once the dS pass has read dP^T(g).
//   256..383  dV          384..511  dK
// MMAs issued by one thread run in order, so S^T(g+1) goes out after dK(g)
// (the last reader of the S^T columns), and dP^T(g+1) after the drain warps
// have read dQ^T(g) out of TMEM.
// Shared memory: K, V (32 KB each), two Q slots, one dO slot, the dS tile
// (32 KB each) and a 16 KB staging tile for the dQ, dK and dV copies out.
// Warps: 0..7 P/dS (warpgroup w: query columns 64w .. 64w + 63 of every K/V
// row), 8..15 drain (warpgroup u: dQ^T columns 64u .. 64u + 63, so all of
// dQ^T leaves TMEM in one load; dV / dK dims 64u .. 64u + 63 at the end of an
// item), 16 TMA, 17 MMA issuer.
// For THD, warp 18 writes the exact zeros of the padding rows of dK and dV
// (this CTA's slice) while the others compute.
// dQ leaves TMEM in one load and goes out per warp, 32 dims x 16 query rows
// per TMA copy: a reduce-add into the fp32 accumulator (ATOMIC) or a store
// into this K/V tile's slab (SPLIT).  One 16 KB copy at a time through a
// shared tile ran at ~11 bytes per clock per SM, which bounded the step; eight
// independent warps keep eight copies in flight.  The scale of dK is applied
// on the way out, that of dQ in the postprocess pass.
#include <cuda_runtime.h>

#include "bwd_items.cuh"
#include "launch.h"

namespace attn {
namespace {

struct Bwd128 {
  static constexpr int D = 128, BN = 128, BM = 128, HALF = 64;
  static constexpr int TILE = 128 * 128 * 2;      // one bf16 128 x 128 tile (two 64-column panels)
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE, OFF_DO = 4 * TILE,
                       OFF_DS = 6 * TILE;
  static constexpr int SMEM = 7 * TILE + 1024;
  static constexpr int THREADS = 576;
  static constexpr int THREADS_PAD = 608;   // with the padding warp (THD)
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384;
  // packed P^T / dS^T columns of K-step kk (queries 16 kk .. 16 kk + 15) of
  // the dV / dK MMAs: warpgroup kk / 4 holds them
  __host__ __device__ static constexpr uint32_t pt_col(int kk) {
    return COL_S + 64 * (kk >> 2) + 8 * (kk & 3);
  }
  __host__ __device__ static constexpr uint32_t dst_col(int kk) { return pt_col(kk) + 32; }
  // dynamic + the kernel's static shared memory (barriers, one row of LSE and
  // Delta: about 1.2 KB) within the 227 KB a CTA may use
  static_assert(SMEM + 1536 <= 227 * 1024, "shared memory budget");
};

// Step order inside an item: query tiles from the last down to the first, the
// query heads of the GQA group innermost.  Every K/V tile of a (batch, kv
// head) then meets query tile i of head h at the same step index,
// (last - i) * groups + h, whatever its first query tile: the ordered SPLIT
// accumulation, where K/V tile jt waits for tiles 0 .. jt-1 at each (i, h),
// keeps all tiles of a head in step instead of throttling each to tile 0.
__device__ __forceinline__ void next_step(int& ih, int& ii, int groups) {
  if (++ih == groups) {
    ih = 0;
    --ii;
  }
}

// kOrdered: the SPLIT mode's fixed-order dQ accumulation (see the drain).
// Each mode is its own instantiation: the drain loop is sensitive to its code
// size (the ATOMIC kernel measured 10% slower with the ordered path compiled
// in).
// kThd: the instantiation for numbering 3 (atomic dQ only); kPad: THD, with
// the padding warp.  The other instantiations carry none of their code: the
// ordered drain loop slowed by 7% with numbering 3 inlined, the dense backward
// by 4% with the padding warp in the kernel.
template <bool kOrdered, bool kThd, bool kPad>
__global__ void __launch_bounds__(kPad ? Bwd128::THREADS_PAD : Bwd128::THREADS, 1)
    attn_bwd128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdArgs a) {
  using C = Bwd128;
  constexpr int BM = C::BM, BN = C::BN, HALF = C::HALF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;     // two slots
  uint8_t* sdO = smem + C::OFF_DO;   // two slots
  uint8_t* sdS = smem + C::OFF_DS;

  __shared__ uint64_t bar_kv_full, bar_kv_empty, bar_qfull[2], bar_qempty[2], bar_dofull[2],
      bar_doempty[2];
  __shared__ uint64_t bar_s, bar_dp, bar_p, bar_ds, bar_dq_full, bar_dq_empty;
  __shared__ uint64_t bar_done, bar_dv_empty, bar_dk_empty;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int s_mma_done;   // the MMA issuer has left its item loop
  __shared__ ThdOrder s_thd;   // the item list of numbering 3
  // -LSE * log2(e) and Delta of the step's query columns; one buffer, so that
  // the tiles and these fit the 227 KB with the 1 KB alignment margin
  __shared__ __align__(16) float s_nlse[BM];
  __shared__ __align__(16) float s_delta[BM];

  const Problem& p = a.p;
  const int warp = warp_id();
  const int total = a.total_items;
  const int G = static_cast<int>(p.fd_grp.d);   // query heads per kv head
  AbortCtx ac{&abort_flag, p.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    s_mma_done = 0;
    mbar_init(&bar_kv_full, 1);
    mbar_init(&bar_kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_qfull[s], 1);
      mbar_init(&bar_qempty[s], 1);
      mbar_init(&bar_dofull[s], 1);
      mbar_init(&bar_doempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, 256);
    mbar_init(&bar_ds, 256);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_empty, 256);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_dv_empty, 256);
    mbar_init(&bar_dk_empty, 256);
    fence_mbar_init();
  }
  if constexpr (kThd)
    if (warp == 1) thd_order_build(p, BN, p.heads_kv * p.batch, s_thd);
  if (warp == 17) tmem_alloc(&tmem_base_sh, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 16) {
    // ---------------- TMA producer ----------------
    // K/V once per item; Q and dO (two slots each) once per step.  dO(g) is
    // last read by dV(g), in the middle of step g, and dP^T(g+2) needs its
    // slot again at the end of step g+1: the load has a whole step to arrive
    // (a dO load under this traffic takes about half a step).  The waits spin:
    // a suspended producer resumes too late to keep a step ahead.
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
        if (!mbar_wait_spin(&bar_kv_empty, (ic & 1) ^ 1, ac)) break;
        mbar_arrive_expect_tx(&bar_kv_full, 2 * C::TILE);
        for (int pn = 0; pn < 2; ++pn) {
          tma_load_4d(&tmK, &bar_kv_full, sK + pn * BN * 128, pn * 64, w.hk, w.seq.row0 + w.kv0,
                      w.seq.b);
          tma_load_4d(&tmV, &bar_kv_full, sV + pn * BN * 128, pn * 64, w.hk, w.seq.row0 + w.kv0,
                      w.seq.b);
        }
        int ih = -1, ii = w.n_i - 1;   // step order: see next_step
        for (int it = 0; it < w.n_it; ++it) {
          next_step(ih, ii, G);
          const int g = gs + it, sl = g & 1, par = ((g >> 1) & 1) ^ 1;
          const int h = w.hk * G + ih;
          const int row = w.seq.row0 + (w.i_start + ii) * BM;
          if (!mbar_wait_spin(&bar_qempty[sl], par, ac)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar_qfull[sl], C::TILE);
          for (int pn = 0; pn < 2; ++pn)
            tma_load_4d(&tmQ, &bar_qfull[sl], sQ + sl * C::TILE + pn * BM * 128, pn * 64, h, row,
                        w.seq.b);
          if (!mbar_wait_spin(&bar_doempty[sl], par, ac)) { ok = false; break; }
          mbar_arrive_expect_tx(&bar_dofull[sl], C::TILE);
          for (int pn = 0; pn < 2; ++pn)
            tma_load_4d(&tmdO, &bar_dofull[sl], sdO + sl * C::TILE + pn * BM * 128, pn * 64, h,
                        row, w.seq.b);
        }
        gs += w.n_it;
        ++ic;
      }
    }
  } else if (warp == 17) {
    // ---------------- MMA issuer (warp-uniform: one elected lane issues) ----------------
    // Per step g: dV(g) after P(g); after dS(g): dK(g), S^T(g+1), dQ^T(g), and
    // dP^T(g+1) once dQ^T(g) has left TMEM.  The first step of an item issues
    // its own S^T and dP^T.
    const uint32_t idS = idesc_bf16(128, BM, false, false);   // S^T, dP^T
    const uint32_t idKV = idesc_bf16(128, 128, false, true);  // dV, dK (A from TMEM)
    const uint32_t idQ = idesc_bf16(128, BM, true, true);     // dQ^T
    const uint64_t dK_k = desc_kmajor_base(smem_u32(sK));
    const uint64_t dV_k = desc_kmajor_base(smem_u32(sV));
    const uint64_t dK_mn = desc_mnmajor_base(smem_u32(sK), BN);
    const uint64_t dQ_k0 = desc_kmajor_base(smem_u32(sQ));
    const uint64_t dQ_mn0 = desc_mnmajor_base(smem_u32(sQ), BM);
    const uint64_t ddO_k0 = desc_kmajor_base(smem_u32(sdO));
    const uint64_t ddO_mn0 = desc_mnmajor_base(smem_u32(sdO), BM);
    const uint64_t ddS_mn = desc_mnmajor_base(smem_u32(sdS), BN);
    auto issue_s = [&](int qs) {   // S^T = K Q^T
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ss_w(tmem + C::COL_S, desc_advance(dK_k, kmajor_step_bytes(BN, kk)),
                  desc_advance(dQ_k0, qs * C::TILE + kmajor_step_bytes(BM, kk)), idS, kk > 0);
      umma_commit_w(&bar_s);
    };
    auto issue_dp = [&](int sl) {  // dP^T = V dO^T
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ss_w(tmem + C::COL_DP, desc_advance(dV_k, kmajor_step_bytes(BN, kk)),
                  desc_advance(ddO_k0, sl * C::TILE + kmajor_step_bytes(BM, kk)), idS, kk > 0);
      umma_commit_w(&bar_dp);
    };
    BwdItem w;
    int k = 0, ic = 0, gs = 0;
    ThdCursor cur;
    bool ok = true;
    while (ok && next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
      if (!mbar_wait_w(&bar_kv_full, ic & 1, ac)) break;
      for (int it = 0; it < w.n_it; ++it) {
        const int g = gs + it, qs = g & 1;
        if (it == 0) {
          if (!mbar_wait_w(&bar_qfull[qs], (g >> 1) & 1, ac)) { ok = false; break; }
          tc_fence_after();
          issue_s(qs);
          // dQ^T of the previous step still occupies the dP^T columns
          if (g > 0 && !mbar_wait_w(&bar_dq_empty, (g - 1) & 1, ac)) { ok = false; break; }
          if (!mbar_wait_w(&bar_dofull[qs], (g >> 1) & 1, ac)) { ok = false; break; }
          tc_fence_after();
          issue_dp(qs);
        }
        // ---- dV(g) += P^T(g) dO(g) ----
        if (!mbar_wait_w(&bar_p, g & 1, ac)) { ok = false; break; }
        // the previous item's epilogue must have read dV out of TMEM
        if (it == 0 && ic > 0 && !mbar_wait_w(&bar_dv_empty, (ic - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
        const uint64_t omn = desc_advance(ddO_mn0, qs * C::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_w(tmem + C::COL_DV, tmem + C::pt_col(kk), desc_advance(omn, mnmajor_step_bytes(kk)),
                    idKV, (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(&bar_doempty[qs]);   // dP^T(g) and dV(g) have read dO(g)
        const bool nx = it + 1 < w.n_it;
        // Q(g+1) has long arrived; testing it here, while the dS pass runs,
        // keeps the barrier round trip off the dK -> S^T(g+1) path
        if (nx && !mbar_wait_w(&bar_qfull[qs ^ 1], ((g + 1) >> 1) & 1, ac)) { ok = false; break; }
        // ---- dK(g) += dS^T(g) Q(g) ----
        if (!mbar_wait_w(&bar_ds, g & 1, ac)) { ok = false; break; }
        if (it == 0 && ic > 0 && !mbar_wait_w(&bar_dk_empty, (ic - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
        const uint64_t qmn = desc_advance(dQ_mn0, qs * C::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_w(tmem + C::COL_DK, tmem + C::dst_col(kk), desc_advance(qmn, mnmajor_step_bytes(kk)),
                    idKV, (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(&bar_qempty[qs]);   // S^T(g) and dK(g) have read Q(g)
        // ---- S^T(g+1) over the P^T / dS^T columns dV(g) and dK(g) have read ----
        if (nx) issue_s(qs ^ 1);
        // ---- dQ^T(g) = K^T dS^T(g) into the dP^T columns ----
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss_w(tmem + C::COL_DP, desc_advance(dK_mn, mnmajor_step_bytes(kk)),
                    desc_advance(ddS_mn, mnmajor_step_bytes(kk)), idQ, kk > 0);
        umma_commit_w(&bar_dq_full);
        // ---- dP^T(g+1) once dQ^T(g) has left TMEM ----
        if (nx) {
          // dO(g+1) first: it arrived a step ago, and its test overlaps the drain
          if (!mbar_wait_w(&bar_dofull[qs ^ 1], ((g + 1) >> 1) & 1, ac)) { ok = false; break; }
          if (!mbar_wait_w(&bar_dq_empty, g & 1, ac)) { ok = false; break; }
          tc_fence_after();
          issue_dp(qs ^ 1);
        }
      }
      if (!ok) break;
      umma_commit_w(&bar_done);       // dV and dK of this item are final
      umma_commit_w(&bar_kv_empty);
      gs += w.n_it;
      ++ic;
    }
    if constexpr (kPad) *reinterpret_cast<volatile int*>(&s_mma_done) = 1;
  } else if (warp < 8) {
    // ---------------- P / dS warpgroups ----------------
    const int tid = threadIdx.x;                       // 0..255
    const int wg = warp >> 2;                          // column half
    const int r = (warp & 3) * 32 + lane_id();         // K/V row in tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int c0 = wg * HALF;
    const float sl2 = a.scale_log2;
    // LSE or Delta of one query column, loaded one step ahead; the loaded value
    // is not touched until the next step, so the load latency stays hidden
    auto fetch = [&](const BwdItem& w, int ih, int ii) -> float {
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
    const uint32_t tS = tmem + lane_base + C::COL_S + c0;    // S^T; P^T at +0, dS^T at +32
    const uint32_t tDP = tmem + lane_base + C::COL_DP + c0;  // dP^T
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    BwdItem w;
    int k = 0, gs = 0;
    ThdCursor cur;
    bool have = next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w);
    float pf = have ? fetch(w, 0, w.n_i - 1) : 0.f;
    bool ok = true;
    while (ok && have) {
      const int kv = w.kv0 + r;                        // K/V row inside the sequence
      const bool kv_ok = kv < w.seq.len;
      int ih = -1, ii = w.n_i - 1;   // step order: see next_step
      for (int it = 0; it < w.n_it; ++it) {
        next_step(ih, ii, G);
        const int g = gs + it;
        const int q0 = (w.i_start + ii) * BM;
        named_bar_sync(1, 256);   // every thread has read the previous step's values
        if (tid < BM) s_nlse[tid] = -pf * kLog2e;   // LSE in the log2 domain, negated
        else s_delta[tid - BM] = pf;
        if (it + 1 < w.n_it) {
          const bool wrap = ih + 1 == G;
          pf = fetch(w, wrap ? 0 : ih + 1, wrap ? ii - 1 : ii);
        } else {
          // last step of the item: look up the next one for the prefetch
          BwdItem wn;
          int kn = k;
          ThdCursor cn = cur;
          if (next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cn, kn, wn))
            pf = fetch(wn, 0, wn.n_i - 1);
        }
        named_bar_sync(1, 256);
        // ---- P^T (K/V row r, query columns c0 .. c0 + 63), two 32-column chunks ----
        if (!mbar_wait(&bar_s, g & 1, ac)) { ok = false; break; }
        tc_fence_after();
        // masking on S: the whole row past the sequence end, the causal
        // triangle on diagonal tiles (columns c < lim hold earlier queries)
        const int lim_all = !kv_ok ? HALF : ((p.causal && q0 < w.kv0 + BN) ? kv - q0 - c0 : 0);
#pragma unroll 1
        for (int c1 = 0; c1 < HALF; c1 += 32) {
          uint32_t u[32];
          tmem_ld32_nowait(tS + c1, u);
          tmem_wait_ld();
          const int lim = lim_all - c1;
          if (lim > 0) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < lim) u[c] = 0xff800000u;   // -inf
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(&s_nlse[c0 + c1 + c]);
            float a0, a1, a2, a3;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), sl2x2,
                             f2_pack(l4.x, l4.y)), a0, a1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), sl2x2,
                             f2_pack(l4.z, l4.w)), a2, a3);
            pk[c / 2] = f2_to_bf16x2(f2_pack(ex2(a0), ex2(a1)));
            pk[c / 2 + 1] = f2_to_bf16x2(f2_pack(ex2(a2), ex2(a3)));
          }
          // over S^T columns c1 / 2 .. c1 / 2 + 15, all read by chunk 0
          tmem_st16p(tS + c1 / 2, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p);
        // ---- dS^T = P^T o (dP^T - Delta) ----
        if (!mbar_wait(&bar_dp, g & 1, ac)) { ok = false; break; }
        // the dS tile is free: dP^T(g) went out after dQ^T(g-1), and its
        // commit arrives only once every earlier MMA has completed
        tc_fence_after();
#pragma unroll 1
        for (int c1 = 0; c1 < HALF; c1 += 32) {
          uint32_t u[32], pp[16];
          tmem_ld32_nowait(tDP + c1, u);
          tmem_ld16_nowait(tS + c1 / 2, pp);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const uint64_t pa = f2_pack(__uint_as_float(pp[c / 2] << 16),
                                        __uint_as_float(pp[c / 2] & 0xffff0000u));
            const uint64_t pb = f2_pack(__uint_as_float(pp[c / 2 + 1] << 16),
                                        __uint_as_float(pp[c / 2 + 1] & 0xffff0000u));
            const float4 d4 = *reinterpret_cast<const float4*>(&s_delta[c0 + c1 + c]);
            pk[c / 2] = f2_to_bf16x2(f2_mul(
                f2_sub(f2_pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), f2_pack(d4.x, d4.y)),
                pa));
            pk[c / 2 + 1] = f2_to_bf16x2(f2_mul(
                f2_sub(f2_pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])),
                       f2_pack(d4.z, d4.w)),
                pb));
          }
          tmem_st16p(tS + 32 + c1 / 2, pk);   // over S^T columns 32 .. 63 of this half
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int ch = (c0 + c1) / 8 + i;
            const uint32_t off = (ch >> 3) * BN * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(sdS + off) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
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
  } else if (warp < 16) {
    // ---------------- drain: dQ every step, dV and dK at the end of an item ----------------
    // dQ^T leaves TMEM in one load (64 query columns per warpgroup) and goes
    // to global memory straight from registers: the lane of a thread is a
    // head dim, so one warp instruction covers 32 consecutive dims (128
    // bytes) of one query row, added into the fp32 accumulator with
    // red.global.add.f32 (ATOMIC; SPLIT in a fixed order, below).  Measured
    // against TMA copies through a shared-memory tile (one 16 KB copy at a
    // time, then eight per-warp 2 KB copies), this keeps the SM's TMA unit
    // for the operand loads, and the freed shared memory holds the second dO
    // slot.
    const int t = threadIdx.x - 256;                   // 0..255
    const int grp = t >> 7;                            // column half
    const int tl = t & 127;                            // TMEM lane: head dim (dQ^T), K/V row (dV, dK)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    BwdItem w;
    int k = 0, ic = 0, gs = 0;
    ThdCursor cur;
    bool ok = true;
    // kOrdered: the ticket the last step's adds are behind, released at the
    // next step once its dQ^T has left TMEM (measured 1.92 ms for the c3
    // backward against 1.99 with releases batched over four steps, 2.36 with
    // the query tiles in ascending order)
    int* pend = nullptr;
    auto release_pending = [&]() {
      if (pend) {
        __threadfence();
        named_bar_sync(2, 256);
        if (t == 0) red_release_gpu_add1(pend);
        pend = nullptr;
      }
    };
    while (ok && next_bwd_item<BN, BM, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
      int ih = -1, ii = w.n_i - 1;   // step order: see next_step
      for (int it = 0; it < w.n_it; ++it) {
        next_step(ih, ii, G);
        const int g = gs + it;
        const int h = w.hk * G + ih;
        const int q = (w.i_start + ii) * BM + 64 * grp;   // first query row of this half
        if (!mbar_wait(&bar_dq_full, g & 1, ac)) { ok = false; break; }
        tc_fence_after();
        uint32_t u[64];
        tmem_ld32_nowait(tmem + lane_base + C::COL_DP + 64 * grp, u);
        tmem_ld32_nowait(tmem + lane_base + C::COL_DP + 64 * grp + 32, u + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_dq_empty);
        const int nq = min(64, w.seq.len - q);
        float* gq = a.dq_acc + ((static_cast<size_t>(w.seq.b) * p.heads_q + h) * p.rows_total +
                                w.seq.row0 + q) * C::D + tl;
        if constexpr (!kOrdered) {
          // The 64 adds per thread are paced over the step: a burst of them
          // fills the load/store queues the P/dS warps' shared-memory accesses
          // go through on the step's critical path.  After every 16 adds the
          // thread sleeps 400 ns unless the next step's dQ^T is already
          // waiting (c3 backward 1.447 -> 1.332 ms; a fixed 650 ns pause made
          // the drain the bottleneck, 1.62 ms, hence the test).
          if (nq > 0) {
            const uint32_t next_full = smem_u32(&bar_dq_full);
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              if (c < nq) atomicAdd(gq + static_cast<size_t>(c) * C::D, __uint_as_float(u[c]));
              if ((c & 15) == 15 && c < 63 && !mbar_test_wait(next_full, (g + 1) & 1)) __nanosleep(400);
            }
          }
        } else {
          // SPLIT (bitwise reproducible): the partials of a query tile go into
          // the accumulator in ascending K/V tile order.  K/V tile jt waits
          // until the tile's ticket says jt earlier tiles are in, stores (jt = 0:
          // the first contribution, the accumulator is not cleared) or adds,
          // and lets the next tile in.  A ticket only waits for items earlier
          // in the static item list (smaller jt), which every CTA walks in
          // order, and all CTAs are resident, so the waits cannot form a cycle;
          // holding a ticket back by one step does not change that (tile 0
          // never waits, and the last one is released at the end of the item).
          const int slot = w.x0 + (w.i_start + ii) * w.xs;
          release_pending();
          // a sequence longer than max_seqlen (flagged) can reach past the
          // ticket slots: its query tiles there are left out
          if (slot >= a.n_x) {
            if (t == 0 && p.err) atomicOr(p.err, ATTN_DEVERR_SEQLEN);
            continue;
          }
          int* tk = a.dq_ticket + (static_cast<size_t>(w.seq.b) * p.heads_q + h) * a.n_x + slot;
          if (t == 0) wait_ticket(tk, w.jt, ac);   // raises the abort flag if it runs out
          named_bar_sync(2, 256);
          if (*reinterpret_cast<volatile int*>(&abort_flag)) { ok = false; break; }
          if (nq > 0) {
            if (w.jt == 0) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c < nq) gq[static_cast<size_t>(c) * C::D] = __uint_as_float(u[c]);
            } else {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c < nq) atomicAdd(gq + static_cast<size_t>(c) * C::D, __uint_as_float(u[c]));
            }
          }
          pend = tk;
        }
      }
      if constexpr (kOrdered) release_pending();   // the item's last query tiles
      if (!ok) break;
      // ---- dV and dK (x scale) of this item: dims 64 grp .. 64 grp + 63 of row kv ----
      if (!mbar_wait(&bar_done, ic & 1, ac)) break;
      tc_fence_after();
      const int kv = w.kv0 + tl;
      const size_t grow = static_cast<size_t>(w.seq.b) * p.rows_total + w.seq.row0 + kv;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? C::COL_DV : C::COL_DK) + 64 * grp;
        const float mul = which == 0 ? 1.0f : p.scale;
        uint32_t pkx[32];
        {
          uint32_t x[64];
          tmem_ld32_nowait(tmem + lane_base + col, x);
          tmem_ld32_nowait(tmem + lane_base + col + 32, x + 32);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(which == 0 ? &bar_dv_empty : &bar_dk_empty);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pkx[c] = pack_bf16(__uint_as_float(x[2 * c]) * mul, __uint_as_float(x[2 * c + 1]) * mul);
        }
        // rows past the end of the sequence (or of the tensor) are not written
        if (kv < w.seq.len) {
          __nv_bfloat16* gdst =
              (which == 0 ? a.dv : a.dk) + (grow * p.heads_kv + w.hk) * C::D + 64 * grp;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(gdst + 8 * c) =
                make_uint4(pkx[4 * c], pkx[4 * c + 1], pkx[4 * c + 2], pkx[4 * c + 3]);
        }
      }
      gs += w.n_it;
      ++ic;
    }
  } else if constexpr (kPad) {
    // ---------------- warp 18: THD padding rows of dK and dV ----------------
    // Rows at or past cu_seqlens[num_seqs] are outputs of exact zeros; the CTA
    // writes its share of both tensors during the kernel, 4 KB at a time with
    // a 1 us pause while the MMA issuer still has items, so that the stores
    // neither crowd the load/store path of the other roles nor, once the
    // items are done, hold the CTA back.
    {
      const int lane = lane_id();
      const int end = valid_end(p);
      const size_t per_row = static_cast<size_t>(p.heads_kv) * C::D / 8;   // 16-byte words
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 17) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
    tmem_relinquish();
  }
}

}  // namespace

cudaError_t launch_attn_bwd128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dO, const BwdArgs& a, int grid, cudaStream_t st) {
  using C = Bwd128;
  const bool pad = a.pad_zero != 0;
  auto kern = a.split ? (pad ? attn_bwd128_kernel<true, false, true> : attn_bwd128_kernel<true, false, false>)
              : a.x_major == 3 ? attn_bwd128_kernel<false, true, true>
              : (pad ? attn_bwd128_kernel<false, false, true> : attn_bwd128_kernel<false, false, false>);
  const int threads = pad ? C::THREADS_PAD : C::THREADS;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, threads, C::SMEM, st>>>(q, k, v, dO, a);
  return cudaGetLastError();
}

}  // namespace attn
