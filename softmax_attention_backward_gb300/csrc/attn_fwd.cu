// Dense / GQA / THD attention forward with the row log-sum-exp saved for the
// backward (the `flashattn_fwd` stage of "[Example] Introduce split+sum
// template, and optimize atomic_add performance for bwd examples",
// tile-ai/tilelang #940, code-graph section).
//
// Work item = two 128-row query tiles of one (batch, query head); the CTA that
// runs it streams 128-row K/V tiles through a TMA ring:
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
// The grid is persistent (one CTA per SM walking a static item list, longest
// first; not for THD at D = 128): the next item's query tiles load into a
// second buffer and its first S MMAs run while the softmax warps write out the
// previous O.  A query tile that does not reach one of the item's K/V tiles
// still observes that tile's loads and releases their ring slots, so every
// issuer stays within one phase of every slot.
#include <cuda_runtime.h>

#include "launch.h"
#include "thd_order.cuh"

namespace attn {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                   // rows per query tile
  // rows per key/value tile: 64 for D = 128, so that S (64 columns), P (32
  // packed columns) and O (128 columns) of both query tiles fit in TMEM with
  // P in columns of its own
  static constexpr int BN = (D == 128) ? 64 : 128;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int NSLOT = 6;                  // K/V ring slots (D = 128: 5 measured 4% slower)
  static constexpr int QBUFS = 2;                  // query-pair buffers (next item prefetch)
  static constexpr int SMEM = QBUFS * 2 * Q_BYTES + NSLOT * KV_BYTES + 1024;
  static constexpr int THREADS = 352;
  static constexpr int THREADS_PAD = 384;   // with the padding warp (THD)
  static constexpr uint32_t TMEM_COLS = 512;
  // S0, S1 in columns [0, 2 BN); O0, O1 in [256, 256 + 2 D); each tile's P (BN/2
  // packed columns) in a region of its own, so S_w(j+1) can be computed while
  // the softmax of tile j runs: after S for D = 128, after O for D = 64.
  static constexpr uint32_t COL_S0 = 0, COL_S1 = BN, COL_O0 = 256, COL_O1 = 256 + D;
  static constexpr bool SEP_P = true;
  static constexpr uint32_t COL_P0 = (D == 128) ? 2 * BN : 256 + 2 * D;
  static constexpr uint32_t COL_P1 = COL_P0 + BN / 2;
  static_assert(2 * BN + BN <= 256 || D != 128, "S and P of both tiles below O");
  static_assert(256 + 2 * D <= 512 && (D == 128 || 256 + 2 * D + BN <= 512), "TMEM budget");
};

// One work item: the two 128-row query tiles m0 .. m0 + 255 of query head h;
// tile w meets n_w[w] key/value tiles, the pair n_kv = max of both.
struct FwdItem {
  SeqRef seq;
  int h, m0, n_w[2], n_kv;
};

// Advances the CTA's round counter `k` to its next valid item (same dealing
// as the backward: round k takes items k*G .. k*G + G - 1 in snake order).
// Numbering (`x_major`): 1 = pair slot slowest, so the list runs from the
// longest items to the shortest; 0 = pair slot fastest within each (batch,
// head), i.e. blockIdx order of the one-CTA-per-item grid.  Under causal
// masking the last pair of a sequence is the longest, so slots are reversed.
template <int BM, int BN, bool kThd>
__device__ __forceinline__ bool next_fwd_item(const Problem& p, int total, int n_x, int x_major,
                                              const FastDiv& fd_nbh, const FastDiv& fd_nx,
                                              const ThdOrder& thd, ThdCursor& cur, int& k,
                                              FwdItem& w) {
  const int G = gridDim.x, c = blockIdx.x;
  const int n_bh = p.heads_q * p.batch;
  if constexpr (kThd) {   // causal THD, the list of thd_order.cuh (numbering 3)
    for (; k * G < thd.n_items; ++k) {
      const int idx = k * G + ((k & 1) ? (G - 1 - c) : c);
      if (idx >= thd.n_items) continue;
      int pos, h;
      if (!thd_locate(thd, n_bh, fd_nbh, idx, cur, pos, h)) return false;
      const int sq = thd.seq[pos];
      const int t0 = __ldg(p.cu_seqlens + sq), t1 = __ldg(p.cu_seqlens + sq + 1);
      w.h = h;
      w.seq.b = 0;
      w.seq.row0 = t0;
      w.seq.len = t1 > t0 ? t1 - t0 : 0;
      w.m0 = (cur.v - 1) * 2 * BM;   // the pair of level v
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int r0 = w.m0 + t * BM;
        w.n_w[t] = r0 >= w.seq.len ? 0 : (min(w.seq.len, r0 + BM) + BN - 1) / BN;
      }
      w.n_kv = max(w.n_w[0], w.n_w[1]);
      ++k;
      return true;
    }
    return false;
  }
  for (; k * G < total; ++k) {
    const int idx = k * G + ((k & 1) ? (G - 1 - c) : c);
    if (idx >= total) continue;
    int bh, x;
    if (x_major) {
      x = static_cast<int>(fdiv(idx, fd_nbh));
      bh = idx - x * n_bh;
    } else {
      bh = static_cast<int>(fdiv(idx, fd_nx));
      x = idx - bh * n_x;
    }
    const int b = static_cast<int>(fdiv(bh, p.fd_hq));
    w.h = bh - b * p.heads_q;
    int pair;
    if (x_major == 2) {
      // THD: slot x is pair rank x / num_seqs of sequence x % num_seqs, so the
      // longest pairs of every sequence come first; ranks past a sequence's
      // end are empty
      const int q = static_cast<int>(fdiv(static_cast<uint32_t>(x), p.fd_ns));
      const int sq = x - q * p.num_seqs;
      const int t0 = __ldg(p.cu_seqlens + sq), t1 = __ldg(p.cu_seqlens + sq + 1);
      const int len = t1 > t0 ? t1 - t0 : 0;
      const int np = (len + 2 * BM - 1) / (2 * BM);
      // a sequence longer than max_seqlen may have pairs past the last slot
      if (q == 0 && np > 0 && (np - 1) * p.num_seqs + sq >= n_x && p.err)
        atomicOr(p.err, ATTN_DEVERR_SEQLEN);
      if (q >= np) continue;
      w.seq.b = 0;
      w.seq.row0 = t0;
      w.seq.len = len;
      pair = q;
    } else if (!decode_tile(p, x, b, 2 * BM, w.seq, pair)) {
      continue;
    }
    if (p.causal) pair = (w.seq.len + 2 * BM - 1) / (2 * BM) - 1 - pair;
    w.m0 = pair * 2 * BM;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = w.m0 + t * BM;
      if (r0 >= w.seq.len) {
        w.n_w[t] = 0;
      } else {
        const int kv_end = p.causal ? min(w.seq.len, r0 + BM) : w.seq.len;
        w.n_w[t] = (kv_end + BN - 1) / BN;
      }
    }
    w.n_kv = max(w.n_w[0], w.n_w[1]);
    if (w.n_kv <= 0) continue;
    ++k;
    return true;
  }
  return false;
}

// kThd: the instantiation for numbering 3; kPad: THD, with warp 11 writing
// the padding rows of O and LSE during the computation.  The others carry
// none of their code (the dense forward measured 2% slower with numbering 3
// in the same kernel).
template <int D, bool kThd, bool kPad>
__global__ void __launch_bounds__(kPad ? FwdCfg<D>::THREADS_PAD : FwdCfg<D>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int PANELS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                                   // QBUFS x 2 tiles
  uint8_t* sRing = sQ + C::QBUFS * 2 * C::Q_BYTES;      // NSLOT tiles

  __shared__ uint64_t bar_q[C::QBUFS], bar_qempty[C::QBUFS];
  __shared__ uint64_t bar_full[C::NSLOT], bar_empty[C::NSLOT];
  __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2], bar_sfree[2], bar_stagger;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int s_mma_done;   // an MMA issuer has left its item loop
  __shared__ ThdOrder s_thd;   // the item list of numbering 3

  const Problem& p = a.p;
  const int warp = warp_id();
  const int total = a.total_items;
  AbortCtx ac{&abort_flag, p.err};

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    abort_flag = 0;
    s_mma_done = 0;
    for (int b = 0; b < C::QBUFS; ++b) {
      mbar_init(&bar_q[b], 1);
      mbar_init(&bar_qempty[b], 2);      // released by both issuers
    }
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
  if constexpr (kThd)
    if (warp == 1) thd_order_build(p, 2 * C::BM, p.heads_q * p.batch, s_thd);
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
      auto issue_q = [&](const FwdItem& it, int icq) {
        const int qb = icq % C::QBUFS;
        mbar_arrive_expect_tx(&bar_q[qb], 2 * C::Q_BYTES);
        for (int t = 0; t < 2; ++t)
          for (int pn = 0; pn < PANELS; ++pn)
            tma_load_4d(&tmQ, &bar_q[qb], sQ + (qb * 2 + t) * C::Q_BYTES + pn * C::BM * 128,
                        pn * 64, it.h, it.seq.row0 + it.m0 + t * C::BM, it.seq.b);
      };
      FwdItem w, wn;
      int k = 0, ic = 0, gring = 0;
      ThdCursor cur;
      bool have = next_fwd_item<C::BM, C::BN, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w);
      bool ok = true;
      if (have) {
        if (mbar_wait(&bar_qempty[0], 1, ac)) issue_q(w, 0);
        else ok = false;
      }
      while (ok && have) {
        const int hk = static_cast<int>(fdiv(w.h, p.fd_grp));
        // the next item's query pair is loaded as soon as its buffer frees
        // (with two buffers: when the previous item's S MMAs are done), while
        // this item's K/V tiles stream through the ring
        const bool have_next = next_fwd_item<C::BM, C::BN, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, wn);
        bool q_pending = have_next;
        const int nqb = (ic + 1) % C::QBUFS;
        const uint32_t nq_par = (((ic + 1) / C::QBUFS) & 1) ^ 1;
        for (int i = 0; ok && i < 2 * w.n_kv; ++i) {
          const int gi = gring + i;
          const int slot = gi % C::NSLOT, use = gi / C::NSLOT;
          const uint32_t slot_addr = smem_u32(&bar_empty[slot]);
          const uint32_t slot_par = (use & 1) ^ 1;
          // bounded wait on the ring slot that also polls the next query buffer
          uint64_t t0 = 0;
          while (true) {
            if (q_pending && mbar_try_wait(smem_u32(&bar_qempty[nqb]), nq_par)) {
              issue_q(wn, ic + 1);
              q_pending = false;
            }
            if (mbar_try_wait(slot_addr, slot_par)) break;
            if (t0 == 0) t0 = globaltimer();
            if (*reinterpret_cast<volatile int*>(&abort_flag)) { ok = false; break; }
            if (globaltimer() - t0 > kWaitLimitNs) {
              raise_error(ac, ATTN_DEVERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          if (!ok) break;
          const CUtensorMap* m = (i & 1) ? &tmV : &tmK;
          uint8_t* dst = sRing + slot * C::KV_BYTES;
          mbar_arrive_expect_tx(&bar_full[slot], C::KV_BYTES);
          for (int pn = 0; pn < PANELS; ++pn)
            tma_load_4d(m, &bar_full[slot], dst + pn * C::BN * 128, pn * 64, hk,
                        w.seq.row0 + (i >> 1) * C::BN, w.seq.b);
        }
        if (ok && q_pending) {
          if (mbar_wait(&bar_qempty[nqb], nq_par, ac)) issue_q(wn, ic + 1);
          else ok = false;
        }
        gring += 2 * w.n_kv;
        ++ic;
        w = wn;
        have = have_next;
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ---------------- MMA issuer of query tile t ----------------
    const int t = warp - 9;
    {   // warp-uniform: one elected lane issues
      const uint32_t idS = idesc_bf16(C::BM, C::BN, false, false);
      const uint32_t idO = idesc_bf16(C::BM, D, false, true);
      const uint64_t dR_k0 = desc_kmajor_base(smem_u32(sRing));
      const uint64_t dR_mn0 = desc_mnmajor_base(smem_u32(sRing), C::BN);
      const uint32_t tS = tmem + (t ? C::COL_S1 : C::COL_S0);
      const uint32_t tO = tmem + (t ? C::COL_O1 : C::COL_O0);
      const uint32_t tP = tmem + (t ? C::COL_P1 : C::COL_P0);
      FwdItem w;
      int k = 0, ic = 0, gring = 0, cs = 0;   // cs: S tiles of this query tile so far
      ThdCursor cur;
      bool ok = true;
      while (ok && next_fwd_item<C::BM, C::BN, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
        const int qb = ic % C::QBUFS, qu = ic / C::QBUFS;
        const int nt = w.n_w[t];
        if (!mbar_wait_w(&bar_q[qb], qu & 1, ac)) break;
        // Tile 1 starts one softmax phase after tile 0 (when P_0(0) of the
        // first item is ready), so that one tile's softmax overlaps the other
        // tile's MMAs instead of both running in lockstep.  bar_stagger
        // completes exactly once.
        if (t == 1 && ic == 0 && !mbar_wait_w(&bar_stagger, 0, ac)) break;
        const uint64_t dQt = desc_kmajor_base(smem_u32(sQ + (qb * 2 + t) * C::Q_BYTES));
        auto issue_s = [&](int j) -> bool {
          const int gi = gring + 2 * j, sk = gi % C::NSLOT;
          if (!mbar_wait_w(&bar_full[sk], (gi / C::NSLOT) & 1, ac)) return false;
          tc_fence_after();
          const uint64_t kd = desc_advance(dR_k0, sk * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss_w(tS, desc_advance(dQt, kmajor_step_bytes(C::BM, kk)),
                    desc_advance(kd, kmajor_step_bytes(C::BN, kk)), idS, kk > 0);
          umma_commit_w(&bar_s[t]);
          umma_commit_w(&bar_empty[sk]);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int gi = gring + 2 * j + 1, sv = gi % C::NSLOT;
          if (!mbar_wait_w(&bar_full[sv], (gi / C::NSLOT) & 1, ac)) return false;
          if (!mbar_wait_w(&bar_p[t], (cs + j) & 1, ac)) return false;
          if (t == 0 && ic == 0 && j == 0 && lane_id() == 0) mbar_arrive(&bar_stagger);
          tc_fence_after();
          const uint64_t vd = desc_advance(dR_mn0, sv * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)   // P: 8 packed columns per 16 keys
            umma_ts_w(tO, tP + 8 * kk, desc_advance(vd, mnmajor_step_bytes(kk)), idO,
                    (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&bar_o[t]);
          umma_commit_w(&bar_empty[sv]);
          return true;
        };
        if (C::SEP_P) {
          // S(j+1) as soon as the softmax has read S(j); PV(j) once P(j) is
          // ready.  S(0) of an item waits for the read of the previous S.
          for (int j = 0; ok && j < nt; ++j) {
            if (j == 0) {
              if (cs > 0 && !mbar_wait_w(&bar_sfree[t], (cs - 1) & 1, ac)) { ok = false; break; }
              if (!issue_s(0)) { ok = false; break; }
            }
            if (j + 1 < nt) {
              if (!mbar_wait_w(&bar_sfree[t], (cs + j) & 1, ac) || !issue_s(j + 1)) {
                ok = false;
                break;
              }
            }
            if (!issue_pv(j)) ok = false;
          }
        } else {
          // S(j), PV(j), S(j+1), ...: MMAs of one thread execute in order, so
          // S(j+1) cannot overwrite P(j) (stored over S) before PV(j) read it
          for (int j = 0; ok && j < nt; ++j)
            if (!issue_s(j) || !issue_pv(j)) ok = false;
        }
        // K/V tiles of the item this query tile does not reach: its issuer
        // still waits for each load and releases the slot itself.  A parity
        // wait is only sound while the waiter is at most one phase behind;
        // releasing skipped slots on the tile's behalf would let the ring run
        // on, and this tile's next wait on a slot would then see a completed
        // phase of matching parity that is not the one it waits for (found
        // with THD sequences whose last query pair has one tile past the end).
        for (int j = nt; ok && j < w.n_kv; ++j) {
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int gi = gring + 2 * j + kv, sl = gi % C::NSLOT;
            if (!mbar_wait_w(&bar_full[sl], (gi / C::NSLOT) & 1, ac)) { ok = false; break; }
            if (lane_id() == 0) mbar_arrive(&bar_empty[sl]);
          }
        }
        // the query tile is free once this tile's S MMAs have completed
        if (ok) {
          if (nt > 0) umma_commit_w(&bar_qempty[qb]);
          else if (lane_id() == 0) mbar_arrive(&bar_qempty[qb]);
        }
        gring += 2 * w.n_kv;
        cs += nt;
        ++ic;
      }
    }
    if constexpr (kPad) *reinterpret_cast<volatile int*>(&s_mma_done) = 1;
  } else if (kPad ? warp < 8 : true) {
    // ---------------- softmax warpgroups ----------------
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int tr = threadIdx.x & 127;        // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = tmem + lane_base + (t ? C::COL_O1 : C::COL_O0);
    const uint32_t tP = tmem + lane_base + (t ? C::COL_P1 : C::COL_P0);
    const float sl2 = a.scale_log2;
    FwdItem w;
    int k = 0, cs = 0;
    ThdCursor cur;
    bool ok = true;
    while (ok && next_fwd_item<C::BM, C::BN, kThd>(p, total, a.n_x, a.x_major, a.fd_nbh, a.fd_nx, s_thd, cur, k, w)) {
      const int row = w.m0 + t * C::BM + tr;   // row inside the sequence
      const int nt = w.n_w[t];
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nt; ++j) {
        const int c = cs + j;
        // without a separate P region, S_t(j) complete also means PV_t(j-1) is
        // complete (same issuer, in order)
        if (!mbar_wait(&bar_s[t], c & 1, ac)) { ok = false; break; }
        tc_fence_after();
        float s[C::BN];
        {
          uint32_t u[C::BN];
#pragma unroll
          for (int cc = 0; cc < C::BN; cc += 32) tmem_ld32_nowait(tS + cc, u + cc);
          tmem_wait_ld();
          if (C::SEP_P) {
            tc_fence_before();
            mbar_arrive(&bar_sfree[t]);
          }
#pragma unroll
          for (int cc = 0; cc < C::BN; ++cc) s[cc] = __uint_as_float(u[cc]);
        }
        const int kv0 = j * C::BN;
        const bool need_mask =
            (kv0 + C::BN > w.seq.len) || (p.causal && kv0 + C::BN - 1 > w.m0 + t * C::BM);
        if (need_mask) {
          const int lim = p.causal ? min(w.seq.len - 1, row) : w.seq.len - 1;
#pragma unroll
          for (int cc = 0; cc < C::BN; ++cc)
            if (kv0 + cc > lim) s[cc] = -INFINITY;
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
        const float mt =
            fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7]))) * sl2;
        const float m_new = fmaxf(m_run, mt);
        const bool grow = m_new > m_run + 8.0f;          // also true on the first finite max
        const float m_use = grow ? m_new : m_run;
        const float alpha = grow ? ex2(m_run - m_use) : 1.0f;
        const float msub = (m_use == -INFINITY) ? 0.f : m_use;
        const bool warp_rescale = j > 0 && __any_sync(0xffffffffu, grow);
        // P = 2^(S * scale * log2 e - m): packed fp32x2 argument, row sum in
        // four packed partial sums, bf16 pairs for the PV MMA
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t nm2 = f2_pack(-msub, -msub);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[C::BN / 2];
#pragma unroll
        for (int cc = 0; cc < C::BN; cc += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[cc], s[cc + 1]), sl2x2, nm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          rs2[(cc >> 1) & 3] = f2_add(rs2[(cc >> 1) & 3], f2_pack(p0, p1));
          pk[cc / 2] = pack_bf16(p0, p1);
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
          if (!mbar_wait(&bar_o[t], (c - 1) & 1, ac)) { ok = false; break; }
          tc_fence_after();
        }
        if (warp_rescale) {
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t r[32];
            tmem_ld32_nowait(tO + cc, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + cc, r);
          }
        }
        // P (bf16 pairs): BN / 2 packed columns
#pragma unroll
        for (int cc = 0; cc < C::BN / 2; cc += 32) tmem_st32(tP + cc, pk + cc);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p[t]);
      }
      // ---- epilogue: O / l, LSE (the next item's first PV waits for the P
      // this warpgroup writes after reading O here) ----
      if (ok && nt > 0 && mbar_wait(&bar_o[t], (cs + nt - 1) & 1, ac)) {
        tc_fence_after();
        const bool valid = row < w.seq.len;
        const float inv_l = (l_run > 0.f) ? 1.0f / l_run : 0.f;
        const size_t grow_idx = (static_cast<size_t>(w.seq.b) * p.rows_total + w.seq.row0 + row);
        __nv_bfloat16* orow = a.o + (grow_idx * p.heads_q + w.h) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t r[32];
          tmem_ld32_nowait(tO + cc, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[i + 0]) * inv_l, __uint_as_float(r[i + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(r[i + 2]) * inv_l, __uint_as_float(r[i + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(r[i + 4]) * inv_l, __uint_as_float(r[i + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(r[i + 6]) * inv_l, __uint_as_float(r[i + 7]) * inv_l);
            if (valid) *reinterpret_cast<uint4*>(orow + cc + i) = v;
          }
        }
        if (valid) {
          const float lse = (l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
          size_t li;
          if (p.cu_seqlens)
            li = static_cast<size_t>(w.h) * p.rows_total + w.seq.row0 + row;
          else
            li = (static_cast<size_t>(w.seq.b) * p.heads_q + w.h) * p.rows_total + row;
          a.lse[li] = lse;
        }
      }
      cs += nt;
    }
  } else if constexpr (kPad) {
    // ---------------- warp 11: THD padding rows of O and LSE ----------------
    // Rows at or past cu_seqlens[num_seqs]: O exact zeros, LSE -inf.  The CTA
    // writes its slice during the computation, 4 KB of O at a time with a 1 us
    // pause while the MMA issuers still have items.
    const int lane = lane_id();
    const int end = valid_end(p);
    const uint32_t rows = static_cast<uint32_t>(p.rows_total - end);
    const size_t per_row = static_cast<size_t>(p.heads_q) * D / 8;   // 16-byte words of O
    const size_t n = rows * per_row;
    const size_t lo = n * blockIdx.x / gridDim.x, hi = n * (blockIdx.x + 1) / gridDim.x;
    uint4* o4 = reinterpret_cast<uint4*>(a.o) + static_cast<size_t>(end) * per_row;
    int it = 0;
    for (size_t i = lo + lane; i < hi; i += 32) {
      o4[i] = make_uint4(0u, 0u, 0u, 0u);
      if ((++it & 7) == 0 && !*reinterpret_cast<volatile int*>(&s_mma_done)) __nanosleep(1000);
    }
    const uint64_t nl = static_cast<uint64_t>(rows) * static_cast<uint32_t>(p.heads_q);
    const uint32_t llo = static_cast<uint32_t>(nl * blockIdx.x / gridDim.x);
    const uint32_t lhi = static_cast<uint32_t>(nl * (blockIdx.x + 1) / gridDim.x);
    for (uint32_t i = llo + lane; i < lhi; i += 32) {
      const uint32_t hh = i / rows, r = i - hh * rows;
      a.lse[static_cast<size_t>(hh) * p.rows_total + end + r] = -INFINITY;
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
template <int D>
cudaError_t launch_attn_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x, cudaStream_t st) {
  using C = FwdCfg<D>;
  const bool pad = a.p.cu_seqlens != nullptr;
  auto kern = !pad ? attn_fwd_kernel<D, false, false>
              : a.x_major == 3 ? attn_fwd_kernel<D, true, true> : attn_fwd_kernel<D, false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid_x, pad ? C::THREADS_PAD : C::THREADS, C::SMEM, st>>>(q, k, v, a);
  return cudaGetLastError();
}

template cudaError_t launch_attn_fwd<64>(const CUtensorMap&, const CUtensorMap&,
                                         const CUtensorMap&, const FwdArgs&, int, cudaStream_t);
template cudaError_t launch_attn_fwd<128>(const CUtensorMap&, const CUtensorMap&,
                                          const CUtensorMap&, const FwdArgs&, int, cudaStream_t);

}  // namespace attn
