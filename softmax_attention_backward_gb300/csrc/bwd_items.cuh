// Work items of the dense / GQA / THD backward kernels and their static
// schedule over a persistent grid (shared by the D = 64 and D = 128 kernels).
#pragma once

#include "attn.h"
#include "common.cuh"
#include "thd_order.cuh"

namespace attn {

// One work item: K/V tile `jt` (rows kv0 .. kv0 + 127 of the sequence) of kv
// head `hk`, and the n_it = groups * n_i query tiles it meets.  x0 + xs * i
// numbers query tile i of the sequence among the n_x slots of a (batch, head):
// x0 is the slot of the sequence's first tile and xs = 1 (slots sequence by
// sequence; 0 and 1 for dense problems), or x0 is the sequence and xs the
// number of sequences (slots tile-major, see next_bwd_item).
struct BwdItem {
  SeqRef seq;
  int hk, jt, kv0, i_start, n_i, n_it, x0, xs;
};

// Advances the CTA's round counter `k` to its next valid item.  Round k of
// the CTA grid takes items k*G .. k*G + G - 1, dealt in snake order (CTA c
// takes c in even rounds and G - 1 - c in odd ones) to even out the per-CTA
// work; with one CTA per item (G = total) this is plain blockIdx order.
// Numbering (`x_major`):
//  * 1 (persistent grid): tile slot x slowest, so the list runs from the
//    longest items to the shortest under causal masking (tile 0 of a sequence
//    meets every query tile, the last tile only the last one);
//  * 2 (persistent grid, THD): as 1, but slot x is tile x / num_seqs of
//    sequence x % num_seqs, so the first tiles of every sequence come before
//    the later tiles of any (numbered sequence by sequence, a long sequence's
//    first tiles would come after a shorter one's last ones); slots past a
//    sequence's end are empty;
//  * 3 (persistent grid, causal THD of at most 32 sequences): the list of
//    thd_order.cuh, in descending order of work without empty positions;
//  * 0 (one CTA per item): tile slot fastest within each (batch, kv head),
//    in reverse, so CTAs resident together work on the same heads.
template <int BN, int BM, bool kThd>
__device__ __forceinline__ bool next_bwd_item(const Problem& p, int total, int n_x, int x_major,
                                              const FastDiv& fd_nbh, const FastDiv& fd_nx,
                                              const ThdOrder& thd, ThdCursor& cur, int& k,
                                              BwdItem& w) {
  const int G = gridDim.x, c = blockIdx.x;
  const int groups = static_cast<int>(p.fd_grp.d);
  const int n_bh = p.heads_kv * p.batch;
  if constexpr (kThd) {   // numbering 3 (the other numberings carry none of its code)
    for (; k * G < thd.n_items; ++k) {
      const int idx = k * G + ((k & 1) ? (G - 1 - c) : c);
      if (idx >= thd.n_items) continue;
      int pos, h;
      if (!thd_locate(thd, n_bh, fd_nbh, idx, cur, pos, h)) return false;
      const int sq = thd.seq[pos];
      const int t0 = __ldg(p.cu_seqlens + sq), t1 = __ldg(p.cu_seqlens + sq + 1);
      w.hk = h;
      w.seq.b = 0;
      w.seq.row0 = t0;
      w.seq.len = t1 > t0 ? t1 - t0 : 0;
      w.x0 = sq;
      w.xs = p.num_seqs;
      w.jt = thd.n_sorted[pos] - cur.v;   // K/V tile meeting v query tiles
      w.kv0 = w.jt * BN;
      w.i_start = w.kv0 / BM;
      w.n_i = (w.seq.len + BM - 1) / BM - w.i_start;
      w.n_it = groups * w.n_i;
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
    const int b = static_cast<int>(fdiv(bh, p.fd_hkv));
    w.hk = bh - b * p.heads_kv;
    int jt;
    if (x_major == 2) {
      const int q = static_cast<int>(fdiv(static_cast<uint32_t>(x), p.fd_ns));
      const int sq = x - q * p.num_seqs;
      const int t0 = __ldg(p.cu_seqlens + sq), t1 = __ldg(p.cu_seqlens + sq + 1);
      const int len = t1 > t0 ? t1 - t0 : 0;
      const int nt = (len + BN - 1) / BN;
      // a sequence longer than max_seqlen may have tiles past the last slot
      if (q == 0 && nt > 0 && (nt - 1) * p.num_seqs + sq >= n_x && p.err)
        atomicOr(p.err, ATTN_DEVERR_SEQLEN);
      if (q >= nt) continue;
      jt = q;
      w.seq.b = 0;
      w.seq.row0 = t0;
      w.seq.len = len;
      w.x0 = sq;
      w.xs = p.num_seqs;
    } else {
      if (!decode_tile(p, x, b, BN, w.seq, jt)) continue;
      w.x0 = x - jt;
      w.xs = 1;
      if (!x_major && p.causal) jt = (w.seq.len + BN - 1) / BN - 1 - jt;
    }
    w.jt = jt;
    w.kv0 = jt * BN;
    w.i_start = p.causal ? w.kv0 / BM : 0;
    w.n_i = (w.seq.len + BM - 1) / BM - w.i_start;
    w.n_it = groups * w.n_i;
    if (w.n_it <= 0) continue;
    ++k;
    return true;
  }
  return false;
}

}  // namespace attn
