// Item order of the persistent kernels for causal THD packs of at most 32
// sequences (numbering 3 of next_fwd_item / next_bwd_item): the items in
// descending order of work, with no empty list positions.
//
// A sequence of n units (forward: 256-row query-tile pairs; backward: 128-row
// K/V tiles) has one unit at every work level v = 1 .. n: forward pair v - 1
// meets about 2v K/V tiles, backward K/V tile n - v meets v query tiles.  The
// list runs from the top level down; level v holds, for every sequence with
// n >= v, its unit of that level for every head (head fastest).  Dealt to the
// CTAs in snake order, the list then approaches the greedy longest-first
// assignment, where the numbering by unit rank (numbering 2) gave the same
// rank of a short and a long sequence the same place although their work
// differs.  Within a sequence the backward still meets its K/V tiles in
// ascending order, which the ordered dQ accumulation relies on.
#pragma once

#include "attn.h"
#include "common.cuh"

namespace attn {

constexpr int kThdOrderSeqs = 32;

struct ThdOrder {
  int n_sorted[kThdOrderSeqs];   // units per sequence, descending (ties: lower index first)
  int seq[kThdOrderSeqs];        // sequence of each sorted position
  int ns;                        // sequences
  int n_items;                   // items in the list (units x heads)
};

// A role's position in the list: level v (0 before the first lookup), the
// list index where the level starts, and how many sequences reach it.
struct ThdCursor {
  int v = 0, start = 0, cnt = 0;
};

// Fills `o` (one full warp; p.num_seqs <= 32).  Units past the max_seqlen
// bound are dropped and flagged as ATTN_DEVERR_SEQLEN.
__device__ __forceinline__ void thd_order_build(const Problem& p, int unit_rows, int n_bh,
                                                ThdOrder& o) {
  const int lane = threadIdx.x & 31;
  const int ns = p.num_seqs;
  const int umax = (p.max_seqlen + unit_rows - 1) / unit_rows;
  int n = 0;
  if (lane < ns) {
    const int t0 = __ldg(p.cu_seqlens + lane), t1 = __ldg(p.cu_seqlens + lane + 1);
    const int len = t1 > t0 ? t1 - t0 : 0;
    n = (len + unit_rows - 1) / unit_rows;
    if (n > umax) {
      if (p.err) atomicOr(p.err, ATTN_DEVERR_SEQLEN);
      n = umax;
    }
  }
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kThdOrderSeqs; ++j) {
    const int nj = __shfl_sync(0xffffffffu, n, j);
    rank += (j < ns && j != lane && (nj > n || (nj == n && j < lane))) ? 1 : 0;
  }
  if (lane < ns) {
    o.n_sorted[rank] = n;
    o.seq[rank] = lane;
  }
  int tot = n;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  if (lane == 0) {
    o.ns = ns;
    o.n_items = tot * n_bh;
  }
}

// List index idx (non-decreasing from call to call on one cursor) -> the
// sorted position `pos` and head `h` of the item, its level in c.v; false
// when idx is past the end of the list.
__device__ __forceinline__ bool thd_locate(const ThdOrder& o, int n_bh, const FastDiv& fd_nbh,
                                           int idx, ThdCursor& c, int& pos, int& h) {
  if (c.v == 0 && c.start == 0 && c.cnt == 0) {   // first lookup: the top level
    c.v = o.ns > 0 ? o.n_sorted[0] : 0;
    while (c.cnt < o.ns && o.n_sorted[c.cnt] >= c.v && c.v > 0) ++c.cnt;
  }
  while (c.v > 0 && idx >= c.start + c.cnt * n_bh) {
    c.start += c.cnt * n_bh;
    --c.v;
    while (c.cnt < o.ns && o.n_sorted[c.cnt] >= c.v && c.v > 0) ++c.cnt;
  }
  if (c.v <= 0) return false;
  const int r = idx - c.start;
  pos = static_cast<int>(fdiv(static_cast<uint32_t>(r), fd_nbh));
  h = r - pos * n_bh;
  return true;
}

}  // namespace attn
