// DSA lightning indexer: logits, top-k selection and backward ("[2/2] Add
// TileLang fused DSA kernels support with THD and CP & Clean up", Megatron-LM
// #5049: fused indexer forward with logits cleaning, fused indexer backward,
// top-k with -1 sentinels / compact prefix).  Formulas and layouts: dsa.h.
//
// dsa_indexer_logits_kernel (tcgen05): one CTA per (query tile i, key tile j)
// of 128 x 128 tokens.  The key tile loads once; the 64 (or fewer) query-head
// tiles stream through a 4-stage TMA ring, and for each head h the issuer
// computes Z_h = Q_h K^T (M = N = 128, K = 128) into one of four TMEM buffers
// while eight epilogue warps fold the previous heads into their fp32 logits,
// acc += w[t, h] * relu(Z_h) (each warp owns 32 rows x 64 columns).  Key tiles
// wholly after the query tile only write -inf.
//
// dsa_topk_kernel: one CTA per row; the visible part of the row is loaded
// into shared memory as order-preserving 32-bit keys and the k-th largest is
// found by up to four 8-bit radix passes (warp-aggregated histogram atomics, a
// warp-parallel digit pick, and an early stop once a digit's bin holds exactly
// the keys still needed); the selected positions (ties toward the smaller
// index) are then compacted in index order, each warp walking a contiguous
// segment with ballot counts and one scan of the warp totals, which yields the
// ascending key order directly.
//
// dsa_indexer_bwd_kernel (tcgen05): one CTA per token.  Its query heads
// (64 x 128) load once; its key rows are gathered 64 slots at a time.  Per
// chunk: Z = Q K^T (M = 64 heads, N = 64 slots); the epilogue warps form
// dZ = g w act'(Z) (bf16 [head][slot] tile) and accumulate dw; then
// dQ^T += K^T dZ^T (M = 128 dims, N = 64 heads) and two dK pieces
// dZ^T Q_p (M = 64 slots, N = 64 dims) which four drain warps add into the
// fp32 dK accumulator with vector reductions.
#include <cuda_runtime.h>

#include "dsa.h"
#include "launch.h"

namespace attn {
namespace {

// ---------------------------------------------------------------------------
// Indexer logits
// ---------------------------------------------------------------------------
constexpr int IX_T = 128;                       // tokens per tile (query and key)
constexpr int IX_D = 128;                       // index head dim
constexpr int IX_MAXH = 64;                     // index heads
constexpr int IX_NQ = 4;                        // query-head stages
constexpr int IX_NZ = 4;                        // TMEM Z buffers (128 columns each)
constexpr int IX_TILE = IX_T * IX_D * 2;        // 32 KB bf16 tile (two 64-dim panels)
constexpr int IX_SMEM = IX_TILE * (1 + IX_NQ) + IX_MAXH * IX_T * 4 + 1024;
constexpr int IX_THREADS = 320;                 // 8 epilogue warps, TMA warp, MMA warp

struct IxArgs {
  const float* w;
  float* logits;
  const int32_t* cu;
  int T, H, nseq, ld, use_relu;
  int32_t* err;
};

// First key token visible to query t (its sequence start), and whether t sees
// any key at all (THD padding tokens see none).
__device__ __forceinline__ void seq_of(const int32_t* cu, int nseq, int T, int t, int& lo,
                                       bool& any) {
  if (!cu) {
    lo = 0;
    any = t < T;
    return;
  }
  const int end = __ldg(cu + nseq);
  if (t >= end || t < __ldg(cu)) {
    lo = 0;
    any = false;
    return;
  }
  int a = 0, b = nseq;                          // last n with cu[n] <= t
  while (b - a > 1) {
    const int m = (a + b) >> 1;
    if (__ldg(cu + m) <= t) a = m; else b = m;
  }
  lo = __ldg(cu + a);
  any = true;
}

__global__ void __launch_bounds__(IX_THREADS, 1)
    dsa_indexer_logits_kernel(const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmK, const IxArgs a) {
  const int jt = blockIdx.x, it = blockIdx.y;
  const int t0 = it * IX_T, s0 = jt * IX_T;
  const int warp = warp_id(), lane = lane_id();
  if (jt > it) {
    // every key of the tile comes after every query of the tile
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int e = threadIdx.x; e < IX_T * (IX_T / 4); e += IX_THREADS) {
      const int r = e / (IX_T / 4), c = (e % (IX_T / 4)) * 4;
      const int t = t0 + r, s = s0 + c;
      if (t >= a.T || s >= a.T) continue;
      float* dst = a.logits + static_cast<size_t>(t) * a.ld + s;
      if (s + 3 < a.T) {
        *reinterpret_cast<float4*>(dst) = ninf;
      } else {
        for (int k = 0; s + k < a.T; ++k) dst[k] = -INFINITY;
      }
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sQ = sK + IX_TILE;                   // IX_NQ stages
  float* sW = reinterpret_cast<float*>(sQ + IX_NQ * IX_TILE);   // [head][row]
  __shared__ uint64_t bar_k, bar_qf[IX_NQ], bar_qe[IX_NQ], bar_zf[IX_NZ], bar_ze[IX_NZ];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  AbortCtx ac{&abort_flag, a.err};
  const int H = a.H;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_k, 1);
    for (int i = 0; i < IX_NQ; ++i) {
      mbar_init(&bar_qf[i], 1);
      mbar_init(&bar_qe[i], 1);
    }
    for (int i = 0; i < IX_NZ; ++i) {
      mbar_init(&bar_zf[i], 1);
      mbar_init(&bar_ze[i], 256);
    }
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, 512);
  if (warp < 8) {
    // weights of the tile's query rows, transposed to [head][row]
    for (int e = threadIdx.x; e < H * IX_T; e += 256) {
      const int h = e / IX_T, r = e % IX_T;
      const int t = t0 + r;
      sW[e] = t < a.T ? __ldg(a.w + static_cast<size_t>(t) * H + h) : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(&bar_k, IX_TILE);
#pragma unroll
      for (int pn = 0; pn < 2; ++pn)
        tma_load_4d(&tmK, &bar_k, sK + pn * IX_T * 128, pn * 64, 0, s0, 0);
      for (int h = 0; h < H; ++h) {
        const int st = h % IX_NQ;
        if (!mbar_wait(&bar_qe[st], ((h / IX_NQ) & 1) ^ 1, ac)) break;
        mbar_arrive_expect_tx(&bar_qf[st], IX_TILE);
#pragma unroll
        for (int pn = 0; pn < 2; ++pn)
          tma_load_4d(&tmQ, &bar_qf[st], sQ + st * IX_TILE + pn * IX_T * 128, pn * 64, h, t0, 0);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    const uint32_t idZ = idesc_bf16(128, 128, false, false);
    const uint64_t dK = desc_kmajor_base(smem_u32(sK));
    bool ok = mbar_wait_w(&bar_k, 0, ac);
    for (int h = 0; ok && h < H; ++h) {
      const int st = h % IX_NQ, zb = h % IX_NZ;
      if (!mbar_wait_w(&bar_qf[st], (h / IX_NQ) & 1, ac)) { ok = false; break; }
      if (!mbar_wait_w(&bar_ze[zb], ((h / IX_NZ) & 1) ^ 1, ac)) { ok = false; break; }
      tc_fence_after();
      const uint64_t dQ = desc_kmajor_base(smem_u32(sQ + st * IX_TILE));
#pragma unroll
      for (int kk = 0; kk < IX_D / 16; ++kk)
        umma_ss_w(tmem + zb * 128, desc_advance(dQ, kmajor_step_bytes(IX_T, kk)),
                  desc_advance(dK, kmajor_step_bytes(IX_T, kk)), idZ, kk > 0 ? 1u : 0u);
      umma_commit_w(&bar_zf[zb]);
      umma_commit_w(&bar_qe[st]);
    }
  } else {
    // ---------------- epilogue: acc += w relu(Z_h), then mask and store ----------------
    const int q = warp & 3, half = warp >> 2;
    const int r = 32 * q + lane;                 // tile row (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float acc[64];
#pragma unroll
    for (int k = 0; k < 64; ++k) acc[k] = 0.f;
    bool ok = true;
    for (int h = 0; h < H; ++h) {
      const int zb = h % IX_NZ;
      if (!mbar_wait(&bar_zf[zb], (h / IX_NZ) & 1, ac)) { ok = false; break; }
      tc_fence_after();
      uint32_t u[64];
      tmem_ld32_nowait(tmem + lane_base + zb * 128 + 64 * half, u);
      tmem_ld32_nowait(tmem + lane_base + zb * 128 + 64 * half + 32, u + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_ze[zb]);
      const float wv = sW[h * IX_T + r];
      const uint64_t w2 = f2_pack(wv, wv);
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        float z0 = __uint_as_float(u[k]), z1 = __uint_as_float(u[k + 1]);
        if (a.use_relu) {
          z0 = fmaxf(z0, 0.f);
          z1 = fmaxf(z1, 0.f);
        }
        float lo, hi;
        f2_unpack(f2_fma(w2, f2_pack(z0, z1), f2_pack(acc[k], acc[k + 1])), lo, hi);
        acc[k] = lo;
        acc[k + 1] = hi;
      }
    }
    const int t = t0 + r;
    if (ok && t < a.T) {
      int lo;
      bool any;
      seq_of(a.cu, a.nseq, a.T, t, lo, any);
      float* dst = a.logits + static_cast<size_t>(t) * a.ld;
      const int sb = s0 + 64 * half;
#pragma unroll
      for (int k = 0; k < 64; k += 4) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = sb + k + e;
          v[e] = (any && s >= lo && s <= t) ? acc[k + e] : -INFINITY;
        }
        const int s = sb + k;
        if (s + 3 < a.T) {
          *reinterpret_cast<float4*>(dst + s) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
          for (int e = 0; e < 4 && s + e < a.T; ++e) dst[s + e] = v[e];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
    tmem_relinquish();
  }
}

// ---------------------------------------------------------------------------
// Top-k selection
// ---------------------------------------------------------------------------
constexpr int TK_THREADS = 512;
constexpr int TK_MAXN = 8192;                   // visible keys held in shared memory per pass

// Order-preserving key of a float (larger float -> larger key); NaN -> 0.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;
  // -0.0 takes the key of +0.0: equal values, so the index decides between them
  const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(TK_THREADS) dsa_topk_kernel(const IxArgs a, int K,
                                                             int32_t* idx, int32_t* length,
                                                             float* scores) {
  __shared__ uint32_t s_key[TK_MAXN];
  __shared__ int s_hist[256];
  __shared__ int s_warp[2 * (TK_THREADS / 32)];
  __shared__ uint32_t s_sel[3];                 // digit chosen, keys still needed, its bin count
  const int t = blockIdx.x;
  int lo;
  bool any;
  seq_of(a.cu, a.nseq, a.T, t, lo, any);
  const int n = any ? t - lo + 1 : 0;
  int32_t* irow = idx + static_cast<size_t>(t) * K;
  float* srow = scores + static_cast<size_t>(t) * K;
  const float* lrow = a.logits + static_cast<size_t>(t) * a.ld;
  if (n <= K) {
    for (int i = threadIdx.x; i < K; i += TK_THREADS) {
      irow[i] = i < n ? lo + i : -1;
      srow[i] = i < n ? lrow[lo + i] : -INFINITY;
    }
    if (threadIdx.x == 0) length[t] = n;
    return;
  }
  // n > K (n <= T <= TK_MAXN): keys of the visible part of the row
  for (int i = threadIdx.x; i < n; i += TK_THREADS) s_key[i] = order_key(lrow[lo + i]);
  // Radix select of the K-th largest key, 8 bits per pass from the top.  A pass
  // stops the search early when the chosen digit's bin holds exactly the keys
  // still needed: then every key of that prefix class is taken.
  uint32_t prefix = 0, pmask = 0;
  int remaining = K;                            // keys still to take inside the prefix class
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += TK_THREADS) s_hist[i] = 0;
    __syncthreads();
    // histogram of the next digit within the prefix class; lanes holding the
    // same digit add once (the top digits of a row take few distinct values)
    for (int i0 = 0; i0 < n; i0 += TK_THREADS) {
      const int i = i0 + threadIdx.x;
      int dg = -1;
      if (i < n) {
        const uint32_t u = s_key[i];
        if ((u & pmask) == prefix) dg = static_cast<int>((u >> shift) & 0xFF);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, dg);
      if (dg >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[dg], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255 - 8l .. 248 - 8l; suffix counts by an inclusive scan
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = s_hist[255 - 8 * lane - j];
        tot += cnt[j];
      }
      int inc = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, inc >= remaining);
      const int L = __ffs(hit) - 1;              // first lane reaching `remaining` (exists: total >= remaining)
      if (lane == L) {
        int before = inc - tot, d = 255 - 8 * lane - 7, c = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (before + cnt[j] >= remaining) {
            d = 255 - 8 * lane - j;
            c = cnt[j];
            break;
          }
          before += cnt[j];
        }
        s_sel[0] = static_cast<uint32_t>(d);
        s_sel[1] = static_cast<uint32_t>(remaining - before);
        s_sel[2] = static_cast<uint32_t>(c);
      }
    }
    __syncthreads();
    prefix |= s_sel[0] << shift;
    pmask |= 0xFFu << shift;
    remaining = static_cast<int>(s_sel[1]);
    const bool exact = static_cast<int>(s_sel[2]) == remaining;
    __syncthreads();
    if (exact) break;
  }
  // take every key whose prefix class is above `prefix` and the first
  // `remaining` keys of the class itself (smallest indices first); compact in
  // index order.  A taken key's slot is the number of taken keys before it:
  // (keys above the class before it) + min(keys of the class before it,
  // remaining).  Each warp walks a contiguous segment of the row 32 keys at a
  // time, its lanes on consecutive keys (conflict-free shared-memory reads),
  // and counts with ballots; two walks (counts, then slots) around one scan of
  // the warp totals.  (A thread walking its own contiguous run of n / 512 keys
  // read shared memory with an n / 512-word stride between lanes: up to a
  // 16-way bank conflict on every access.)
  constexpr int NW = TK_THREADS / 32;
  const int seg = (n + NW - 1) / NW;
  const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  int c_above = 0, c_eq = 0;
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const bool v = i < w1;
    const uint32_t u = v ? (s_key[i] & pmask) : 0u;
    c_above += __popc(__ballot_sync(0xffffffffu, v && u > prefix));
    c_eq += __popc(__ballot_sync(0xffffffffu, v && u == prefix));
  }
  if (lane == 0) {
    s_warp[warp] = c_above;
    s_warp[NW + warp] = c_eq;
  }
  __syncthreads();
  int ab = 0, eb = 0, tot_above = 0, tot_eq = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const int x = s_warp[w], y = s_warp[NW + w];
    if (w < warp) {
      ab += x;
      eb += y;
    }
    tot_above += x;
    tot_eq += y;
  }
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const bool v = i < w1;
    const uint32_t u = v ? (s_key[i] & pmask) : 0u;
    const bool above = v && u > prefix, in_class = v && u == prefix;
    const unsigned ma = __ballot_sync(0xffffffffu, above), me = __ballot_sync(0xffffffffu, in_class);
    const int ra = ab + __popc(ma & lt), re = eb + __popc(me & lt);
    if (above || (in_class && re < remaining)) {
      const int pos = ra + min(re, remaining);
      irow[pos] = lo + i;
      srow[pos] = lrow[lo + i];
    }
    ab += __popc(ma);
    eb += __popc(me);
  }
  const int tot_sel = tot_above + min(tot_eq, remaining);
  for (int i = tot_sel + threadIdx.x; i < K; i += TK_THREADS) {
    irow[i] = -1;
    srow[i] = -INFINITY;
  }
  if (threadIdx.x == 0) length[t] = tot_sel;
}

// ---------------------------------------------------------------------------
// Indexer backward
// ---------------------------------------------------------------------------
constexpr int IB_HB = 64;                       // heads (M of Z)
constexpr int IB_NK = 64;                       // slots per chunk
constexpr int IB_D = 128;
constexpr int IB_Q_BYTES = IB_HB * IB_D * 2;    // 16 KB
constexpr int IB_K_BYTES = IB_NK * IB_D * 2;    // 16 KB
constexpr int IB_T_BYTES = IB_HB * IB_NK * 2;   // dZ tile, 8 KB
constexpr int IB_SMEM = IB_Q_BYTES + 2 * IB_K_BYTES + IB_T_BYTES + 1024;   // two key chunks
constexpr int IB_THREADS = 352;                 // 0..3 epilogue, 4..7 dK drain, 8..9 gather, 10 MMA
constexpr uint32_t IB_TMEM_COLS = 256;
constexpr uint32_t IB_COL_Z = 0, IB_COL_DQ = 64, IB_COL_PC0 = 128, IB_COL_PC1 = 192;

struct IbArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const float* w;
  const int32_t* idx;
  const float* grad;
  __nv_bfloat16* dq;
  float* dk_acc;
  float* dw;
  int T, H, K, use_relu;
  int32_t* err;
};

__device__ __forceinline__ uint32_t ib_off(int row, int ch, int rows) {
  return (ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ void red_add_v4(float* addr, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(x), "f"(y),
               "f"(z), "f"(w)
               : "memory");
}

__global__ void __launch_bounds__(IB_THREADS, 2) dsa_indexer_bwd_kernel(const IbArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + IB_Q_BYTES;                // two chunk buffers
  uint8_t* sdZ = sK + 2 * IB_K_BYTES;           // [head][slot] bf16, 128-byte rows
  __shared__ uint64_t bar_in, bar_k_full[2], bar_k_empty[2], bar_z_full, bar_z_free, bar_dz_full;
  __shared__ uint64_t bar_dz_free, bar_pc_full[2], bar_pc_free[2], bar_dq_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int s_row[8][IB_NK];               // key row of each slot (-1: none), by chunk mod 8
  __shared__ float s_g[2][IB_NK];               // slot gradients (0 for empty slots), by chunk mod 2
  __shared__ float s_w[IB_HB];
  __shared__ int s_red[IB_THREADS / 32];

  const int t = blockIdx.x;
  const int H = a.H;
  const int warp = warp_id(), lane = lane_id();
  AbortCtx ac{&abort_flag, a.err};

  int nchunks;
  {
    const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
    int last = -1;
    for (int s = threadIdx.x; s < a.K; s += IB_THREADS) {
      const int j = __ldg(irow + s);
      if (j >= 0 && j < a.T) last = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    if (lane == 0) s_red[warp] = last;
    if (threadIdx.x == 0) {
      abort_flag = 0;
      mbar_init(&bar_in, 64);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bar_k_full[b], 64);
        mbar_init(&bar_k_empty[b], 1);
      }
      mbar_init(&bar_z_full, 1);
      mbar_init(&bar_z_free, 128);
      mbar_init(&bar_dz_full, 128);
      mbar_init(&bar_dz_free, 1);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bar_pc_full[b], 1);
        mbar_init(&bar_pc_free[b], 128);
      }
      mbar_init(&bar_dq_done, 1);
      fence_mbar_init();
    }
    if (threadIdx.x < IB_HB) s_w[threadIdx.x] = threadIdx.x < H ? __ldg(a.w + static_cast<size_t>(t) * H + threadIdx.x) : 0.f;
    if (warp == 10) tmem_alloc(&tmem_base_sh, IB_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int m = -1;
    for (int w = 0; w < IB_THREADS / 32; ++w) m = max(m, s_red[w]);
    nchunks = (m + IB_NK) / IB_NK;
  }
  const uint32_t tmem = tmem_base_sh;

  if (warp == 8 || warp == 9) {
    // ---------------- gather producers ----------------
    const int pt = threadIdx.x - 256;            // 0..63
    const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
    const float* grow = a.grad + static_cast<size_t>(t) * a.K;
    if (nchunks > 0) {
      const __nv_bfloat16* qb = a.q + static_cast<size_t>(t) * H * IB_D;
      for (int id = pt; id < IB_HB * (IB_D / 8); id += 64) {
        const int r = id / (IB_D / 8), ch = id % (IB_D / 8);
        const bool v = r < H;
        cp_async16(smem_u32(sQ) + ib_off(r, ch, IB_HB),
                   v ? static_cast<const void*>(qb + r * IB_D + ch * 8) : static_cast<const void*>(a.q),
                   v ? 16u : 0u);
      }
      cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      // buffer b was last read by the MMAs of chunk c - 2
      if (!mbar_wait_w(&bar_k_empty[b], ((c >> 1) & 1) ^ 1, ac)) break;
      const int slot = c * IB_NK + pt;
      const int j = slot < a.K ? __ldg(irow + slot) : -1;
      const bool valid = j >= 0 && j < a.T;
      if (!valid && j != -1 && a.err) atomicOr(a.err, ATTN_DEVERR_INDEX_RANGE);
      const int jr = valid ? j : -1;
      s_row[c & 7][pt] = jr;
      s_g[c & 1][pt] = valid ? __ldg(grow + slot) : 0.f;
      const uint32_t base = smem_u32(sK + b * IB_K_BYTES);
      const int rw = pt & ~31;
#pragma unroll
      for (int kk = 0; kk < IB_D / 8; ++kk) {    // 32 rows x 16 chunks / 32 lanes
        const int e = 32 * kk + lane;
        const int rl = e / (IB_D / 8), ch = e - rl * (IB_D / 8);
        const int jj = __shfl_sync(0xffffffffu, jr, rl);
        cp_async16(base + ib_off(rw + rl, ch, IB_NK),
                   jj >= 0 ? static_cast<const void*>(a.k + static_cast<size_t>(jj) * IB_D + ch * 8)
                           : static_cast<const void*>(a.k),
                   jj >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      if (c == 0) mbar_arrive(&bar_in);
      mbar_arrive(&bar_k_full[b]);
    }
    cp_async_wait<0>();
  } else if (warp == 10) {
    // ---------------- MMA issuer ----------------
    if (nchunks > 0) {
      const uint32_t idZ = idesc_bf16(64, IB_NK, false, false);       // Z (heads x slots)
      const uint32_t idQ = idesc_bf16(128, IB_HB, true, false);       // dQ^T (dims x heads)
      const uint32_t idK = idesc_bf16(64, 64, true, true);            // dK pieces (slots x dims)
      const uint64_t dQk = desc_kmajor_base(smem_u32(sQ));
      const uint64_t ddZk = desc_kmajor_base(smem_u32(sdZ));
      const uint64_t ddZmn = desc_mnmajor_base(smem_u32(sdZ), IB_HB);
      bool ok = mbar_wait_w(&bar_in, 0, ac);
      int gp = 0;
      for (int c = 0; ok && c < nchunks; ++c) {
        const int b = c & 1;
        const uint64_t dKk = desc_kmajor_base(smem_u32(sK + b * IB_K_BYTES));
        const uint64_t dKmn = desc_mnmajor_base(smem_u32(sK + b * IB_K_BYTES), IB_NK);
        if (!mbar_wait_w(&bar_k_full[b], (c >> 1) & 1, ac)) { ok = false; break; }
        if (c > 0 && !mbar_wait_w(&bar_z_free, (c - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < IB_D / 16; ++kk)
          umma_ss_w(tmem + IB_COL_Z, desc_advance(dQk, kmajor_step_bytes(IB_HB, kk)),
                    desc_advance(dKk, kmajor_step_bytes(IB_NK, kk)), idZ, kk > 0 ? 1u : 0u);
        umma_commit_w(&bar_z_full);
        if (!mbar_wait_w(&bar_dz_full, c & 1, ac)) { ok = false; break; }
        tc_fence_after();
        // dQ^T(dims, heads) += K^T(dims, slots) dZ^T(slots, heads)
#pragma unroll
        for (int kk = 0; kk < IB_NK / 16; ++kk)
          umma_ss_w(tmem + IB_COL_DQ, desc_advance(dKmn, mnmajor_step_bytes(kk)),
                    desc_advance(ddZk, kmajor_step_bytes(IB_HB, kk)), idQ,
                    (c > 0 || kk > 0) ? 1u : 0u);
        umma_commit_w(&bar_k_empty[b]);          // the key rows of this chunk are no longer read
        // dK pieces: D(slots, dims 64p..) = dZ^T(slots, heads) Q_p(heads, dims)
        for (int p = 0; p < IB_D / 64; ++p, ++gp) {
          const int b = gp & 1, use = gp >> 1;
          if (!mbar_wait_w(&bar_pc_free[b], (use & 1) ^ 1, ac)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dQmn = desc_mnmajor_base(smem_u32(sQ + p * IB_HB * 128), IB_HB);
#pragma unroll
          for (int kk = 0; kk < IB_HB / 16; ++kk)
            umma_ss_w(tmem + (b ? IB_COL_PC1 : IB_COL_PC0), desc_advance(ddZmn, mnmajor_step_bytes(kk)),
                      desc_advance(dQmn, mnmajor_step_bytes(kk)), idK, kk > 0 ? 1u : 0u);
          umma_commit_w(&bar_pc_full[b]);
        }
        if (!ok) break;
        umma_commit_w(&bar_dz_free);             // the dZ tile of this chunk is read
      }
      if (ok) umma_commit_w(&bar_dq_done);
    }
  } else if (warp >= 4) {
    // ---------------- dK drain (warps 4..7) ----------------
    const int qq = warp - 4;
    const bool active = lane < 16;
    const int slot = 16 * qq + (lane & 15);      // slot row of the M = 64 piece
    const uint32_t lane_base = static_cast<uint32_t>(32 * qq) << 16;
    int gp = 0;
    bool ok = true;
    for (int c = 0; ok && c < nchunks; ++c) {
      for (int p = 0; p < IB_D / 64; ++p, ++gp) {
        const int b = gp & 1, use = gp >> 1;
        if (!mbar_wait(&bar_pc_full[b], use & 1, ac)) { ok = false; break; }
        tc_fence_after();
        uint32_t u[64];
        const uint32_t src = tmem + lane_base + (b ? IB_COL_PC1 : IB_COL_PC0);
        tmem_ld32_nowait(src, u);
        tmem_ld32_nowait(src + 32, u + 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar_pc_free[b]);
        const int j = active ? s_row[c & 7][slot] : -1;
        if (j >= 0) {
          float* dst = a.dk_acc + static_cast<size_t>(j) * IB_D + 64 * p;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            red_add_v4(dst + 4 * i, __uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                       __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
        }
      }
    }
  } else {
    // ---------------- epilogue: dZ, dw (warps 0..3) and dQ ----------------
    const int qq = warp;
    const bool active = lane < 16;
    const int row = 16 * qq + (lane & 15);       // head row held by this lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * qq) << 16;
    bool ok = nchunks == 0 || mbar_wait(&bar_in, 0, ac);
    const float wv = s_w[row];
    float dw = 0.f;
    for (int c = 0; ok && c < nchunks; ++c) {
      if (!mbar_wait(&bar_z_full, c & 1, ac)) { ok = false; break; }
      if (!mbar_wait(&bar_k_full[c & 1], (c >> 1) & 1, ac)) { ok = false; break; }   // slot gradients
      tc_fence_after();
      uint32_t uz[64];
      tmem_ld32_nowait(tmem + lane_base + IB_COL_Z, uz);
      tmem_ld32_nowait(tmem + lane_base + IB_COL_Z + 32, uz + 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_z_free);
      const float* g = s_g[c & 1];
      uint32_t pz[32];
#pragma unroll
      for (int cc = 0; cc < 64; cc += 2) {
        const float z0 = __uint_as_float(uz[cc]), z1 = __uint_as_float(uz[cc + 1]);
        const float g0 = g[cc], g1 = g[cc + 1];
        float a0, a1, d0, d1;
        if (a.use_relu) {
          a0 = fmaxf(z0, 0.f);
          a1 = fmaxf(z1, 0.f);
          d0 = z0 > 0.f ? g0 * wv : 0.f;
          d1 = z1 > 0.f ? g1 * wv : 0.f;
        } else {
          a0 = z0;
          a1 = z1;
          d0 = g0 * wv;
          d1 = g1 * wv;
        }
        dw = fmaf(g0, a0, dw);
        dw = fmaf(g1, a1, dw);
        pz[cc / 2] = pack_bf16(d0, d1);
      }
      // the dZ tile of chunk c - 1 must have been read
      if (c > 0) {
        if (!mbar_wait(&bar_dz_free, (c - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
      }
      if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t off = row * 128 + ((i ^ (row & 7)) << 4);
          *reinterpret_cast<uint4*>(sdZ + off) =
              make_uint4(pz[4 * i], pz[4 * i + 1], pz[4 * i + 2], pz[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_dz_full);
    }
    if (ok && active && row < H) a.dw[static_cast<size_t>(t) * H + row] = dw;
    // ---- dQ = (dQ^T)^T, bf16: lane = dim 32 qq + lane, columns = heads ----
    if (ok) {
      const bool have = nchunks > 0 && mbar_wait(&bar_dq_done, 0, ac);
      tc_fence_after();
      __nv_bfloat16* qbase = a.dq + static_cast<size_t>(t) * H * IB_D;
      const int d = 32 * qq + lane;
#pragma unroll
      for (int h0 = 0; h0 < IB_HB; h0 += 32) {
        uint32_t o[32];
        if (have) {
          tmem_ld32_nowait(tmem + lane_base + IB_COL_DQ + h0, o);
          tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int h = h0 + i;
          if (h < H)
            qbase[static_cast<size_t>(h) * IB_D + d] =
                __float2bfloat16_rn(have ? __uint_as_float(o[i]) : 0.f);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, IB_TMEM_COLS);
    tmem_relinquish();
  }
}

__global__ void __launch_bounds__(256) dsa_zero_f32_kernel(float4* p, size_t n4) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) dsa_cast_bf16_kernel(const float* acc, __nv_bfloat16* out,
                                                           size_t n8) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a0 = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 a1 = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a0.x, a0.y);
    o.y = pack_bf16(a0.z, a0.w);
    o.z = pack_bf16(a1.x, a1.y);
    o.w = pack_bf16(a1.z, a1.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

bool aligned(const void* p, unsigned m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; }

attn_status_t check(const dsa_indexer_problem_t* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->tokens < 0 || p->heads <= 0 || p->head_dim <= 0) return ATTN_ERR_INVALID_ARG;
  if (p->head_dim != IX_D || p->heads > IX_MAXH) return ATTN_ERR_UNSUPPORTED;
  if (p->cu_seqlens) {
    if (p->num_seqs <= 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned(p->cu_seqlens, 4)) return ATTN_ERR_ALIGNMENT;
  }
  return ATTN_OK;
}

IxArgs make_ix(const dsa_indexer_problem_t* p) {
  IxArgs a{};
  a.cu = p->cu_seqlens;
  a.T = p->tokens;
  a.H = p->heads;
  a.nseq = p->cu_seqlens ? p->num_seqs : 0;
  a.ld = p->logits_ld;
  a.use_relu = p->use_relu ? 1 : 0;
  a.err = p->error_word;
  return a;
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t dsa_indexer_fwd(const dsa_indexer_problem_t* p, const void* q,
                                         const void* k, const float* w, float* logits,
                                         attn_stream_t stream) {
  attn_status_t s = check(p);
  if (s != ATTN_OK) return s;
  if (p->logits_ld < p->tokens || p->logits_ld % 4 != 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->tokens) * p->logits_ld >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (p->tokens == 0) return ATTN_OK;
  if (!q || !k || !w || !logits) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 16) || !aligned(logits, 16))
    return ATTN_ERR_ALIGNMENT;
  CUtensorMap tmQ, tmK;
  if (!make_bf16_tile_map(&tmQ, q, 1, p->tokens, p->heads, IX_D, IX_T) ||
      !make_bf16_tile_map(&tmK, k, 1, p->tokens, 1, IX_D, IX_T))
    return ATTN_ERR_CUDA;
  IxArgs a = make_ix(p);
  a.w = w;
  a.logits = logits;
  const int nt = (p->tokens + IX_T - 1) / IX_T;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaFuncSetAttribute(dsa_indexer_logits_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, IX_SMEM);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  dsa_indexer_logits_kernel<<<dim3(nt, nt), IX_THREADS, IX_SMEM, st>>>(tmQ, tmK, a);
  return cuda_status(cudaGetLastError());
}

extern "C" attn_status_t dsa_topk(const dsa_indexer_problem_t* p, const float* logits,
                                  int32_t* idx, int32_t* length, float* scores,
                                  attn_stream_t stream) {
  attn_status_t s = check(p);
  if (s != ATTN_OK) return s;
  if (p->topk <= 0 || p->topk > TK_MAXN) return ATTN_ERR_UNSUPPORTED;
  if (p->tokens > TK_MAXN) return ATTN_ERR_UNSUPPORTED;
  if (p->logits_ld < p->tokens || p->logits_ld % 4 != 0) return ATTN_ERR_INVALID_ARG;
  if (p->tokens == 0) return ATTN_OK;
  if (!logits || !idx || !length || !scores) return ATTN_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || !aligned(idx, 16) || !aligned(length, 16) || !aligned(scores, 16))
    return ATTN_ERR_ALIGNMENT;
  IxArgs a = make_ix(p);
  a.logits = const_cast<float*>(logits);
  dsa_topk_kernel<<<p->tokens, TK_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      a, p->topk, idx, length, scores);
  return cuda_status(cudaGetLastError());
}

extern "C" size_t dsa_indexer_bwd_workspace_size(const dsa_indexer_problem_t* p) {
  if (check(p) != ATTN_OK) return 0;
  return static_cast<size_t>(p->tokens) * IB_D * sizeof(float);
}

extern "C" attn_status_t dsa_indexer_bwd(const dsa_indexer_problem_t* p, const void* q,
                                         const void* k, const float* w, const int32_t* idx,
                                         const float* grad, void* dq, void* dk, float* dw,
                                         void* workspace, size_t workspace_bytes,
                                         attn_stream_t stream) {
  attn_status_t s = check(p);
  if (s != ATTN_OK) return s;
  if (p->topk <= 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->tokens) * p->topk >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (p->tokens == 0) return ATTN_OK;
  if (!q || !k || !w || !idx || !grad || !dq || !dk || !dw) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(w, 16) || !aligned(idx, 16) ||
      !aligned(grad, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dw, 16))
    return ATTN_ERR_ALIGNMENT;
  const size_t need = dsa_indexer_bwd_workspace_size(p);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return ATTN_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* acc = static_cast<float*>(workspace);
  const size_t n4 = static_cast<size_t>(p->tokens) * IB_D / 4;
  dsa_zero_f32_kernel<<<resident_grid(dsa_zero_f32_kernel, n4, 256), 256, 0, st>>>(
      reinterpret_cast<float4*>(acc), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  IbArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.w = w;
  a.idx = idx;
  a.grad = grad;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk_acc = acc;
  a.dw = dw;
  a.T = p->tokens;
  a.H = p->heads;
  a.K = p->topk;
  a.use_relu = p->use_relu ? 1 : 0;
  a.err = p->error_word;
  if ((e = cudaFuncSetAttribute(dsa_indexer_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                IB_SMEM)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  dsa_indexer_bwd_kernel<<<p->tokens, IB_THREADS, IB_SMEM, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return ATTN_ERR_CUDA;
  const size_t n8 = static_cast<size_t>(p->tokens) * IB_D / 8;
  dsa_cast_bf16_kernel<<<resident_grid(dsa_cast_bf16_kernel, n8, 256), 256, 0, st>>>(
      acc, static_cast<__nv_bfloat16*>(dk), n8);
  return cuda_status(cudaGetLastError());
}
