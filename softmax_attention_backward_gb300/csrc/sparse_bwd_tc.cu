// Top-k sparse attention backward on tcgen05 (SparseMLA style, "[2/2] Add
// TileLang fused DSA kernels support with THD and CP", Megatron-LM #5049:
// sparse MLA backward with preprocess/postprocess; one shared KV head, dim
// 576 = 512 latent + 64 rope, v_channels 512, -1 for empty top-k slots).
//
// Work item = one token t and a block of 64 query heads; CTA b takes the items
// b, b + gridDim.x, b + 2 gridDim.x, ... in that order.  Q [64 x 576], dO
// [64 x 512], LSE and Delta of the item load once; the token's key rows are
// gathered 64 slots at a time (16-byte cp.async, SW128 K-major layout).  Per
// chunk of slots s (KV rows K_s, V_s = the first 512 dims of K_s):
//   S    = Q K^T      dP = dO V^T          (M = 64 heads, N = 64 slots, TMEM)
//   P    = exp(S c - LSE),  dS = P o (dP - Delta) c        (softmax warps)
//   dQ^T += K^T dS^T  (value dims on TMEM lanes: four M = 128 tiles for dims
//                      0..511 and one M = 64 tile for dims 512..575, 64 heads)
//   dKV[s]^T += Q^T dS + [dO | 0]^T P   in five pieces of value dims (four
//                      M = 128 pieces for dims 0..511, one M = 64 piece for
//                      512..575; N = 64 slots), each drained from TMEM into
//                      an fp32 dKV accumulator while the next piece is
//                      computed (two piece buffers): a lane holds one dim of
//                      every slot; groups of four lanes transpose 4 x 4
//                      blocks by shuffles and add 16-byte vectors, eight
//                      lanes to 128 bytes of one key row
// P and dS go through shared memory as bf16 [head][slot] tiles, which serve
// as the K-major B operand of dQ^T and the MN-major B operand of the dKV
// pieces.  The scale c is folded into dS, so dQ and dKV need none later.
// An M = 64 accumulator keeps row r in TMEM lane 32 (r / 16) + r % 16.
//
// dKV accumulators.  Shared mode (a.slabs == 0, one item per CTA): every CTA
// adds into one [T, 576] accumulator, so the order of the adds into a key row
// follows the timing.  Slab mode (a.slabs == gridDim.x): CTA b adds only into
// its own accumulator slab b.  A token names a key row at most once, so an
// item adds at most once into each slab address; between items the drain
// warps fence and meet at a named barrier, so a slab address receives its
// adds in the CTA's fixed item order, and the slabs are summed later in slab
// order: the result is bitwise reproducible.  dQ is the same in both modes.
//
// Warp roles (352 threads): 0..3 softmax and dQ epilogue, 4..7 dKV drain,
// 8..9 gather producers, 10 MMA issuer.  The chunk counts per token come from
// the preprocess.  Every wait is a bounded mbarrier wait.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

namespace {

constexpr int SB_HB = 64;                      // heads per item
constexpr int SB_NK = kSparseChunk;            // key slots per chunk
constexpr int SB_DQK = 576, SB_DV = 512;
constexpr int SB_Q_BYTES = SB_HB * SB_DQK * 2;
constexpr int SB_DO_BYTES = SB_HB * SB_DV * 2;
constexpr int SB_KV_BYTES = SB_NK * SB_DQK * 2;
constexpr int SB_T_BYTES = SB_HB * SB_NK * 2;  // P or dS tile
constexpr int SB_SMEM = SB_Q_BYTES + SB_DO_BYTES + SB_KV_BYTES + 2 * SB_T_BYTES + 1024;
constexpr int SB_THREADS = 352;
constexpr int SB_PRODUCERS = 64;               // warps 8..9
static_assert(SB_PRODUCERS == SB_NK, "one producer lane holds each slot's index");
constexpr int SB_PIECES = 5;                   // dKV^T pieces: dims 128 p.. (p < 4), 512..575
constexpr uint32_t SB_TMEM_COLS = 512;
constexpr uint32_t SB_COL_S = 0, SB_COL_DP = 64;
constexpr uint32_t SB_COL_DQ = 128;            // five dQ^T tiles of 64 columns
constexpr uint32_t SB_COL_PC = 448;            // dKV piece buffer 0 (buffer 1 = the dP columns)
constexpr uint32_t SB_BAR_DRAIN = 1;           // named barrier of the four drain warps

__device__ __forceinline__ uint32_t sb_off(int row, int ch, int rows) {
  return (ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

}  // namespace

__global__ void __launch_bounds__(SB_THREADS, 1) sparse_bwd_tc_kernel(const SparseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + SB_Q_BYTES;
  uint8_t* sKV = sdO + SB_DO_BYTES;
  uint8_t* sP = sKV + SB_KV_BYTES;               // [head][slot] bf16, 128-byte rows
  uint8_t* sdS = sP + SB_T_BYTES;

  __shared__ uint64_t bar_in, bar_kv_full, bar_kv_empty, bar_s_full, bar_s_free, bar_ds_full;
  __shared__ uint64_t bar_pds_free, bar_pc_full[2], bar_pc_free[2], bar_dq_done, bar_dq_free;
  __shared__ uint64_t bar_qdo_free;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  // KV row of each slot (-1: none) by chunk mod 4: the drain of a chunk's
  // last pieces may still read its rows while the producer fills chunk + 2
  __shared__ int s_row[4][SB_NK];
  __shared__ uint32_t s_valid[2][2];
  __shared__ float s_lse2[SB_HB];                // LSE * log2(e)
  __shared__ float s_delta[SB_HB];

  const int nhb = (a.H + SB_HB - 1) / SB_HB;
  const int n_items = a.T * nhb;
  const int warp = warp_id(), lane = lane_id();
  AbortCtx ac{&abort_flag, a.err};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_in, SB_PRODUCERS);
    mbar_init(&bar_kv_full, SB_PRODUCERS);
    mbar_init(&bar_kv_empty, 1);
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_s_free, 128);
    mbar_init(&bar_ds_full, 128);
    mbar_init(&bar_pds_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_pc_full[b], 1);
      mbar_init(&bar_pc_free[b], 128);
    }
    mbar_init(&bar_dq_done, 1);
    mbar_init(&bar_dq_free, 128);
    mbar_init(&bar_qdo_free, 1);
    fence_mbar_init();
  }
  if (warp == 10) tmem_alloc(&tmem_base_sh, SB_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // Every role walks the same item sequence and skips the same empty items;
  // g counts chunks and ni non-empty items over the whole sequence, which sets
  // the barrier phases.
  if (warp == 8 || warp == 9) {
    // ---------------- producers: each item's inputs, then its chunks ----------------
    const int pt = threadIdx.x - 256;              // 0..63
    int g = 0, ni = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int t = item / nhb, hb = (item - t * nhb) * SB_HB;
      const int nh = min(SB_HB, a.H - hb);
      const int nchunks = __ldg(a.nch + t);
      if (nchunks == 0) continue;
      // Q, dO, LSE and Delta of the previous item: read until its last MMAs
      if (ni > 0 && !mbar_wait_w(&bar_qdo_free, (ni - 1) & 1, ac)) { ok = false; break; }
      const int32_t* irow = a.idx + static_cast<size_t>(t) * a.K;
      const __nv_bfloat16* qb = a.q + (static_cast<size_t>(t) * a.H + hb) * SB_DQK;
      const __nv_bfloat16* ob = a.dout + (static_cast<size_t>(t) * a.H + hb) * SB_DV;
      for (int id = pt; id < SB_HB * (SB_DQK / 8); id += SB_PRODUCERS) {
        const int r = id / (SB_DQK / 8), ch = id % (SB_DQK / 8);
        const bool v = r < nh;
        cp_async16(smem_u32(sQ) + sb_off(r, ch, SB_HB),
                   v ? static_cast<const void*>(qb + r * SB_DQK + ch * 8) : static_cast<const void*>(a.q),
                   v ? 16u : 0u);
      }
      for (int id = pt; id < SB_HB * (SB_DV / 8); id += SB_PRODUCERS) {
        const int r = id / (SB_DV / 8), ch = id % (SB_DV / 8);
        const bool v = r < nh;
        cp_async16(smem_u32(sdO) + sb_off(r, ch, SB_HB),
                   v ? static_cast<const void*>(ob + r * SB_DV + ch * 8) : static_cast<const void*>(a.dout),
                   v ? 16u : 0u);
      }
      cp_async_commit();
      // LSE (log2 domain) and Delta of the item's heads; rows past H give P = 0
      const size_t li = static_cast<size_t>(t) * a.H + hb + pt;
      s_lse2[pt] = pt < nh ? __ldg(a.lse_in + li) * kLog2e : INFINITY;
      s_delta[pt] = pt < nh ? __ldg(a.delta + li) : 0.f;
      for (int c = 0; c < nchunks; ++c, ++g) {
        // the single chunk buffer was last read by dQ^T of the previous chunk
        // (warp-uniform answer: the lanes exchange indices below)
        if (!mbar_wait_w(&bar_kv_empty, (g & 1) ^ 1, ac)) { ok = false; break; }
        const int cb = g & 1;
        const int slot = c * SB_NK + pt;
        const int j = (slot < a.K) ? __ldg(irow + slot) : -1;
        const bool valid = j >= 0 && j < a.T;
        if (!valid && j != -1 && a.err) atomicOr(a.err, ATTN_DEVERR_INDEX_RANGE);
        const int jr = valid ? j : -1;
        s_row[g & 3][pt] = jr;
        const uint32_t m32 = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) s_valid[cb][pt >> 5] = m32;
        // each producer warp gathers the 32 rows whose indices its lanes hold, in
        // (row, 16-byte column) order, taking a row's index by a shuffle rather
        // than a load per copy; the chunk's gather is on the critical path (one
        // buffer), and it runs faster the more copies are issued back to back,
        // so the 72 copies of a lane are fully unrolled
        const uint32_t base = smem_u32(sKV);
        const int rw = pt & ~31;
#pragma unroll
        for (int k = 0; k < SB_DQK / 8; ++k) {   // 32 rows x 72 columns / 32 lanes
          const int e = 32 * k + lane;
          const int rl = e / (SB_DQK / 8), ch = e - rl * (SB_DQK / 8);
          const int jj = __shfl_sync(0xffffffffu, jr, rl);
          cp_async16(base + sb_off(rw + rl, ch, SB_NK),
                     (jj >= 0) ? static_cast<const void*>(a.kv + static_cast<size_t>(jj) * SB_DQK + ch * 8)
                               : static_cast<const void*>(a.kv),
                     (jj >= 0) ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        if (c == 0) mbar_arrive(&bar_in);
        mbar_arrive(&bar_kv_full);
      }
      ++ni;
    }
    cp_async_wait<0>();
  } else if (warp == 10) {
    // ---------------- MMA issuer (warp-uniform: one elected lane issues) ----------------
    const uint32_t idS = idesc_bf16(64, SB_NK, false, false);        // S, dP
    const uint32_t idQ128 = idesc_bf16(128, SB_HB, true, false);     // dQ^T tiles
    const uint32_t idQ64 = idesc_bf16(64, SB_HB, true, false);       // dQ^T dims 512..575
    const uint32_t idKV128 = idesc_bf16(128, SB_NK, true, true);     // dKV^T pieces 0..3
    const uint32_t idKV64 = idesc_bf16(64, SB_NK, true, true);       // dKV^T piece 4
    const uint64_t dQk = desc_kmajor_base(smem_u32(sQ));
    const uint64_t ddOk = desc_kmajor_base(smem_u32(sdO));
    const uint64_t dKk = desc_kmajor_base(smem_u32(sKV));
    const uint64_t ddSk = desc_kmajor_base(smem_u32(sdS));
    const uint64_t dPmn = desc_mnmajor_base(smem_u32(sP), SB_HB);
    const uint64_t ddSmn = desc_mnmajor_base(smem_u32(sdS), SB_HB);
    int g = 0, ni = 0;
    int gp = 0;                                  // dKV pieces issued so far
    int n1 = 0;                                  // pieces issued into buffer 1 (the dP columns)
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int nchunks = __ldg(a.nch + item / nhb);
      if (nchunks == 0) continue;
      if (!mbar_wait_w(&bar_in, ni & 1, ac)) { ok = false; break; }
      for (int c = 0; c < nchunks; ++c, ++g) {
        if (!mbar_wait_w(&bar_kv_full, g & 1, ac)) { ok = false; break; }
        // S and dP columns: read by the softmax of the previous chunk, and the
        // last dKV piece that used the dP columns drained
        if (g > 0 && !mbar_wait_w(&bar_s_free, (g - 1) & 1, ac)) { ok = false; break; }
        if (n1 > 0 && !mbar_wait_w(&bar_pc_free[1], (n1 - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 4
        for (int kk = 0; kk < SB_DQK / 16; ++kk)
          umma_ss_w(tmem + SB_COL_S, desc_advance(dQk, kmajor_step_bytes(SB_HB, kk)),
                    desc_advance(dKk, kmajor_step_bytes(SB_NK, kk)), idS, kk > 0);
#pragma unroll 4
        for (int kk = 0; kk < SB_DV / 16; ++kk)
          umma_ss_w(tmem + SB_COL_DP, desc_advance(ddOk, kmajor_step_bytes(SB_HB, kk)),
                    desc_advance(dKk, kmajor_step_bytes(SB_NK, kk)), idS, kk > 0);
        umma_commit_w(&bar_s_full);
        if (!mbar_wait_w(&bar_ds_full, g & 1, ac)) { ok = false; break; }
        // the dQ^T columns of the previous item: read out by its epilogue
        if (c == 0 && ni > 0 && !mbar_wait_w(&bar_dq_free, (ni - 1) & 1, ac)) { ok = false; break; }
        tc_fence_after();
        // dQ^T(dims, heads) += K^T(dims, slots) dS^T(slots, heads)
#pragma unroll
        for (int m = 0; m < 5; ++m) {
          const uint64_t dKmn = desc_mnmajor_base(smem_u32(sKV + 2 * m * SB_NK * 128), SB_NK);
#pragma unroll
          for (int kk = 0; kk < SB_NK / 16; ++kk)
            umma_ss_w(tmem + SB_COL_DQ + 64 * m, desc_advance(dKmn, mnmajor_step_bytes(kk)),
                      desc_advance(ddSk, kmajor_step_bytes(SB_HB, kk)), m < 4 ? idQ128 : idQ64,
                      (c > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_w(&bar_kv_empty);                // K and V of this chunk are no longer read
        // dKV^T pieces: D(dims 128p.., slots) = Q_p^T dS + dO_p^T P
        for (int p = 0; p < SB_PIECES; ++p, ++gp) {
          const int b = gp & 1, use = gp >> 1;
          if (!mbar_wait_w(&bar_pc_free[b], (use & 1) ^ 1, ac)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dst = tmem + (b ? SB_COL_DP : SB_COL_PC);
          const uint64_t dQmn = desc_mnmajor_base(smem_u32(sQ + 2 * p * SB_HB * 128), SB_HB);
#pragma unroll
          for (int kk = 0; kk < SB_HB / 16; ++kk)
            umma_ss_w(dst, desc_advance(dQmn, mnmajor_step_bytes(kk)),
                      desc_advance(ddSmn, mnmajor_step_bytes(kk)), p < 4 ? idKV128 : idKV64, kk > 0);
          if (p < 4) {
            const uint64_t ddOmn = desc_mnmajor_base(smem_u32(sdO + 2 * p * SB_HB * 128), SB_HB);
#pragma unroll
            for (int kk = 0; kk < SB_HB / 16; ++kk)
              umma_ss_w(dst, desc_advance(ddOmn, mnmajor_step_bytes(kk)),
                        desc_advance(dPmn, mnmajor_step_bytes(kk)), idKV128, 1u);
          }
          umma_commit_w(&bar_pc_full[b]);
          if (b == 1) ++n1;
        }
        if (!ok) break;
        umma_commit_w(&bar_pds_free);                // P and dS tiles of this chunk are read
      }
      if (!ok) break;
      umma_commit_w(&bar_qdo_free);                  // the item's Q and dO are no longer read
      umma_commit_w(&bar_dq_done);
      ++ni;
    }
  } else if (warp >= 4) {
    // ---------------- dKV drain (warps 4..7) ----------------
    // warp q reads TMEM lanes 32 q..32 q + 31: dims 128 p + 32 q + lane of
    // pieces 0..3; of the M = 64 piece 4, lanes 0..15 hold dims 512 + 16 q + lane
    const int q = warp - 4;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float* const acc =
        a.dkv_acc + (a.slabs > 0 ? static_cast<size_t>(blockIdx.x) * a.T * SB_DQK : size_t(0));
    int g = 0, gp = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const int nchunks = __ldg(a.nch + item / nhb);
      if (nchunks == 0) continue;
      for (int c = 0; ok && c < nchunks; ++c, ++g) {
        int j0 = -1, j1 = -1;   // slot rows of the chunk, shuffled to the warp slot by slot
        for (int p = 0; p < SB_PIECES; ++p, ++gp) {
          const int b = gp & 1, use = gp >> 1;
          if (!mbar_wait_w(&bar_pc_full[b], use & 1, ac)) { ok = false; break; }
          tc_fence_after();
          uint32_t u[64];
          const uint32_t src = tmem + lane_base + (b ? SB_COL_DP : SB_COL_PC);
          tmem_ld32_nowait(src, u);
          tmem_ld32_nowait(src + 32, u + 32);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&bar_pc_free[b]);
          if (p == 0) {   // written before the chunk's first piece was issued
            j0 = s_row[g & 3][lane];
            j1 = s_row[g & 3][32 + lane];
          }
          const bool lane_ok = p < 4 || lane < 16;
          const int d = p < 4 ? 128 * p + 32 * q + lane : 512 + 16 * q + (lane & 15);
          // four lanes (dims d0..d0 + 3) transpose their 4 x 4 block of four
          // slots by two butterfly exchanges, so that lane r then holds dims
          // d0..d0 + 3 of slot s0 + r: one 16-byte add per lane, eight lanes
          // covering 128 bytes of the same key row
          const int r = lane & 3;
          const bool hi = (r & 2) != 0, od = (r & 1) != 0;
          const int d0 = d - r;
#pragma unroll
          for (int s0 = 0; s0 < SB_NK; s0 += 4) {
            float v0 = __uint_as_float(u[s0]), v1 = __uint_as_float(u[s0 + 1]);
            float v2 = __uint_as_float(u[s0 + 2]), v3 = __uint_as_float(u[s0 + 3]);
            float x0 = __shfl_xor_sync(0xffffffffu, hi ? v0 : v2, 2);
            float x1 = __shfl_xor_sync(0xffffffffu, hi ? v1 : v3, 2);
            if (hi) { v0 = x0; v1 = x1; } else { v2 = x0; v3 = x1; }
            x0 = __shfl_xor_sync(0xffffffffu, od ? v0 : v1, 1);
            x1 = __shfl_xor_sync(0xffffffffu, od ? v2 : v3, 1);
            if (od) { v0 = x0; v2 = x1; } else { v1 = x0; v3 = x1; }
            const int j = __shfl_sync(0xffffffffu, s0 < 32 ? j0 : j1, (s0 & 31) + r);
            if (j >= 0 && lane_ok) red_add_v4(acc + static_cast<size_t>(j) * SB_DQK + d0, v0, v1, v2, v3);
          }
        }
      }
      if (a.slabs > 0) {
        // this item's adds into the slab are performed before any add of the
        // next item; the four warps leave together, on one common answer
        __threadfence();
        ok = named_bar_and(SB_BAR_DRAIN, 128, ok && !*reinterpret_cast<volatile int*>(&abort_flag));
      }
      if (!ok) break;
    }
  } else {
    // ---------------- softmax (P, dS) and dQ epilogue (warps 0..3) ----------------
    const int q = warp;
    const bool active = lane < 16;
    const int row = 16 * q + (lane & 15);          // head row held by this lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const float sl2 = a.scale_log2, sc = a.scale;
    int g = 0, ni = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int t = item / nhb, hb = (item - t * nhb) * SB_HB;
      const int nh = min(SB_HB, a.H - hb);
      const int nchunks = __ldg(a.nch + t);
      bool have = false;
      if (nchunks > 0) {
        if (!mbar_wait_w(&bar_in, ni & 1, ac)) { ok = false; break; }
        const float lse2 = s_lse2[row], dlt = s_delta[row];
        for (int c = 0; c < nchunks; ++c, ++g) {
          if (!mbar_wait_w(&bar_s_full, g & 1, ac)) { ok = false; break; }
          if (!mbar_wait_w(&bar_kv_full, g & 1, ac)) { ok = false; break; }   // valid mask of the chunk
          tc_fence_after();
          uint32_t pp[32], pd[32];
          const unsigned long long vm = static_cast<unsigned long long>(s_valid[g & 1][0]) |
                                        (static_cast<unsigned long long>(s_valid[g & 1][1]) << 32);
          // S and dP in two 32-column halves: with all 128 values live at once
          // the role spilled (c5 backward 13.59 ms against 13.39 this way)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t us[32], ud[32];
            tmem_ld32_nowait(tmem + lane_base + SB_COL_S + 32 * hf, us);
            tmem_ld32_nowait(tmem + lane_base + SB_COL_DP + 32 * hf, ud);
            tmem_wait_ld();
            if (hf == 1) {
              tc_fence_before();
              mbar_arrive(&bar_s_free);
            }
#pragma unroll
            for (int cc = 0; cc < 32; cc += 2) {
              const int col = 32 * hf + cc;
              float p0 = ex2(fmaf(__uint_as_float(us[cc]), sl2, -lse2));
              float p1 = ex2(fmaf(__uint_as_float(us[cc + 1]), sl2, -lse2));
              if (!((vm >> col) & 1ull)) p0 = 0.f;
              if (!((vm >> (col + 1)) & 1ull)) p1 = 0.f;
              const float d0 = p0 * (__uint_as_float(ud[cc]) - dlt) * sc;
              const float d1 = p1 * (__uint_as_float(ud[cc + 1]) - dlt) * sc;
              pp[col / 2] = pack_bf16(p0, p1);
              pd[col / 2] = pack_bf16(d0, d1);
            }
          }
          // the P / dS tiles of the previous chunk must have been read by its dKV pieces
          if (g > 0) {
            if (!mbar_wait_w(&bar_pds_free, (g - 1) & 1, ac)) { ok = false; break; }
            tc_fence_after();
          }
          if (active) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t off = row * 128 + ((i ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(sP + off) = make_uint4(pp[4 * i], pp[4 * i + 1], pp[4 * i + 2], pp[4 * i + 3]);
              *reinterpret_cast<uint4*>(sdS + off) = make_uint4(pd[4 * i], pd[4 * i + 1], pd[4 * i + 2], pd[4 * i + 3]);
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&bar_ds_full);
        }
        if (!ok) break;
        if (!mbar_wait_w(&bar_dq_done, ni & 1, ac)) { ok = false; break; }
        tc_fence_after();
        have = true;
      }
      // ---- dQ = (dQ^T)^T (the scale is in dS), bf16; zeros for a token without slots ----
      __nv_bfloat16* qbase = a.dq + (static_cast<size_t>(t) * a.H + hb) * SB_DQK;
#pragma unroll 1
      for (int m = 0; m < 5; ++m) {
        // tiles 0..3: lane = dim 128 m + 32 q + lane; tile 4 (M = 64): lanes
        // 0..15 of each quarter hold dims 512 + 16 q + lane
        const bool lane_ok = m < 4 || active;
        const int d = m < 4 ? 128 * m + 32 * q + lane : 512 + 16 * q + (lane & 15);
#pragma unroll
        for (int h0 = 0; h0 < SB_HB; h0 += 32) {
          uint32_t o[32];
          if (have) {
            tmem_ld32_nowait(tmem + lane_base + SB_COL_DQ + 64 * m + h0, o);
            tmem_wait_ld();
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int h = h0 + i;
            if (lane_ok && h < nh)
              qbase[static_cast<size_t>(h) * SB_DQK + d] =
                  __float2bfloat16_rn(have ? __uint_as_float(o[i]) : 0.f);
          }
        }
      }
      if (have) {
        tc_fence_before();
        mbar_arrive(&bar_dq_free);
        ++ni;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, SB_TMEM_COLS);
    tmem_relinquish();
  }
}

cudaError_t launch_sparse_bwd_main(const SparseArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(sparse_bwd_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SB_SMEM);
  if (e != cudaSuccess) return e;
  const int items = a.T * ((a.H + SB_HB - 1) / SB_HB);
  const int grid = a.slabs > 0 ? a.slabs : items;
  if (grid <= 0) return cudaSuccess;
  sparse_bwd_tc_kernel<<<grid, SB_THREADS, SB_SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
