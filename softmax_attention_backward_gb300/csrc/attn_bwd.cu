// Dense / GQA / THD attention backward (the `flash_bwd` stage of "[Example]
// Introduce split+sum template, and optimize atomic_add performance for bwd
// examples", tile-ai/tilelang #940: atomic and split variants).
//
// KV-tile-major: one CTA owns a 128-row K/V tile of one kv head and walks the
// query tiles of every query head of its GQA group, so dK and dV stay in TMEM
// for the whole CTA and are stored once (the group reduction of the #940 GQA
// backward, where dK is indexed by head // groups, happens on chip, without
// atomics).  Per query tile i of head h (KV rows j, query rows q):
//   S^T  = K Q_i^T            (TMEM)   P^T  = exp2(S^T * c - LSE_q * log2 e)
//   dP^T = V dO_i^T           (TMEM)   dS^T = P^T o (dP^T - Delta_q)
//   dV  += P^T dO_i           (TMEM)   dK  += dS^T Q_i           (TMEM)
//   dQ_i  = dS K  (D = 64, 128-row query tiles)  or
//   dQ_i^T = K^T dS^T (D = 128, 64-row query tiles), streamed out of TMEM and
//   either added with fp32 atomics into one accumulator (ATOMIC) or stored into
//   the partial slab of this KV tile (SPLIT, summed in order later).
// Roles: warp 8 TMA, warp 9 MMA issue, warps 0..3 P/dS (one KV row per
// thread), warps 4..7 dQ drain.  The scale factor of dK is applied in the
// epilogue and that of dQ in the finalize pass.
#include <cuda_runtime.h>

#include "launch.h"

namespace attn {

template <int D>
struct BwdCfg {
  static constexpr int BN = 128;                      // KV rows per CTA
  static constexpr int BM = (D == 64) ? 128 : 64;     // query rows per step
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QT_BYTES = BM * D * 2;
  static constexpr int PT_BYTES = BN * BM * 2;
  static constexpr int NST = 2;                       // Q/dO stages
  static constexpr int SMEM = 2 * KV_BYTES + 2 * NST * QT_BYTES + 2 * PT_BYTES + 1024;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BM;
  static constexpr uint32_t COL_DV = 2 * BM;
  static constexpr uint32_t COL_DK = 2 * BM + D;
  static constexpr uint32_t COL_DQ = 2 * BM + 2 * D;  // two 64-column buffers
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void red_add(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM, BN = C::BN;
  constexpr int PANELS = D / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::KV_BYTES;
  uint8_t* sQ = sV + C::KV_BYTES;                 // NST stages
  uint8_t* sdO = sQ + C::NST * C::QT_BYTES;       // NST stages
  uint8_t* sPt = sdO + C::NST * C::QT_BYTES;
  uint8_t* sdS = sPt + C::PT_BYTES;

  __shared__ uint64_t bar_kv, bar_qfull[C::NST], bar_qempty[C::NST];
  __shared__ uint64_t bar_s, bar_dp, bar_p, bar_ds, bar_pt_empty, bar_ds_empty, bar_done;
  __shared__ uint64_t bar_dq_full[2], bar_dq_empty[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float s_lse[2][BM], s_delta[2][BM];

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
      mbar_init(&bar_qempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_ds, 128);
    mbar_init(&bar_pt_empty, 1);
    mbar_init(&bar_ds_empty, 1);
    mbar_init(&bar_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_dq_full[b], 1);
      mbar_init(&bar_dq_empty[b], 128);
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
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane_id() == 0) {
      const uint32_t idSD = idesc_bf16(128, BM, false, false);   // S^T, dP^T
      const uint32_t idKV = idesc_bf16(128, D, false, true);     // dV, dK
      const uint32_t idQ = idesc_bf16(128, 64, true, true);      // dQ or dQ^T
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ),
                     adO = smem_u32(sdO), aPt = smem_u32(sPt), adS = smem_u32(sdS);
      auto issue_s = [&](int it) {
        const uint32_t q = aQ + (it % C::NST) * C::QT_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tmem + C::COL_S, desc_kmajor(aK, BN, k), desc_kmajor(q, BM, k), idSD, k > 0);
        umma_commit(&bar_s);
      };
      auto issue_dp = [&](int it) {
        const uint32_t o = adO + (it % C::NST) * C::QT_BYTES;
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tmem + C::COL_DP, desc_kmajor(aV, BN, k), desc_kmajor(o, BM, k), idSD, k > 0);
        umma_commit(&bar_dp);
      };
      bool ok = mbar_wait(&bar_kv, 0, ac) && mbar_wait(&bar_qfull[0], 0, ac);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % C::NST;
        const uint32_t q = aQ + st * C::QT_BYTES, o = adO + st * C::QT_BYTES;
        // dV += P^T dO_i
        if (!mbar_wait(&bar_p, it & 1, ac)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          umma_ss(tmem + C::COL_DV, desc_kmajor(aPt, BN, k), desc_mnmajor(o, BM, k), idKV,
                  (it > 0 || k > 0) ? 1u : 0u);
        umma_commit(&bar_pt_empty);
        // next S^T as soon as its inputs are in
        if (it + 1 < n_it) {
          if (!mbar_wait(&bar_qfull[(it + 1) % C::NST], ((it + 1) / C::NST) & 1, ac)) break;
          tc_fence_after();
          issue_s(it + 1);
        }
        // dK += dS^T Q_i ; dQ
        if (!mbar_wait(&bar_ds, it & 1, ac)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BM / 16; ++k)
          umma_ss(tmem + C::COL_DK, desc_kmajor(adS, BN, k), desc_mnmajor(q, BM, k), idKV,
                  (it > 0 || k > 0) ? 1u : 0u);
        const int qb = it & 1, qu = it >> 1;
        if (!mbar_wait(&bar_dq_empty[qb], (qu & 1) ^ 1, ac)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          if (D == 64)   // dQ[q, d] = dS[q, kv] K[kv, d]
            umma_ss(tmem + C::COL_DQ + 64 * qb, desc_mnmajor(adS, BN, k),
                    desc_mnmajor(aK, BN, k), idQ, k > 0);
          else           // dQ^T[d, q] = K^T[d, kv] dS^T[kv, q]
            umma_ss(tmem + C::COL_DQ + 64 * qb, desc_mnmajor(aK, BN, k),
                    desc_mnmajor(adS, BN, k), idQ, k > 0);
        }
        umma_commit(&bar_dq_full[qb]);
        umma_commit(&bar_ds_empty);
        umma_commit(&bar_qempty[st]);
        if (it + 1 < n_it) issue_dp(it + 1);
      }
      umma_commit(&bar_done);
    }
  } else if (warp < 4) {
    // ---------------- P / dS warpgroup (one KV row per thread) ----------------
    const int r = threadIdx.x;                         // KV row in tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int kv = kv0 + r;                            // KV row inside the sequence
    const bool kv_ok = kv < seq.len;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = hk * G + it / n_i;
      const int q0 = (i_start + it % n_i) * BM;
      const int buf = it & 1;
      if (r < BM) {
        const int q = q0 + r;
        float l = INFINITY, dl = 0.f;
        if (q < seq.len) {
          size_t li;
          if (p.cu_seqlens)
            li = static_cast<size_t>(h) * p.rows_total + seq.row0 + q;
          else
            li = (static_cast<size_t>(seq.b) * p.heads_q + h) * p.rows_total + q;
          l = __ldg(a.lse + li) * kLog2e;
          dl = __ldg(a.delta + li);
        }
        s_lse[buf][r] = l;
        s_delta[buf][r] = dl;
      }
      named_bar_sync(1, 128);
      // ---- P^T row ----
      if (!mbar_wait(&bar_s, it & 1, ac)) { ok = false; break; }
      tc_fence_after();
      float pv[BM];
#pragma unroll
      for (int c = 0; c < BM; c += 32) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + C::COL_S + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) pv[c + i] = __uint_as_float(u[i]);
      }
      const bool diag = p.causal && (q0 < kv0 + BN);
#pragma unroll
      for (int c = 0; c < BM; ++c) {
        float e = ex2(fmaf(pv[c], sl2, -s_lse[buf][c]));
        if (!kv_ok || (diag && q0 + c < kv)) e = 0.f;
        pv[c] = e;
      }
      if (it > 0 && !mbar_wait(&bar_pt_empty, (it - 1) & 1, ac)) { ok = false; break; }
#pragma unroll
      for (int ch = 0; ch < BM / 8; ++ch) {
        const uint32_t off = (ch >> 3) * BN * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        uint4 v = make_uint4(pack_bf16(pv[ch * 8 + 0], pv[ch * 8 + 1]),
                             pack_bf16(pv[ch * 8 + 2], pv[ch * 8 + 3]),
                             pack_bf16(pv[ch * 8 + 4], pv[ch * 8 + 5]),
                             pack_bf16(pv[ch * 8 + 6], pv[ch * 8 + 7]));
        *reinterpret_cast<uint4*>(sPt + off) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p);
      // ---- dS^T row ----
      if (!mbar_wait(&bar_dp, it & 1, ac)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < BM; c += 32) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + C::COL_DP + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pv[c + i] = pv[c + i] * (__uint_as_float(u[i]) - s_delta[buf][c + i]);
      }
      if (it > 0 && !mbar_wait(&bar_ds_empty, (it - 1) & 1, ac)) { ok = false; break; }
#pragma unroll
      for (int ch = 0; ch < BM / 8; ++ch) {
        const uint32_t off = (ch >> 3) * BN * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
        uint4 v = make_uint4(pack_bf16(pv[ch * 8 + 0], pv[ch * 8 + 1]),
                             pack_bf16(pv[ch * 8 + 2], pv[ch * 8 + 3]),
                             pack_bf16(pv[ch * 8 + 4], pv[ch * 8 + 5]),
                             pack_bf16(pv[ch * 8 + 6], pv[ch * 8 + 7]));
        *reinterpret_cast<uint4*>(sdS + off) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_ds);
    }
    // ---- epilogue: dK (x scale) and dV rows ----
    if (ok && mbar_wait(&bar_done, 0, ac)) {
      tc_fence_after();
      const size_t grow = static_cast<size_t>(seq.b) * p.rows_total + seq.row0 + kv;
      __nv_bfloat16* dkrow = a.dk + (grow * p.heads_kv + hk) * D;
      __nv_bfloat16* dvrow = a.dv + (grow * p.heads_kv + hk) * D;
      const float sc = p.scale;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        uint32_t u[16], w[16];
        tmem_ld16(tmem + lane_base + C::COL_DK + c, u);
        tmem_ld16(tmem + lane_base + C::COL_DV + c, w);
        tmem_wait_ld();
        if (kv_ok) {
          uint4 k0, k1, v0, v1;
          k0.x = pack_bf16(__uint_as_float(u[0]) * sc, __uint_as_float(u[1]) * sc);
          k0.y = pack_bf16(__uint_as_float(u[2]) * sc, __uint_as_float(u[3]) * sc);
          k0.z = pack_bf16(__uint_as_float(u[4]) * sc, __uint_as_float(u[5]) * sc);
          k0.w = pack_bf16(__uint_as_float(u[6]) * sc, __uint_as_float(u[7]) * sc);
          k1.x = pack_bf16(__uint_as_float(u[8]) * sc, __uint_as_float(u[9]) * sc);
          k1.y = pack_bf16(__uint_as_float(u[10]) * sc, __uint_as_float(u[11]) * sc);
          k1.z = pack_bf16(__uint_as_float(u[12]) * sc, __uint_as_float(u[13]) * sc);
          k1.w = pack_bf16(__uint_as_float(u[14]) * sc, __uint_as_float(u[15]) * sc);
          v0.x = pack_bf16(__uint_as_float(w[0]), __uint_as_float(w[1]));
          v0.y = pack_bf16(__uint_as_float(w[2]), __uint_as_float(w[3]));
          v0.z = pack_bf16(__uint_as_float(w[4]), __uint_as_float(w[5]));
          v0.w = pack_bf16(__uint_as_float(w[6]), __uint_as_float(w[7]));
          v1.x = pack_bf16(__uint_as_float(w[8]), __uint_as_float(w[9]));
          v1.y = pack_bf16(__uint_as_float(w[10]), __uint_as_float(w[11]));
          v1.z = pack_bf16(__uint_as_float(w[12]), __uint_as_float(w[13]));
          v1.w = pack_bf16(__uint_as_float(w[14]), __uint_as_float(w[15]));
          *reinterpret_cast<uint4*>(dkrow + c) = k0;
          *reinterpret_cast<uint4*>(dkrow + c + 8) = k1;
          *reinterpret_cast<uint4*>(dvrow + c) = v0;
          *reinterpret_cast<uint4*>(dvrow + c + 8) = v1;
        }
      }
    }
  } else {
    // ---------------- dQ drain (warps 4..7) ----------------
    const int t = threadIdx.x - 128;
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
      const int qb = it & 1, qu = it >> 1;
      if (!mbar_wait(&bar_dq_full[qb], qu & 1, ac)) break;
      tc_fence_after();
      uint32_t u[64];
      {
        uint32_t (&u0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[0]);
        uint32_t (&u1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[32]);
        tmem_ld32(tmem + lane_base + C::COL_DQ + 64 * qb, u0);
        tmem_ld32(tmem + lane_base + C::COL_DQ + 64 * qb + 32, u1);
        tmem_wait_ld();
      }
      tc_fence_before();
      mbar_arrive(&bar_dq_empty[qb]);
      if (!slab_ok) continue;
      if (D == 64) {
        // lane = query row, 64 columns = head dims
        const int q = q0 + t;
        if (q < seq.len) {
          float* dst = base + ((static_cast<size_t>(seq.b) * p.rows_total + seq.row0 + q) *
                                   p.heads_q + h) * D;
          if (a.split) {
#pragma unroll
            for (int c = 0; c < 64; c += 4)
              *reinterpret_cast<float4*>(dst + c) =
                  make_float4(__uint_as_float(u[c]), __uint_as_float(u[c + 1]),
                              __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
          } else {
#pragma unroll
            for (int c = 0; c < 64; c += 4)
              red_add_v4(dst + c, __uint_as_float(u[c]), __uint_as_float(u[c + 1]),
                         __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
          }
        }
      } else {
        // lane = head dim, 64 columns = query rows
        const int d = t;
        const int nq = min(BM, seq.len - q0);
        float* dst = base + ((static_cast<size_t>(seq.b) * p.rows_total + seq.row0 + q0) *
                                 p.heads_q + h) * D + d;
        const size_t rs = static_cast<size_t>(p.heads_q) * D;
        if (a.split) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < nq) dst[c * rs] = __uint_as_float(u[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < nq) red_add(dst + c * rs, __uint_as_float(u[c]));
        }
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
