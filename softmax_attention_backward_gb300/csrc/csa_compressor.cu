// CSA compressor gated-softmax pooling, forward and backward ("CSA: add fused
// Compressor forward+backward CuTe-DSL kernels (ported from Megatron-LM)",
// cudnn-frontend #427): per compressed row, a window of `ratio` tokens (and,
// with coff == 2, the previous block's tokens through the other column half),
// a softmax over the window per output dim and the weighted sum.  The formulas
// and layouts are documented in dsa.h.
//
// Both kernels are HBM-bound streams.  A CTA of 256 threads covers 16 rows x
// 64 dims: 16 threads per row, 4 dims (one 8-byte bf16x4 load) per thread, so a
// half-warp reads one 128-byte line of a token row.  Every (token, column) is
// read by exactly one window, so the kernels read kv and score once.
// The backward writes dkv / dscore by disjoint stores, lets the owner of each
// never-read slot write its exact zero (the last block of a segment: its own
// first-half columns and the tail tokens; a grid-stride sweep: segments shorter
// than ratio and the padding tokens), and sums dape in two fixed-order stages
// (per CTA row group into a workspace slab, then over the slabs), so all
// outputs are bitwise reproducible.
#include <cuda_runtime.h>

#include <type_traits>

#include "dsa.h"
#include "launch.h"

namespace attn {
namespace {

constexpr int kDC = 64;                 // dims per CTA column chunk
constexpr int kVec = 4;                 // dims per thread
constexpr int kTPR = kDC / kVec;        // threads per row
constexpr int kRPB = 16;                // rows per CTA pass
constexpr int kThreads = kTPR * kRPB;   // 256

struct CsaArgs {
  const __nv_bfloat16* kv;
  const __nv_bfloat16* score;
  const float* ape;
  const __nv_bfloat16* dout;
  __nv_bfloat16* out;
  __nv_bfloat16* dkv;
  __nv_bfloat16* dscore;
  float* partial;           // [row groups][ratio][coff * D]
  const int32_t* cu;
  const int32_t* cuc;
  int T, C, nseq, D, ld;    // ld = coff * D
  int32_t* err;
};

// Segment boundaries (cu_seqlens, cu_seqlens_comp) as the kernels read them:
// staged once per CTA in shared memory when there are at most kSegCache
// segments (one global round trip instead of two dependent ones per row),
// else straight from global memory.
constexpr int kSegCache = 511;
struct SegTab {
  const int32_t* cu;
  const int32_t* cuc;
};

__device__ __forceinline__ SegTab stage_segments(const CsaArgs& a, int32_t* s_cu, int32_t* s_cuc) {
  if (a.nseq > kSegCache) return SegTab{a.cu, a.cuc};   // CTA-uniform
  for (int i = threadIdx.x; i <= a.nseq; i += blockDim.x) {
    s_cu[i] = __ldg(a.cu + i);
    s_cuc[i] = __ldg(a.cuc + i);
  }
  __syncthreads();
  return SegTab{s_cu, s_cuc};
}

// Token range and compressed rows of segment n, validated on the device.
struct Seg {
  int tok0, len, row0, nb;
  bool ok;
};

__device__ __forceinline__ Seg load_seg(const CsaArgs& a, const SegTab& tb, int n, int ratio) {
  Seg s;
  const int t0 = tb.cu[n], t1 = tb.cu[n + 1];
  const int c0 = tb.cuc[n], c1 = tb.cuc[n + 1];
  s.ok = 0 <= t0 && t0 <= t1 && t1 <= a.T && 0 <= c0 && c0 <= c1 && c1 <= a.C;
  s.tok0 = min(max(t0, 0), a.T);
  s.len = s.ok ? t1 - t0 : 0;
  s.row0 = c0;
  s.nb = s.len / ratio;
  if (s.ok && c1 - c0 != s.nb) s.ok = false;
  if (!s.ok) {
    s.len = 0;
    s.nb = 0;
  }
  return s;
}

// Segment of compressed row c (the last n with cuc[n] <= c), or -1.
__device__ __forceinline__ int row_segment(const CsaArgs& a, const SegTab& tb, int c) {
  if (c < tb.cuc[0] || c >= tb.cuc[a.nseq]) return -1;
  int lo = 0, hi = a.nseq;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tb.cuc[mid] <= c) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void flag(const CsaArgs& a, int bit) {
  if (a.err) atomicOr(a.err, bit);
}

__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float* f) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  f[0] = x.x; f[1] = x.y; f[2] = y.x; f[3] = y.y;
}

__device__ __forceinline__ void st4(__nv_bfloat16* p, const float* f) {
  uint2 u;
  u.x = pack_bf16(f[0], f[1]);
  u.y = pack_bf16(f[2], f[3]);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ void st4_zero(__nv_bfloat16* p) {
  *reinterpret_cast<uint2*>(p) = make_uint2(0u, 0u);
}

// Window of row c (block b of a segment starting at tok0): entry e reads token
// tok(e) at column offset off(e) with position r(e).  Own entries first.
template <int R, int COFF>
struct Win {
  static constexpr int N = R * COFF;
  __device__ static int tok(int e, int t0) { return e < R ? t0 + e : t0 - R + (e - R); }
  __device__ static int off(int e, int D) { return (COFF == 2 && e < R) ? D : 0; }
  __device__ static int r(int e) { return e < R ? e : e - R; }
  __device__ static int part(int e) { return (COFF == 2 && e < R) ? 1 : 0; }
};

__device__ __forceinline__ void unpack4(uint2 u, float* f) {
  const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  f[0] = x.x; f[1] = x.y; f[2] = y.x; f[3] = y.y;
}

// APE of the thread's 4 dims for every window entry (the same for every row),
// times log2 e: the softmax runs in base 2.
template <int R, int COFF>
__device__ __forceinline__ void load_ape(const CsaArgs& a, int d, float (&ap)[R * COFF][4]) {
  using Wn = Win<R, COFF>;
#pragma unroll
  for (int e = 0; e < Wn::N; ++e) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(
        a.ape + static_cast<size_t>(Wn::r(e)) * a.ld + Wn::off(e, a.D) + d));
    ap[e][0] = x.x * kLog2e; ap[e][1] = x.y * kLog2e; ap[e][2] = x.z * kLog2e; ap[e][3] = x.w * kLog2e;
  }
}

// Loads the window entries of one row for the 4 dims at d as packed bf16 (kv
// and score); entries of the previous block (e >= R) are loaded from the row's
// own first token when b == 0 and masked later.
template <int R, int COFF>
__device__ __forceinline__ void load_window(const CsaArgs& a, int t0, bool has_prev, int d,
                                            uint2 (&v)[R * COFF], uint2 (&s)[R * COFF]) {
  using Wn = Win<R, COFF>;
#pragma unroll
  for (int e = 0; e < Wn::N; ++e) {
    const bool on = e < R || has_prev;
    const int t = on ? Wn::tok(e, t0) : t0;
    const size_t off = static_cast<size_t>(t) * a.ld + Wn::off(e, a.D) + d;
    v[e] = __ldg(reinterpret_cast<const uint2*>(a.kv + off));
    s[e] = __ldg(reinterpret_cast<const uint2*>(a.score + off));
  }
}

// Softmax over the window per dim (masked entries excluded) and the pooled
// output; the weights go to w when W is true.  Base 2: with ap holding
// log2 e * ape, (score + ape) log2 e is one FMA per entry and dim, and the
// exponent is ex2.approx.
template <int R, int COFF, bool W>
__device__ __forceinline__ void pool(const uint2 (&v)[R * COFF], const uint2 (&sr)[R * COFF],
                                     const float (&ap)[R * COFF][4], bool has_prev,
                                     float (&w)[W ? R * COFF : 1][4], float* o) {
  constexpr int N = R * COFF;
  // the exponent argument is recomputed in the second pass rather than kept:
  // one FMA against 4 N live registers
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if (e >= R && !has_prev) continue;
    float x[4];
    unpack4(sr[e], x);
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], fmaf(x[k], kLog2e, ap[e][k]));
  }
  float z[4] = {0.f, 0.f, 0.f, 0.f}, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < N; ++e) {
    float x[4], y[4];
    unpack4(sr[e], x);
    unpack4(v[e], y);
    const bool on = e < R || has_prev;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float ew = on ? ex2(fmaf(x[k], kLog2e, ap[e][k]) - m[k]) : 0.f;
      if (W) w[W ? e : 0][k] = ew;
      z[k] += ew;
      acc[k] = fmaf(ew, y[k], acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float inv = __fdividef(1.f, z[k]);
    if (W) {
#pragma unroll
      for (int e = 0; e < N; ++e) w[W ? e : 0][k] *= inv;
    }
    o[k] = acc[k] * inv;
  }
}

// Window of row c into registers; false when c is a padding row or belongs to a
// rejected segment.
template <int R, int COFF>
__device__ __forceinline__ bool fwd_row(const CsaArgs& a, const SegTab& tb, int c, int d,
                                        uint2 (&v)[R * COFF], uint2 (&sc)[R * COFF],
                                        bool& has_prev) {
  const int n = row_segment(a, tb, c);
  if (n < 0) return false;
  const Seg s = load_seg(a, tb, n, R);
  const int b = c - s.row0;
  if (!s.ok || b >= s.nb) {
    if (threadIdx.x % kTPR == 0) flag(a, ATTN_DEVERR_LAYOUT);
    return false;
  }
  has_prev = b > 0;
  load_window<R, COFF>(a, s.tok0 + b * R, has_prev, d, v, sc);
  return true;
}

// Persistent grid: each thread takes RPT rows per pass (c, c + stride, ...),
// all windows loaded before any is reduced, so that RPT times the loads are in
// flight and the per-row segment lookups overlap.  RPT = 1 when the rows fit in
// about four CTAs per SM that way (more threads for the short problems), else 2.
template <int R, int COFF, int RPT>
__global__ void __launch_bounds__(kThreads, (R * COFF <= 8) ? 2 : 1) csa_fwd_kernel(const CsaArgs a) {
  constexpr int N = R * COFF;
  __shared__ int32_t s_cu[kSegCache + 1], s_cuc[kSegCache + 1];
  const int tx = threadIdx.x % kTPR, ty = threadIdx.x / kTPR;
  const int d = blockIdx.x * kDC + tx * kVec;
  const int stride = gridDim.y * kRPB;
  float ap[N][4];
  load_ape<R, COFF>(a, d, ap);   // in flight while the segment table is staged
  const SegTab tb = stage_segments(a, s_cu, s_cuc);
  float unused[1][4];
  for (int c = blockIdx.y * kRPB + ty; c < a.C; c += RPT * stride) {
    uint2 v[RPT][N], sc[RPT][N];
    bool hp[RPT], on[RPT];
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      hp[u] = false;
      on[u] = c + u * stride < a.C && fwd_row<R, COFF>(a, tb, c + u * stride, d, v[u], sc[u], hp[u]);
    }
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
      if (c + u * stride >= a.C) continue;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      if (on[u]) pool<R, COFF, false>(v[u], sc[u], ap, hp[u], unused, o);
      st4(a.out + static_cast<size_t>(c + u * stride) * a.D + d, o);
    }
  }
}

// Shared memory of the backward: per thread, the running dape sums of its
// 4 dims for every window entry, [entry * 4 + k][thread] (conflict-free).
template <int R, int COFF>
constexpr int bwd_smem_bytes() { return R * COFF * 4 * kThreads * 4; }

template <int R, int COFF>
__global__ void __launch_bounds__(kThreads, (R * COFF <= 8) ? 2 : 1) csa_bwd_kernel(const CsaArgs a) {
  constexpr int N = R * COFF;
  extern __shared__ float dacc[];              // [N * 4][kThreads]
  __shared__ int32_t s_cu[kSegCache + 1], s_cuc[kSegCache + 1];
  const int tx = threadIdx.x % kTPR, ty = threadIdx.x / kTPR;
  const int d = blockIdx.x * kDC + tx * kVec;
  float ap[N][4];
  load_ape<R, COFF>(a, d, ap);   // in flight while the segment table is staged
  for (int i = 0; i < N * 4; ++i) dacc[i * kThreads + threadIdx.x] = 0.f;
  const SegTab tb = stage_segments(a, s_cu, s_cuc);

  for (int c = blockIdx.y * kRPB + ty; c < a.C; c += gridDim.y * kRPB) {
    const int n = row_segment(a, tb, c);
    if (n < 0) continue;                       // padding row: its dout is ignored
    const Seg s = load_seg(a, tb, n, R);
    const int b = c - s.row0;
    if (!s.ok || b >= s.nb) {
      if (tx == 0) flag(a, ATTN_DEVERR_LAYOUT);
      continue;
    }
    const int t0 = s.tok0 + b * R;
    uint2 v[N], sr[N];
    float w[N][4], o[4], g[4];
    load_window<R, COFF>(a, t0, b > 0, d, v, sr);
    ld4(a.dout + static_cast<size_t>(c) * a.D + d, g);
    pool<R, COFF, true>(v, sr, ap, b > 0, w, o);
#pragma unroll
    for (int e = 0; e < N; ++e) {
      if (e >= R && b == 0) continue;          // no previous block
      float x[4], dk[4], ds[4];
      unpack4(v[e], x);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        dk[k] = w[e][k] * g[k];
        ds[k] = dk[k] * (x[k] - o[k]);
        dacc[(e * 4 + k) * kThreads + threadIdx.x] += ds[k];
      }
      const size_t off = static_cast<size_t>(Win<R, COFF>::tok(e, t0)) * a.ld +
                         Win<R, COFF>::off(e, a.D) + d;
      st4(a.dkv + off, dk);
      st4(a.dscore + off, ds);
    }
    if (b == s.nb - 1) {
      // last block of the segment: the zeros nobody else reads or writes
      if (COFF == 2) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const size_t off = static_cast<size_t>(t0 + r) * a.ld + d;
          st4_zero(a.dkv + off);
          st4_zero(a.dscore + off);
        }
      }
      for (int t = t0 + R; t < s.tok0 + s.len; ++t) {
#pragma unroll
        for (int h = 0; h < COFF; ++h) {
          const size_t off = static_cast<size_t>(t) * a.ld + h * a.D + d;
          st4_zero(a.dkv + off);
          st4_zero(a.dscore + off);
        }
      }
    }
  }

  // Segments without a compressed row (shorter than ratio, or rejected
  // layouts): every token is zero.  Then the padding tokens.
  for (int n = blockIdx.y * kRPB + ty; n < a.nseq; n += gridDim.y * kRPB) {
    const Seg s = load_seg(a, tb, n, R);
    if (s.nb > 0) continue;
    int t_lo = s.tok0, t_hi = s.tok0 + s.len;
    if (!s.ok) {                                // zero what the segment claims, in bounds
      t_lo = min(max(tb.cu[n], 0), a.T);
      t_hi = min(max(tb.cu[n + 1], t_lo), a.T);
      if (tx == 0) flag(a, ATTN_DEVERR_LAYOUT);
    }
    for (int t = t_lo; t < t_hi; ++t) {
#pragma unroll
      for (int h = 0; h < COFF; ++h) {
        const size_t off = static_cast<size_t>(t) * a.ld + h * a.D + d;
        st4_zero(a.dkv + off);
        st4_zero(a.dscore + off);
      }
    }
  }
  const int end = min(max(tb.cu[a.nseq], 0), a.T);
  for (int t = end + blockIdx.y * kRPB + ty; t < a.T; t += gridDim.y * kRPB) {
#pragma unroll
    for (int h = 0; h < COFF; ++h) {
      const size_t off = static_cast<size_t>(t) * a.ld + h * a.D + d;
      st4_zero(a.dkv + off);
      st4_zero(a.dscore + off);
    }
  }

  // dape partial of this CTA (rows blockIdx.y, dims of chunk blockIdx.x): the
  // 16 rows of the CTA are added in row order.
  __syncthreads();
  float* slab = a.partial + static_cast<size_t>(blockIdx.y) * R * a.ld;
  for (int i = threadIdx.x; i < N * kDC; i += kThreads) {
    const int e = i / kDC, dd = i % kDC;
    const int col = (dd / kVec) , k = dd % kVec;
    float sum = 0.f;
#pragma unroll
    for (int row = 0; row < kRPB; ++row) sum += dacc[(e * 4 + k) * kThreads + row * kTPR + col];
    slab[static_cast<size_t>(Win<R, COFF>::r(e)) * a.ld + Win<R, COFF>::off(e, a.D) +
         blockIdx.x * kDC + dd] = sum;
  }
}

// dape[i] = sum over row groups g (ascending, in eight interleaved lanes that
// are then added in lane order) of partial[g][i].
__global__ void __launch_bounds__(256) csa_dape_reduce_kernel(const float* partial, int groups,
                                                              int n, float* dape) {
  __shared__ float red[8][33];
  const int x = threadIdx.x & 31, y = threadIdx.x >> 5;
  const int i = blockIdx.x * 32 + x;
  float sum = 0.f;
  if (i < n)
    for (int g = y; g < groups; g += 8) sum += partial[static_cast<size_t>(g) * n + i];
  red[y][x] = sum;
  __syncthreads();
  if (y == 0 && i < n) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += red[k][x];
    dape[i] = t;
  }
}

template <typename F>
cudaError_t dispatch(int ratio, int coff, F&& f) {
  if (coff == 2) {
    if (ratio == 4) return f(std::integral_constant<int, 4>{}, std::integral_constant<int, 2>{});
    if (ratio == 2) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 2>{});
    if (ratio == 8) return f(std::integral_constant<int, 8>{}, std::integral_constant<int, 2>{});
  } else {
    if (ratio == 4) return f(std::integral_constant<int, 4>{}, std::integral_constant<int, 1>{});
    if (ratio == 2) return f(std::integral_constant<int, 2>{}, std::integral_constant<int, 1>{});
    if (ratio == 8) return f(std::integral_constant<int, 8>{}, std::integral_constant<int, 1>{});
  }
  return cudaErrorInvalidValue;
}

bool aligned(const void* p, unsigned m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; }

attn_status_t check(const csa_compressor_problem_t* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->tokens < 0 || p->comp_capacity < 0 || p->num_seqs <= 0 || p->head_dim <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (p->coff != 1 && p->coff != 2) return ATTN_ERR_UNSUPPORTED;
  if (p->ratio != 2 && p->ratio != 4 && p->ratio != 8) return ATTN_ERR_UNSUPPORTED;
  if (p->head_dim % kDC != 0 || p->head_dim > 1024) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->tokens) * p->coff * p->head_dim >= (int64_t(1) << 31) ||
      static_cast<int64_t>(p->comp_capacity) * p->head_dim >= (int64_t(1) << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (!p->cu_seqlens || !p->cu_seqlens_comp) return ATTN_ERR_INVALID_ARG;
  if (!aligned(p->cu_seqlens, 4) || !aligned(p->cu_seqlens_comp, 4)) return ATTN_ERR_ALIGNMENT;
  return ATTN_OK;
}

// Row groups (grid.y) of the backward: about four CTAs per SM in total.
int bwd_row_groups(const csa_compressor_problem_t* p) {
  const int ndc = p->head_dim / kDC;
  const int sms = sm_count() > 0 ? sm_count() : 1;
  const int need = (p->comp_capacity + kRPB - 1) / kRPB;
  const int cap = (4 * sms + ndc - 1) / ndc;
  return need < 1 ? 1 : (need < cap ? need : cap);
}

CsaArgs make_args(const csa_compressor_problem_t* p) {
  CsaArgs a{};
  a.cu = p->cu_seqlens;
  a.cuc = p->cu_seqlens_comp;
  a.T = p->tokens;
  a.C = p->comp_capacity;
  a.nseq = p->num_seqs;
  a.D = p->head_dim;
  a.ld = p->coff * p->head_dim;
  a.err = p->error_word;
  return a;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t csa_compressor_fwd(const csa_compressor_problem_t* p, const void* kv,
                                            const void* score, const float* ape, void* out,
                                            attn_stream_t stream) {
  const attn_status_t s = check(p);
  if (s != ATTN_OK) return s;
  if (p->comp_capacity == 0) return ATTN_OK;    // no output row: nothing to write
  if (!ape || !out || (p->tokens > 0 && (!kv || !score))) return ATTN_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(ape, 16) || !aligned(out, 16))
    return ATTN_ERR_ALIGNMENT;
  CsaArgs a = make_args(p);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.score = static_cast<const __nv_bfloat16*>(score);
  a.ape = ape;
  a.out = static_cast<__nv_bfloat16*>(out);
  // about four CTAs per SM: one row per thread and pass when the rows fit
  // that way, else two
  const int ndc = p->head_dim / kDC;
  const int sms = sm_count() > 0 ? sm_count() : 1;
  const int cap = (4 * sms + ndc - 1) / ndc;
  const int need1 = (p->comp_capacity + kRPB - 1) / kRPB;
  const int need2 = (p->comp_capacity + 2 * kRPB - 1) / (2 * kRPB);
  const bool one = need1 <= cap;
  const dim3 grid(ndc, one ? need1 : (need2 < cap ? need2 : cap));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = dispatch(p->ratio, p->coff, [&](auto R, auto CF) {
    constexpr int r = decltype(R)::value, cf = decltype(CF)::value;
    if (one) csa_fwd_kernel<r, cf, 1><<<grid, kThreads, 0, st>>>(a);
    else csa_fwd_kernel<r, cf, 2><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
  });
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" size_t csa_compressor_bwd_workspace_size(const csa_compressor_problem_t* p) {
  if (check(p) != ATTN_OK) return 0;
  return static_cast<size_t>(bwd_row_groups(p)) * p->ratio * p->coff * p->head_dim * sizeof(float);
}

extern "C" attn_status_t csa_compressor_bwd(const csa_compressor_problem_t* p, const void* kv,
                                            const void* score, const float* ape, const void* dout,
                                            void* dkv, void* dscore, float* dape, void* workspace,
                                            size_t workspace_bytes, attn_stream_t stream) {
  const attn_status_t s = check(p);
  if (s != ATTN_OK) return s;
  // token buffers may be null when there is no token, dout when there is no
  // compressed row (they are never touched then); dape is always written
  const bool tok = p->tokens > 0;
  if (!ape || !dape || (tok && (!kv || !score || !dkv || !dscore)) ||
      (!dout && p->comp_capacity > 0))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(ape, 16) || !aligned(dout, 16) ||
      !aligned(dkv, 16) || !aligned(dscore, 16) || !aligned(dape, 16))
    return ATTN_ERR_ALIGNMENT;
  const size_t need = csa_compressor_bwd_workspace_size(p);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return ATTN_ERR_ALIGNMENT;
  CsaArgs a = make_args(p);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.score = static_cast<const __nv_bfloat16*>(score);
  a.ape = ape;
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.dkv = static_cast<__nv_bfloat16*>(dkv);
  a.dscore = static_cast<__nv_bfloat16*>(dscore);
  a.partial = static_cast<float*>(workspace);
  const int groups = bwd_row_groups(p);
  const dim3 grid(p->head_dim / kDC, groups);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dispatch(p->ratio, p->coff, [&](auto R, auto CF) {
    constexpr int r = decltype(R)::value, cf = decltype(CF)::value;
    constexpr int smem = bwd_smem_bytes<r, cf>();
    cudaError_t x = cudaFuncSetAttribute(csa_bwd_kernel<r, cf>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (x != cudaSuccess) return x;
    csa_bwd_kernel<r, cf><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  const int n = p->ratio * p->coff * p->head_dim;
  csa_dape_reduce_kernel<<<(n + 31) / 32, 256, 0, st>>>(a.partial, groups, n, dape);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
