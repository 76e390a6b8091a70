// C ABI of the library: argument validation, TMA descriptor encoding and the
// launch sequence of each entry point (declared and documented in attn.h).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "launch.h"
#include "thd_order.cuh"

namespace attn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D map over a bf16 tensor [batch, rows, heads, dim] (dim contiguous), box of
// 64 dims x 1 head x box_rows rows x 1 batch, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* m, const void* ptr, int batch, int rows, int heads, int dim,
              int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(dim) * 2,
                           static_cast<cuuint64_t>(heads) * dim * 2,
                           static_cast<cuuint64_t>(rows) * heads * dim * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over the fp32 dQ accumulator [batch, heads, rows, dim] (head-major), or
// over `n_split` such slabs when n_split > 0 (5-D, slab outermost): box of 32
// dims x 128 rows, 128-byte swizzle, matching the staging layout of the D = 64
// backward kernel.  Rows past `rows` are clipped by the copy.
bool make_dq_map(CUtensorMap* m, float* acc, int batch, int rows, int heads, int dim, int n_split,
                 size_t slab_elems) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t rank = n_split > 0 ? 5 : 4;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch),
                        static_cast<cuuint64_t>(n_split > 0 ? n_split : 1)};
  cuuint64_t strides[4] = {static_cast<cuuint64_t>(dim) * 4,
                           static_cast<cuuint64_t>(rows) * dim * 4,
                           static_cast<cuuint64_t>(heads) * rows * dim * 4,
                           static_cast<cuuint64_t>(slab_elems) * 4};
  cuuint32_t box[5] = {32, 128, 1, 1, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, acc, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a dense/THD problem.  Sets *empty when there is nothing to compute.
attn_status_t check_problem(const attn_problem_t* p, bool* empty) {
  *empty = false;
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->heads_q <= 0 || p->heads_kv <= 0 || p->head_dim <= 0) return ATTN_ERR_INVALID_ARG;
  if (p->heads_q % p->heads_kv) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return ATTN_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->cu_seqlens) {
    if (p->num_seqs <= 0 || p->capacity < 0 || p->max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p->cu_seqlens) & 3u) != 0) return ATTN_ERR_ALIGNMENT;
    if (p->capacity == 0 || p->max_seqlen == 0) *empty = true;
    if (static_cast<int64_t>(p->capacity) * p->heads_q * p->head_dim >= (int64_t(1) << 31))
      return ATTN_ERR_UNSUPPORTED;
  } else {
    if (p->batch < 0 || p->seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if (p->batch == 0 || p->seqlen == 0) *empty = true;
    if (static_cast<int64_t>(p->seqlen) * p->heads_q * p->head_dim >= (int64_t(1) << 31))
      return ATTN_ERR_UNSUPPORTED;
    if (p->batch > 65535) return ATTN_ERR_UNSUPPORTED;
    // the memory-bound passes index (row, head, 8-dim chunk) in 32 bits
    if (static_cast<int64_t>(p->batch) * p->seqlen * p->heads_q * p->head_dim >= (int64_t(1) << 34))
      return ATTN_ERR_UNSUPPORTED;
  }
  if (p->heads_q > 65535) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

Problem to_kernel(const attn_problem_t* p) {
  Problem k;
  const bool thd = p->cu_seqlens != nullptr;
  k.batch = thd ? 1 : p->batch;
  k.rows_total = thd ? p->capacity : p->seqlen;
  k.heads_q = p->heads_q;
  k.heads_kv = p->heads_kv;
  k.causal = p->causal ? 1 : 0;
  k.scale = p->scale;
  k.cu_seqlens = p->cu_seqlens;
  k.num_seqs = thd ? p->num_seqs : 0;
  k.max_seqlen = thd ? p->max_seqlen : p->seqlen;
  k.err = p->error_word;
  k.fd_hq = make_fastdiv(static_cast<uint32_t>(k.heads_q));
  k.fd_hkv = make_fastdiv(static_cast<uint32_t>(k.heads_kv));
  k.fd_grp = make_fastdiv(static_cast<uint32_t>(k.heads_kv > 0 ? k.heads_q / k.heads_kv : 1));
  k.fd_ns = make_fastdiv(static_cast<uint32_t>(k.num_seqs > 0 ? k.num_seqs : 1));
  return k;
}

size_t dq_elems(const Problem& k, int D) {
  return static_cast<size_t>(k.batch) * k.rows_total * k.heads_q * D;
}

int n_kv_tiles(const Problem& k) { return (k.max_seqlen + 127) / 128; }

// SPLIT at head_dim 128 accumulates in a fixed order into one accumulator,
// behind one int32 ticket per (batch, query head, 128-row query tile slot);
// the count is rounded up to whole 16-byte words for the clearing pass.
size_t dq_tickets(const Problem& k) {
  const size_t slots = static_cast<size_t>(
      tile_bound(k.rows_total, k.num_seqs, 128, k.cu_seqlens != nullptr));
  return (static_cast<size_t>(k.batch) * k.heads_q * slots + 3) / 4 * 4;
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }


}  // namespace

attn_status_t validate_dense_problem(const attn_problem_t* p, bool* empty) {
  return check_problem(p, empty);
}

bool make_bf16_tile_map(CUtensorMap* m, const void* ptr, int batch, int rows, int heads, int dim,
                        int box_rows) {
  return make_map(m, ptr, batch, rows, heads, dim, box_rows);
}

// Streaming multiprocessors of the current device (persistent grid size).
int sm_count() {
  constexpr int kMaxDevices = 64;
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported problem";
    case ATTN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_INDEX_RANGE: return "sparse index out of range";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int attn_version(void) { return 100; }

attn_status_t attn_fwd(const attn_problem_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_problem(p, &empty);
  if (s != ATTN_OK) return s;
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Problem kp = to_kernel(p);
  const int D = p->head_dim;
  CUtensorMap mq, mk, mv;
  const int bn = (D == 128) ? 64 : 128;   // key/value tile rows of the forward
  if (!make_map(&mq, q, kp.batch, kp.rows_total, kp.heads_q, D, 128) ||
      !make_map(&mk, k, kp.batch, kp.rows_total, kp.heads_kv, D, bn) ||
      !make_map(&mv, v, kp.batch, kp.rows_total, kp.heads_kv, D, bn))
    return ATTN_ERR_CUDA;
  FwdArgs a;
  a.p = kp;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.scale_log2 = p->scale * kLog2e;
  const int gx = tile_bound(kp.rows_total, kp.num_seqs, 256, kp.cu_seqlens != nullptr);
  const int64_t total = static_cast<int64_t>(gx) * kp.heads_q * kp.batch;
  if (total >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  a.total_items = static_cast<int>(total);
  a.n_x = gx;
  a.fd_nx = make_fastdiv(static_cast<uint32_t>(gx));
  a.fd_nbh = make_fastdiv(static_cast<uint32_t>(kp.heads_q * kp.batch));
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // Persistent grid (one CTA per SM, the next item's query pair prefetched).
  // For THD the slots run pair-rank-major over the sequences (every
  // sequence's longest pairs first) when that numbering fits the slot bound:
  // numbered sequence by sequence, the static list put a long sequence's
  // longest pairs after a shorter one's shortest, and at D = 128 one CTA per
  // item balanced better (c4 forward 766 against 711 TFLOP/s); pair-rank-major
  // it runs at 854.  Causal packs of at most 32 sequences take the list of
  // thd_order.cuh instead (descending work, no empty positions): c4 forward
  // 193 -> 186 us.
  const bool persistent = total > sms;
  a.x_major = persistent ? 1 : 0;
  if (persistent && kp.cu_seqlens &&
      static_cast<int64_t>((kp.max_seqlen + 255) / 256) * kp.num_seqs <= static_cast<int64_t>(gx))
    a.x_major = (kp.causal && kp.num_seqs <= kThdOrderSeqs) ? 3 : 2;
  const int grid = persistent ? sms : static_cast<int>(total);
  cudaError_t e = (D == 64) ? launch_attn_fwd<64>(mq, mk, mv, a, grid, st)
                            : launch_attn_fwd<128>(mq, mk, mv, a, grid, st);
  return cuda_status(e);
}

size_t attn_bwd_workspace_size(const attn_problem_t* p, attn_dq_mode_t mode) {
  bool empty;
  if (check_problem(p, &empty) != ATTN_OK) return 0;
  if (empty) return 0;
  const Problem kp = to_kernel(p);
  const size_t elems = dq_elems(kp, p->head_dim);
  if (mode == ATTN_DQ_SPLIT) {
    if (p->head_dim == 128) return (elems + dq_tickets(kp)) * sizeof(float);
    return elems * sizeof(float) * static_cast<size_t>(n_kv_tiles(kp));
  }
  return elems * sizeof(float);
}

attn_status_t attn_bwd_preprocess(const attn_problem_t* p, attn_dq_mode_t mode, const void* o,
                                  const void* dout, float* delta, void* workspace,
                                  size_t workspace_bytes, attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_problem(p, &empty);
  if (s != ATTN_OK) return s;
  if (mode != ATTN_DQ_ATOMIC && mode != ATTN_DQ_SPLIT) return ATTN_ERR_INVALID_ARG;
  if (!o || !dout || !delta) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(delta)) return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  const size_t need = attn_bwd_workspace_size(p, mode);
  // ATOMIC clears the accumulator; SPLIT at head_dim 128 clears its tickets
  const bool ordered = mode == ATTN_DQ_SPLIT && p->head_dim == 128;
  if ((mode == ATTN_DQ_ATOMIC || ordered) && (!workspace || workspace_bytes < need))
    return ATTN_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return ATTN_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Problem kp = to_kernel(p);
  const size_t elems = dq_elems(kp, p->head_dim);
  float* acc = (mode == ATTN_DQ_ATOMIC) ? static_cast<float*>(workspace) : nullptr;
  const size_t n = (mode == ATTN_DQ_ATOMIC) ? elems : 0;
  float* tickets = ordered ? static_cast<float*>(workspace) + elems : nullptr;
  const size_t nt = ordered ? dq_tickets(kp) : 0;
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* db = static_cast<const __nv_bfloat16*>(dout);
  cudaError_t e = (p->head_dim == 64)
                      ? launch_bwd_preprocess<64>(kp, ob, db, delta, acc, n, tickets, nt, st)
                      : launch_bwd_preprocess<128>(kp, ob, db, delta, acc, n, tickets, nt, st);
  return cuda_status(e);
}

attn_status_t attn_bwd(const attn_problem_t* p, attn_dq_mode_t mode, const void* q,
                       const void* k, const void* v, const void* dout, const float* lse,
                       const float* delta, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_problem(p, &empty);
  if (s != ATTN_OK) return s;
  if (mode != ATTN_DQ_ATOMIC && mode != ATTN_DQ_SPLIT) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !dout || !lse || !delta || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(delta) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  const size_t need = attn_bwd_workspace_size(p, mode);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Problem kp = to_kernel(p);
  const int D = p->head_dim;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, q, kp.batch, kp.rows_total, kp.heads_q, D, 128) ||
      !make_map(&mdo, dout, kp.batch, kp.rows_total, kp.heads_q, D, 128) ||
      !make_map(&mk, k, kp.batch, kp.rows_total, kp.heads_kv, D, 128) ||
      !make_map(&mv, v, kp.batch, kp.rows_total, kp.heads_kv, D, 128))
    return ATTN_ERR_CUDA;
  BwdArgs a;
  a.p = kp;
  a.lse = lse;
  a.delta = delta;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.dq_acc = static_cast<float*>(workspace);
  a.split = (mode == ATTN_DQ_SPLIT) ? 1 : 0;
  a.slab_elems = a.split ? dq_elems(kp, D) : 0;
  a.n_split = a.split ? n_kv_tiles(kp) : 0;
  a.dq_ticket = nullptr;
  if (a.split && D == 128) {   // one accumulator, ordered by tickets (no slabs)
    a.slab_elems = 0;
    a.n_split = 0;
    a.dq_ticket = reinterpret_cast<int*>(a.dq_acc + dq_elems(kp, D));
  }
  a.scale_log2 = p->scale * kLog2e;
  // D = 64 stages dQ tiles one query row per thread, which only the swizzled
  // TMA layout keeps free of bank conflicts.  A THD slab store of a tile that
  // crosses a sequence end would overwrite the next sequence's rows of the
  // same slab, so THD + SPLIT keeps the row-exact bulk copy.
  a.dq_tma = (D == 64 && !(kp.cu_seqlens && a.split)) ? 1 : 0;
  CUtensorMap mdq, mdk, mdv;
  memset(&mdq, 0, sizeof(mdq));
  if (a.dq_tma && !make_dq_map(&mdq, a.dq_acc, kp.batch, kp.rows_total, kp.heads_q, D,
                               a.split ? a.n_split : 0, a.slab_elems))
    return ATTN_ERR_CUDA;
  if (!make_map(&mdk, dk, kp.batch, kp.rows_total, kp.heads_kv, D, 128) ||
      !make_map(&mdv, dv, kp.batch, kp.rows_total, kp.heads_kv, D, 128))
    return ATTN_ERR_CUDA;
  // persistent grid: one CTA per SM over (K/V tile slot x kv head x batch) items
  const int gx = tile_bound(kp.rows_total, kp.num_seqs, 128, kp.cu_seqlens != nullptr);
  const int64_t total = static_cast<int64_t>(gx) * kp.heads_kv * kp.batch;
  if (total >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  a.total_items = static_cast<int>(total);
  a.n_x = gx;
  a.fd_nx = make_fastdiv(static_cast<uint32_t>(gx));
  a.fd_nbh = make_fastdiv(static_cast<uint32_t>(kp.heads_kv * kp.batch));
  // One persistent CTA per SM walks the items, so K/V loads and the dK/dV
  // epilogue of one item overlap the next.
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const bool persistent = total > sms;
  const int grid = persistent ? sms : static_cast<int>(total);
  a.x_major = persistent ? 1 : 0;
  // THD on the persistent grid: list positions tile-major over the sequences
  // (every sequence's first, longest tiles first) when that numbering fits the
  // slot bound, i.e. leaves few empty positions; with atomic dQ, causal packs
  // of at most 32 sequences in the descending-work list of thd_order.cuh
  // (c4 backward 416.6 -> 402.7 us; the split mode measured 3% slower with
  // it and keeps the tile-major list)
  if (persistent && kp.cu_seqlens &&
      static_cast<int64_t>(n_kv_tiles(kp)) * kp.num_seqs <= static_cast<int64_t>(gx))
    a.x_major = (kp.causal && kp.num_seqs <= kThdOrderSeqs && !a.split) ? 3 : 2;
  // THD: the padding rows of dK and dV are written by the main kernel (a warp
  // of its own, during the computation) instead of the postprocess
  a.pad_zero = kp.cu_seqlens ? 1 : 0;
  cudaError_t e = (D == 64) ? launch_attn_bwd<64>(mq, mk, mv, mdo, mdq, mdk, mdv, a, grid, st)
                            : launch_attn_bwd128(mq, mk, mv, mdo, a, grid, st);
  return cuda_status(e);
}

attn_status_t attn_bwd_postprocess(const attn_problem_t* p, attn_dq_mode_t mode,
                                   const void* workspace, size_t workspace_bytes, void* dq,
                                   void* dk, void* dv, attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_problem(p, &empty);
  if (s != ATTN_OK) return s;
  if (mode != ATTN_DQ_ATOMIC && mode != ATTN_DQ_SPLIT) return ATTN_ERR_INVALID_ARG;
  if (!dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  const size_t need = attn_bwd_workspace_size(p, mode);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const Problem kp = to_kernel(p);
  const int D = p->head_dim;
  // SPLIT at head_dim 128 leaves one accumulator (filled in a fixed order),
  // converted like ATOMIC's; head_dim 64 sums its slabs in order
  const int split = (mode == ATTN_DQ_SPLIT && D == 64) ? 1 : 0;
  const size_t slab = split ? dq_elems(kp, D) : 0;
  const int n_split = split ? n_kv_tiles(kp) : 0;
  const float* acc = static_cast<const float*>(workspace);
  auto* dqb = static_cast<__nv_bfloat16*>(dq);
  // THD: attn_bwd wrote the padding rows of dk and dv
  const bool kv_pad_done = kp.cu_seqlens != nullptr;
  auto* dkb = kv_pad_done ? nullptr : static_cast<__nv_bfloat16*>(dk);
  auto* dvb = kv_pad_done ? nullptr : static_cast<__nv_bfloat16*>(dv);
  cudaError_t e = (D == 64) ? launch_dq_finalize<64>(kp, acc, slab, split, n_split, dqb, dkb, dvb, st)
                            : launch_dq_finalize<128>(kp, acc, slab, split, n_split, dqb, dkb, dvb,
                                                      st);
  return cuda_status(e);
}

// ---------------------------------------------------------------------------
// Sparse
// ---------------------------------------------------------------------------
static attn_status_t check_sparse(const sparse_attn_problem_t* p, bool* empty) {
  *empty = false;
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (p->tokens < 0 || p->heads <= 0 || p->topk < 0 || p->dim_qk <= 0 || p->dim_v <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return ATTN_ERR_INVALID_ARG;
  if (p->dim_qk != 576 || p->dim_v != 512) return ATTN_ERR_UNSUPPORTED;
  if (p->heads != 16 && p->heads != 32 && p->heads != 64 && p->heads != 128)
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->tokens) * p->heads * p->dim_qk >= (int64_t(1) << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->tokens) * p->topk >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if (p->tokens > 2147483647 / 2) return ATTN_ERR_UNSUPPORTED;
  if (p->tokens == 0) *empty = true;
  return ATTN_OK;
}

static SparseArgs sparse_args(const sparse_attn_problem_t* p) {
  SparseArgs a{};
  a.T = p->tokens;
  a.H = p->heads;
  a.K = p->topk;
  a.scale = p->scale;
  a.scale_log2 = p->scale * kLog2e;
  a.err = p->error_word;
  return a;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

attn_status_t sparse_attn_fwd(const sparse_attn_problem_t* p, const void* q, const void* kv,
                              const int32_t* idx, void* o, float* lse, attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_sparse(p, &empty);
  if (s != ATTN_OK) return s;
  if (!q || !kv || !o || !lse || (!idx && p->topk > 0)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(idx) & 3u))
    return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  SparseArgs a = sparse_args(p);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.idx = idx;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  return cuda_status(launch_sparse_fwd(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Sparse backward workspace: fp32 dKV accumulator (shared: [T, 576]; slabs:
// slabs x [T, 576]) | Delta [T, H] fp32 | chunk counts [T] int32, each
// 256-byte aligned.
struct SparseBwdWs {
  size_t acc, delta, nch, bytes;
};
static int sparse_slabs(const sparse_attn_problem_t* p) {
  const int64_t items = static_cast<int64_t>(p->tokens) * ((p->heads + 63) / 64);
  return static_cast<int>(items < kSparseSlabs ? items : kSparseSlabs);
}
static SparseBwdWs sparse_bwd_ws(const sparse_attn_problem_t* p, int slabs) {
  SparseBwdWs w{};
  const size_t T = static_cast<size_t>(p->tokens);
  size_t at = 0;
  w.acc = at;   at += align256(static_cast<size_t>(slabs > 0 ? slabs : 1) * T * p->dim_qk * sizeof(float));
  w.delta = at; at += align256(T * p->heads * sizeof(float));
  w.nch = at;   at += align256(T * sizeof(int32_t));
  w.bytes = at;
  return w;
}

size_t sparse_attn_bwd_workspace_size(const sparse_attn_problem_t* p) {
  bool empty;
  if (check_sparse(p, &empty) != ATTN_OK || empty) return 0;
  return sparse_bwd_ws(p, 0).bytes;
}

size_t sparse_attn_bwd_deterministic_workspace_size(const sparse_attn_problem_t* p) {
  bool empty;
  if (check_sparse(p, &empty) != ATTN_OK || empty) return 0;
  return sparse_bwd_ws(p, sparse_slabs(p)).bytes;
}

static attn_status_t sparse_bwd_call(const sparse_attn_problem_t* p, bool deterministic,
                                     const void* q, const void* kv, const int32_t* idx,
                                     const void* o, const void* dout, const float* lse, void* dq,
                                     void* dkv, void* workspace, size_t workspace_bytes,
                                     attn_stream_t stream) {
  bool empty;
  attn_status_t s = check_sparse(p, &empty);
  if (s != ATTN_OK) return s;
  if (!q || !kv || !o || !dout || !lse || !dq || !dkv || (!idx && p->topk > 0))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dkv) || (reinterpret_cast<uintptr_t>(idx) & 3u))
    return ATTN_ERR_ALIGNMENT;
  if (empty) return ATTN_OK;
  const int slabs = deterministic ? sparse_slabs(p) : 0;
  const SparseBwdWs w = sparse_bwd_ws(p, slabs);
  if (!workspace || workspace_bytes < w.bytes) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_ALIGNMENT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SparseArgs a = sparse_args(p);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.idx = idx;
  a.o = static_cast<__nv_bfloat16*>(const_cast<void*>(o));
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.lse_in = lse;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dkv_acc = reinterpret_cast<float*>(ws + w.acc);
  a.nch = reinterpret_cast<int32_t*>(ws + w.nch);
  a.slabs = slabs;
  return cuda_status(launch_sparse_bwd(a, reinterpret_cast<float*>(ws + w.delta),
                                       static_cast<__nv_bfloat16*>(dkv),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

attn_status_t sparse_attn_bwd(const sparse_attn_problem_t* p, const void* q, const void* kv,
                              const int32_t* idx, const void* o, const void* dout,
                              const float* lse, void* dq, void* dkv, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream) {
  return sparse_bwd_call(p, false, q, kv, idx, o, dout, lse, dq, dkv, workspace, workspace_bytes,
                         stream);
}

attn_status_t sparse_attn_bwd_deterministic(const sparse_attn_problem_t* p, const void* q,
                                            const void* kv, const int32_t* idx, const void* o,
                                            const void* dout, const float* lse, void* dq,
                                            void* dkv, void* workspace, size_t workspace_bytes,
                                            attn_stream_t stream) {
  return sparse_bwd_call(p, true, q, kv, idx, o, dout, lse, dq, dkv, workspace, workspace_bytes,
                         stream);
}

}  // extern "C"
