/*
 * attn.h — C ABI of the GB300 (sm_103a) softmax-attention training kernels.
 *
 * Operations (the stages named in "[Example] Introduce split+sum template, and
 * optimize atomic_add performance for bwd examples", tile-ai/tilelang #940,
 * code-graph section: forward -> bwd preprocess -> bwd -> postprocess):
 *
 *   attn_fwd              O = softmax(scale * Q K^T) V per head, and the row
 *                         log-sum-exp LSE_i = ln sum_j exp(scale * q_i . k_j).
 *   attn_bwd_preprocess   Delta_i = sum_d dO_id * O_id; clears the fp32 dQ
 *                         accumulator when dq_mode is ATTN_DQ_ATOMIC (the
 *                         order tickets of ATTN_DQ_SPLIT at head_dim 128).
 *   attn_bwd              recomputes P = exp(scale * Q K^T - LSE) tile by tile
 *                         and forms dV = P^T dO, dP = dO V^T,
 *                         dS = P o (dP - Delta), dK = scale dS^T Q,
 *                         dQ = scale dS K.  dQ is accumulated in the workspace
 *                         with fp32 atomics (ATTN_DQ_ATOMIC; #940 description:
 *                         fp32, never bf16, atomics) or in a fixed order
 *                         (ATTN_DQ_SPLIT; #940 "split+sum template"): at
 *                         head_dim 64 as per-KV-tile partial slabs, at
 *                         head_dim 128 added into one accumulator in
 *                         ascending KV-tile order, each query tile's turn
 *                         kept by an int32 ticket.
 *   attn_bwd_postprocess  dQ = bf16(scale * accumulator) or, for the slabs,
 *                         bf16(scale * sum of the partials in ascending
 *                         KV-tile order).
 *   sparse_attn_fwd/bwd   the same with a per-token top-k key list over one
 *                         shared KV head of 576 = 512 + 64 dims, values the
 *                         first 512 dims ("[2/2] Add TileLang fused DSA kernels
 *                         support with THD and CP", Megatron-LM #5049: SparseMLA
 *                         forward/backward, dim 576 / v_channels 512, -1 slots).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *     never allocates, frees or synchronizes.  Work is enqueued on `stream`.
 *   - bf16 tensors are dense row-major in the documented layout with 16-byte
 *     aligned base pointers; fp32 / int32 tensors likewise.
 *   - Outputs may be uninitialized: every element of every output is written.
 *   - A status other than ATTN_OK means nothing was enqueued.  Problems only the
 *     device can see (an index out of range, a wait that ran out) are OR-ed
 *     into the optional device word `error_word` as ATTN_DEVERR_* bits; read it
 *     after the stream completes.
 *   - Flat element offsets must fit in int32 per tensor row index (< 2^31).
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* attn_stream_t; /* same handle as cudaStream_t */

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent shape */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but outside the supported envelope */
  ATTN_ERR_ALIGNMENT = 3,    /* a base pointer is not 16-byte aligned */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  ATTN_ERR_WORKSPACE = 5,    /* workspace missing or smaller than required */
  ATTN_ERR_INDEX_RANGE = 6,  /* reported through the device error word */
  ATTN_ERR_TIMEOUT = 7       /* reported through the device error word */
} attn_status_t;

/* Bits OR-ed into the device error word. */
#define ATTN_DEVERR_INDEX_RANGE 0x1 /* sparse index outside [-1, T) (slot skipped) */
#define ATTN_DEVERR_TIMEOUT 0x2     /* a pipeline wait exceeded its limit */
#define ATTN_DEVERR_SEQLEN 0x4      /* a THD sequence is longer than max_seqlen */

typedef enum {
  ATTN_DQ_ATOMIC = 0, /* fp32 atomic adds into one accumulator (not bitwise reproducible) */
  ATTN_DQ_SPLIT = 1   /* fixed-order dQ sums: bitwise run-to-run identical */
} attn_dq_mode_t;

/*
 * Shape of a dense or THD-packed problem.
 *
 * Dense (cu_seqlens == NULL): Q, O, dO, dQ are [batch, seqlen, heads_q, head_dim]
 * and K, V, dK, dV are [batch, seqlen, heads_kv, head_dim] (BSHD, the layout of
 * the #940 GQA backward, which indexes dK[b, s, h // groups, d]); LSE and Delta
 * are fp32 [batch, heads_q, seqlen].
 *
 * THD (cu_seqlens != NULL): Q/O/dO/dQ are [capacity, heads_q, head_dim], K/V/dK/dV
 * [capacity, heads_kv, head_dim]; sequence n occupies rows
 * [cu_seqlens[n], cu_seqlens[n+1]); cu_seqlens is int32 [num_seqs + 1], device
 * memory, non-decreasing, cu_seqlens[0] = 0, cu_seqlens[num_seqs] <= capacity
 * (read on the device only, so a captured graph may change it between replays).
 * Rows at or past cu_seqlens[num_seqs] are padding: outputs there are written as
 * exact zeros (LSE as -inf); input rows there must hold finite values and do not
 * affect any result.  LSE and Delta are fp32 [heads_q, capacity].
 * `batch` and `seqlen` are ignored; `max_seqlen` bounds every sequence length.
 *
 * Supported: head_dim in {64, 128}; heads_q a multiple of heads_kv; causal
 * masking is top-left aligned (key j visible to query i iff j <= i, within a
 * sequence).  `scale` multiplies the logits (typically 1/sqrt(head_dim)).
 */
typedef struct {
  int batch;
  int seqlen;
  int heads_q;
  int heads_kv;
  int head_dim;
  int causal;
  float scale;
  const int32_t* cu_seqlens; /* NULL for dense BSHD */
  int num_seqs;
  int capacity;
  int max_seqlen;
  int32_t* error_word; /* optional device int32 */
} attn_problem_t;

/* Forward: q, k, v bf16 -> o bf16, lse fp32 (natural log, scale included). */
attn_status_t attn_fwd(const attn_problem_t* p, const void* q, const void* k, const void* v,
                       void* o, float* lse, attn_stream_t stream);

/* Bytes of device workspace attn_bwd_preprocess/attn_bwd need for `mode`:
 * ATOMIC, the fp32 dQ accumulator (batch x heads_q x rows x head_dim);
 * SPLIT at head_dim 64, one such slab per 128-row KV tile of the longest
 * sequence; SPLIT at head_dim 128, the accumulator plus one int32 ticket per
 * (batch, query head, 128-row tile slot).  Returns 0 for an invalid problem. */
size_t attn_bwd_workspace_size(const attn_problem_t* p, attn_dq_mode_t mode);

/* Backward preprocess: delta fp32 (same layout as lse) = rowsum(dO * O).
 * In ATOMIC mode it also clears the dQ accumulator inside `workspace` (SPLIT at
 * head_dim 128: the tickets), so it must run before attn_bwd with the same
 * workspace and mode. */
attn_status_t attn_bwd_preprocess(const attn_problem_t* p, attn_dq_mode_t mode, const void* o,
                                  const void* dout, float* delta, void* workspace,
                                  size_t workspace_bytes, attn_stream_t stream);

/* Backward main pass: q, k, v, dout bf16; lse, delta fp32 (from attn_fwd and
 * attn_bwd_preprocess) -> dk, dv bf16 (every non-padding row; for THD the
 * padding rows too, as exact zeros) and the fp32 dQ
 * accumulator or partials inside `workspace`.  GQA dK/dV are summed over each
 * KV head's query heads inside the kernel (no atomics on dK/dV).  Must be
 * followed by attn_bwd_postprocess with the same workspace and mode. */
attn_status_t attn_bwd(const attn_problem_t* p, attn_dq_mode_t mode, const void* q,
                       const void* k, const void* v, const void* dout, const float* lse,
                       const float* delta, void* dk, void* dv, void* workspace,
                       size_t workspace_bytes, attn_stream_t stream);

/* Backward postprocess: dq bf16 from the workspace of attn_bwd; for THD it also
 * writes the padding rows (at or past cu_seqlens[num_seqs]) of dq as exact
 * zeros (attn_bwd wrote those of dk and dv).  After it, every element of dq,
 * dk and dv has been written. */
attn_status_t attn_bwd_postprocess(const attn_problem_t* p, attn_dq_mode_t mode,
                                   const void* workspace, size_t workspace_bytes, void* dq,
                                   void* dk, void* dv, attn_stream_t stream);

/*
 * Backward without any caller-provided device memory.  The source pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory at all -- for example a plugin running inside a host framework that
 * owns every device allocation through its own pool, or a latency-critical loop
 * where cudaMalloc (which may synchronize the device) is not allowed -- and so
 * cannot provide the workspace that attn_bwd_preprocess / attn_bwd /
 * attn_bwd_postprocess need.
 *
 * It runs those three stages in ATTN_DQ_ATOMIC mode, with Delta and the fp32 dQ
 * accumulator kept in one static device array of ATTN_FIXED_SCRATCH_BYTES that
 * the library owns; every GPU that loads the library holds that array until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Inputs: q, k, v, o, dout bf16 and lse fp32 (from attn_fwd); outputs dq, dk,
 *     dv bf16 -- all caller-owned device pointers, layouts as in attn_problem_t.
 *   - Capacity: rows * heads_q * (head_dim + 1) * 4 bytes (plus 256 bytes of
 *     alignment) must fit in ATTN_FIXED_SCRATCH_BYTES, with rows = batch * seqlen
 *     (dense) or capacity (THD); larger problems return ATTN_ERR_UNSUPPORTED and
 *     enqueue nothing.
 *   - Set-up: the first call on each device looks up the array's device address
 *     (with that device current) and caches it with the id of the current
 *     context, so make that first call before any stream capture; later calls
 *     only read the cache.  After a device reset (a new primary context) the
 *     next call looks the address up again, which also must not happen under
 *     capture.  Calls must be made with the device that owns `stream` current.
 *   - Validation: the problem is checked exactly as attn_bwd checks it before any
 *     scratch size is computed; invalid problems return that status.
 *   - Sharing: every call uses the same array and leaves its contents behind; the
 *     call clears what must start at zero itself.  Calls whose work overlaps on
 *     the GPU (for example on two streams) race on the array and give wrong
 *     results; serialize them.
 */
#define ATTN_FIXED_SCRATCH_BYTES (16u << 20)

attn_status_t attn_bwd_fixed_scratch(const attn_problem_t* p, const void* q, const void* k,
                                     const void* v, const void* o, const void* dout,
                                     const float* lse, void* dq, void* dk, void* dv,
                                     attn_stream_t stream);

/*
 * Top-k sparse attention over one shared KV head (SparseMLA style).
 * q [tokens, heads, dim_qk] bf16, kv [tokens, dim_qk] bf16 (the key is the whole
 * row; the value is its first dim_v entries), idx int32 [tokens, topk]: token t
 * attends to the rows listed in idx[t]; -1 marks an empty slot; entries must be
 * distinct.  Entries outside [-1, tokens) are skipped and flagged with
 * ATTN_DEVERR_INDEX_RANGE.  o / dout [tokens, heads, dim_v] bf16, lse
 * [tokens, heads] fp32.  A token with no valid slot gets o = 0, lse = -inf.
 * Supported: dim_qk = 576, dim_v = 512, heads in {16, 32, 64, 128}, bf16.
 */
typedef struct {
  int tokens;
  int heads;
  int dim_qk;
  int dim_v;
  int topk;
  float scale;
  int32_t* error_word; /* optional device int32 */
} sparse_attn_problem_t;

attn_status_t sparse_attn_fwd(const sparse_attn_problem_t* p, const void* q, const void* kv,
                              const int32_t* idx, void* o, float* lse, attn_stream_t stream);

/* Workspace bytes for sparse_attn_bwd: fp32 dKV accumulator [tokens, dim_qk],
 * fp32 Delta [tokens, heads] and int32 chunk counts [tokens], each 256-byte
 * aligned. */
size_t sparse_attn_bwd_workspace_size(const sparse_attn_problem_t* p);

/* Backward: dq [tokens, heads, dim_qk] bf16, dkv [tokens, dim_qk] bf16.  Runs the
 * preprocess (Delta, the number of 64-slot chunks up to each token's last
 * valid slot, clearing the accumulator), the main kernel (dQ by disjoint
 * stores, dKV by fp32 atomic adds, so dKV is not bitwise reproducible) and the
 * fp32 -> bf16 cast of dKV. */
attn_status_t sparse_attn_bwd(const sparse_attn_problem_t* p, const void* q, const void* kv,
                              const int32_t* idx, const void* o, const void* dout,
                              const float* lse, void* dq, void* dkv, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream);

/* Deterministic variant of sparse_attn_bwd: the same dq (bitwise) and dkv
 * within rounding, with dkv bitwise reproducible.  The main kernel runs
 * min(152, tokens * ceil(heads / 64)) CTAs; CTA b takes the (token, 64-head
 * block) items b, b + grid, ... in that order and adds its dKV contributions
 * into its own fp32 [tokens, dim_qk] slab of the workspace.  A token names a
 * key row at most once, so an item adds at most once into each slab address,
 * and the CTA orders its items' adds (a fence and a barrier between items):
 * every slab address receives its adds in a fixed order.  The slabs are then
 * summed in slab order and cast to bf16.  The slab count does not depend on the
 * device, so neither does the result.  Index lists that name a key row twice
 * break the contract (the two adds of that item then meet in either order).
 * Workspace: slabs * tokens * dim_qk fp32 plus Delta and the chunk counts (the
 * slabs are cleared by the call); at tokens 8192, 64 heads 2.87 GB for any
 * topk. */
size_t sparse_attn_bwd_deterministic_workspace_size(const sparse_attn_problem_t* p);
attn_status_t sparse_attn_bwd_deterministic(const sparse_attn_problem_t* p, const void* q,
                                            const void* kv, const int32_t* idx, const void* o,
                                            const void* dout, const float* lse, void* dq,
                                            void* dkv, void* workspace, size_t workspace_bytes,
                                            attn_stream_t stream);

/* Self-test of the bounded waits of the library's kernels (one CTA, two roles
 * holding a TMEM allocation): one role waits on an mbarrier that never
 * completes, with a limit of limit_us microseconds (1 .. 1e6), the other on a
 * second such barrier with the kernels' own limit.  The first wait must run out
 * and OR ATTN_DEVERR_TIMEOUT into *error_word (device int32); the second must
 * then stop on the CTA's abort flag; the CTA frees its TMEM and exits.  *result
 * (device int32) gets bit 0 when the first wait ran out, bit 1 when the second
 * stopped and bit 2 when it stopped well before its own limit: 7 when the
 * mechanism works.  Nothing faults or hangs either way. */
attn_status_t attn_wait_selftest(int32_t* error_word, unsigned limit_us, int32_t* result,
                                 attn_stream_t stream);

/* Static description of a status code. */
const char* attn_status_string(attn_status_t s);

/* Library version as major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
