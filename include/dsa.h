/*
 * dsa.h — C ABI of the kernels that surround the sparse attention of the DSA
 * family on GB300 (sm_103a): the lightning indexer (logits, top-k selection,
 * backward), the sparse KL loss that trains it, and the CSA compressor's
 * gated-softmax pooling.
 * Status codes, the stream handle and the device error-word bits are those of
 * attn.h, and every convention listed there holds here too (caller-owned
 * device pointers, no allocation, no host synchronization, every output element
 * written, a status other than ATTN_OK means nothing was enqueued).
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Lightning indexer ("[2/2] Add TileLang fused DSA kernels support with THD and
 * CP & Clean up", Megatron-LM #5049: fused indexer forward with logits
 * cleaning, fused indexer backward returning the gradients of q, k and the
 * weights, top-k returning (topk_indices, topk_length) with -1 sentinels).
 *
 *   logits[t, s] = sum_h w[t, h] * act(<q[t, h], k[s]>)   act = ReLU if use_relu
 *
 * for every key s that query t sees (s <= t within t's sequence); every other
 * entry of the row is written as -inf ("cleaned").
 * Layouts: q bf16 [tokens, heads, 128], k bf16 [tokens, 128], w fp32
 * [tokens, heads], logits fp32 [tokens, logits_ld] (row stride logits_ld, a
 * multiple of 4 and >= tokens; columns past tokens are not written).  THD when
 * cu_seqlens != NULL (device int32 [num_seqs + 1]): tokens at or past
 * cu_seqlens[num_seqs] see no key.  Supported: head_dim 128, 1 <= heads <= 64,
 * 1 <= topk <= 8192 (dsa_topk), tokens * logits_ld < 2^31.
 */
typedef struct {
  int tokens;
  int heads;
  int head_dim;
  int topk;
  int use_relu;
  int logits_ld;
  const int32_t* cu_seqlens; /* optional (THD) */
  int num_seqs;
  int32_t* error_word;       /* optional device int32 */
} dsa_indexer_problem_t;

attn_status_t dsa_indexer_fwd(const dsa_indexer_problem_t* p, const void* q, const void* k,
                              const float* w, float* logits, attn_stream_t stream);

/* Top-k of each logits row over the keys the row's token sees: the
 * min(topk, n_t) largest (ties toward the smaller key index), written in
 * ascending key order to idx int32 [tokens, topk] and padded with -1;
 * length int32 [tokens] = min(topk, n_t) (the compact-prefix form); scores
 * fp32 [tokens, topk] = the selected logits (-inf in padded slots).  A NaN
 * logit ranks below every number. */
attn_status_t dsa_topk(const dsa_indexer_problem_t* p, const float* logits, int32_t* idx,
                       int32_t* length, float* scores, attn_stream_t stream);

/* Workspace bytes of dsa_indexer_bwd: the fp32 dk accumulator [tokens, 128]. */
size_t dsa_indexer_bwd_workspace_size(const dsa_indexer_problem_t* p);

/* Backward of L = sum over valid slots of grad[t, j] * logits[t, idx[t, j]]:
 *   dz = grad[t, j] * w[t, h] * act'(<q[t, h], k[s]>),   s = idx[t, j]
 *   dq[t, h] = sum_j dz k[s];  dk[s] += sum_h dz q[t, h];
 *   dw[t, h] = sum_j grad[t, j] * act(<q[t, h], k[s]>).
 * idx int32 [tokens, topk] (-1 = empty slot; entries outside [-1, tokens) are
 * skipped and flagged ATTN_DEVERR_INDEX_RANGE), grad fp32 [tokens, topk];
 * dq bf16 [tokens, heads, 128], dk bf16 [tokens, 128], dw fp32 [tokens, heads].
 * dk is summed with fp32 atomic adds (not bitwise reproducible). */
attn_status_t dsa_indexer_bwd(const dsa_indexer_problem_t* p, const void* q, const void* k,
                              const float* w, const int32_t* idx, const float* grad, void* dq,
                              void* dk, float* dw, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream);

/*
 * Sparse KL loss of the indexer (the same page's streaming sparse-KL hook; the
 * KL target and normalisation "including all-invalid/empty rows").  With the
 * sparse attention of sparse_attn_fwd (problem `p`, q, kv, its lse, the index
 * lists idx), per token t over its valid slots j:
 *   P[h, j]    = exp(scale <q[t, h], kv[idx[t, j]]> - lse[t, h])
 *   target[j]  = (1 / heads) sum_h P[h, j]
 *   r          = softmax_j(scores[t, j])
 *   loss[t]    = sum_j target[j] (ln target[j] - ln r[j])     (0 ln 0 = 0)
 *   grad[t, j] = r[j] - target[j]      (d loss[t] / d scores[t, j]; 0 in -1 slots)
 * A token without a valid slot gets loss 0.  scores fp32 [tokens, topk] (the
 * indexer's logits at the slots, e.g. dsa_topk's output), loss fp32 [tokens],
 * grad fp32 [tokens, topk], target fp32 [tokens, topk] (optional, may be NULL).
 * The attention probabilities are recomputed chunk by chunk on the tensor cores
 * and reduced over the heads on chip; nothing of size tokens x heads x topk is
 * stored (the per-slot sums wait in `grad`, which the kernel then overwrites).
 * Supported: the sparse_attn_fwd envelope.
 */
attn_status_t dsa_sparse_kl(const sparse_attn_problem_t* p, const void* q, const void* kv,
                            const float* lse, const int32_t* idx, const float* scores,
                            float* loss, float* grad, float* target, attn_stream_t stream);

/* Device error-word bit: a segment's compressed-row count in cu_seqlens_comp
 * differs from floor(length / ratio), or cu_seqlens / cu_seqlens_comp are not
 * non-decreasing within [0, capacity]; the rows of that segment are zero. */
#define ATTN_DEVERR_LAYOUT 0x8

/*
 * CSA compressor gated pooling ("CSA: add fused Compressor forward+backward
 * CuTe-DSL kernels (ported from Megatron-LM)", cudnn-frontend #427, PR
 * description: gather -> + APE -> overlap-window transform (coff == 2) -> fp32
 * softmax over the window -> gated weighted sum -> bf16 cast, THD packed).
 *
 * Segment n holds tokens [cu_seqlens[n], cu_seqlens[n+1]) and compressed rows
 * [cu_seqlens_comp[n], cu_seqlens_comp[n+1]), one row per `ratio` tokens
 * (floor(length / ratio) rows; the remaining tail tokens feed none).  Row c =
 * block b of segment n owns tokens t_r = cu_seqlens[n] + b * ratio + r.
 * For each output dim d its window holds, with D = head_dim:
 *   coff == 1: (kv[t_r, d], score[t_r, d] + ape[r, d]) for r < ratio;
 *   coff == 2: (kv[t_r, D + d], score[t_r, D + d] + ape[r, D + d]) and, when
 *              b > 0, the previous block's (kv[t_r - ratio, d],
 *              score[t_r - ratio, d] + ape[r, d]);
 * and out[c, d] = sum_w softmax_w(score_w) * kv_w, all in fp32, rounded once
 * to bf16.
 *
 * Layouts: kv, score, dkv, dscore bf16 [tokens, coff * head_dim]; ape, dape
 * fp32 [ratio, coff * head_dim]; out, dout bf16 [comp_capacity, head_dim];
 * cu_seqlens and cu_seqlens_comp int32 [num_seqs + 1] in device memory
 * (4-byte aligned; never read by the host, so a captured graph may change
 * them between replays).  `tokens` and `comp_capacity` are the static
 * capacities of the buffers: token rows at or past cu_seqlens[num_seqs] and
 * output rows at or past cu_seqlens_comp[num_seqs] are padding.
 *
 * Supported: head_dim a multiple of 64 up to 1024, ratio in {2, 4, 8},
 * coff in {1, 2}, tokens * coff * head_dim < 2^31.
 */
typedef struct {
  int tokens;        /* rows of kv / score / dkv / dscore */
  int comp_capacity; /* rows of out / dout */
  int num_seqs;
  int head_dim;
  int ratio;
  int coff;
  const int32_t* cu_seqlens;      /* device int32 [num_seqs + 1] */
  const int32_t* cu_seqlens_comp; /* device int32 [num_seqs + 1] */
  int32_t* error_word;            /* optional device int32 */
} csa_compressor_problem_t;

/* Forward: out (bf16); padding rows of out are exact zeros. */
attn_status_t csa_compressor_fwd(const csa_compressor_problem_t* p, const void* kv,
                                 const void* score, const float* ape, void* out,
                                 attn_stream_t stream);

/* Workspace bytes of csa_compressor_bwd: fp32 partial sums of dape, one slab of
 * ratio * coff * head_dim per group of compressed rows. */
size_t csa_compressor_bwd_workspace_size(const csa_compressor_problem_t* p);

/* Backward of L = <out, dout>: dkv = w * dout and dscore = w * dout * (kv - out)
 * at the (token, column) each window entry reads, by disjoint stores; every
 * position no window reads (first-half columns of a segment's last block,
 * tail tokens, segments shorter than ratio, tokens at or past the last
 * segment) gets an exact zero from one owner (the page's backward zero-write
 * commit).  dout rows at or past cu_seqlens_comp[num_seqs] are not read.
 * dape[r, col] sums dscore over all rows: each group of rows writes its
 * partial to the workspace and a second kernel sums the partials in a fixed
 * order, so dkv, dscore and dape are all bitwise run-to-run reproducible (the
 * page accumulates dape with fp32 atomics instead). */
attn_status_t csa_compressor_bwd(const csa_compressor_problem_t* p, const void* kv,
                                 const void* score, const float* ape, const void* dout,
                                 void* dkv, void* dscore, float* dape, void* workspace,
                                 size_t workspace_bytes, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
