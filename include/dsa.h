/*
 * dsa.h — C ABI of the kernels that surround the sparse attention of the DSA
 * family on GB300 (sm_103a): the CSA compressor's gated-softmax pooling.
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
