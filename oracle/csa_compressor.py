"""fp64 CPU oracle of the CSA compressor's gated-softmax pooling, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module: only
the tests, the smoke check and the CPU-baseline leg of the benchmark do.  It
shares no code with the CUDA kernels.

Source: "CSA: add fused Compressor forward+backward CuTe-DSL kernels (ported from
Megatron-LM)" (cudnn-frontend #427), PR description ("What") and the backward
zero-write commit.  The fused region is: gather -> + APE -> overlap-window
transform (coff == 2) -> fp32 softmax over the window -> gated weighted sum ->
bf16 cast, over THD-packed segments, one compressed row per `ratio` tokens.

What is computed (the reading written out; the page names the steps, not the
formulas).  Segment n holds tokens [cu[n], cu[n+1]) and compressed rows
[cu_comp[n], cu_comp[n+1]), with cu_comp[n+1] - cu_comp[n] = floor(len_n / ratio).
kv and score are [tokens, coff * D]; ape is [ratio, coff * D]; out is [rows, D].
Compressed row c = block b of segment n owns the tokens t_r = cu[n] + b*ratio + r,
r = 0..ratio-1.  Its window, per output dim d:

  coff == 1:  ratio entries       (kv[t_r, d],  score[t_r, d] + ape[r, d])
  coff == 2:  2*ratio entries     own part  (kv[t_r, D + d], score[t_r, D + d] + ape[r, D + d])
                                  prev part (kv[u_r, d],     score[u_r, d]     + ape[r, d])
              with u_r = t_r - ratio, the previous block's tokens; the prev part
              is empty for the first block of a segment (its scores are -inf).

  w = softmax over the window of the scores (per d);  out[c, d] = sum_w w * kv_w.

Every (token, column) feeds at most one window entry: the first-half columns of
block b's tokens feed block b+1's prev part, the second half its own part.  The
backward of L = <out, dout> per window entry is

  dkv_w = w * dout[c, d],   dscore_w = w * dout[c, d] * (kv_w - out[c, d]),

scattered back to the entry's (token, column); dape[r, col] sums dscore over
every row.  Positions no window reads (the first-half columns of a segment's
last block, the tokens past the last whole block, segments shorter than ratio,
tokens at or past cu[-1]) get exact zeros, as do output rows at or past
cu_comp[-1] ("backward zero-write" commit: a unique owner writes every slot).
"""
from __future__ import annotations

import torch

F64 = torch.float64


def _f64(x):
    return x.detach().to("cpu", F64)


def comp_lengths(cu_seqlens, ratio):
    """Compressed rows per segment: floor(len / ratio)."""
    cu = [int(x) for x in cu_seqlens.tolist()]
    return [(cu[n + 1] - cu[n]) // ratio for n in range(len(cu) - 1)]


def window(n_tok0, b, r_count, ratio, coff, head_dim):
    """The window of block b of a segment starting at token n_tok0: a list of
    (token, column offset, position r) for every entry; columns are
    offset + d for d in [0, head_dim)."""
    t0 = n_tok0 + b * ratio
    if coff == 1:
        return [(t0 + r, 0, r) for r in range(r_count)]
    own = [(t0 + r, head_dim, r) for r in range(r_count)]
    prev = [] if b == 0 else [(t0 - ratio + r, 0, r) for r in range(r_count)]
    return own + prev


def _rows(cu_seqlens, cu_comp, ratio):
    cu = [int(x) for x in cu_seqlens.tolist()]
    cc = [int(x) for x in cu_comp.tolist()]
    for n in range(len(cu) - 1):
        nb = cc[n + 1] - cc[n]
        if nb != (cu[n + 1] - cu[n]) // ratio:
            raise ValueError(f"segment {n}: {nb} compressed rows for {cu[n + 1] - cu[n]} tokens")
        for b in range(nb):
            yield cc[n] + b, cu[n], b


def compressor_forward(kv, score, ape, cu_seqlens, cu_comp, ratio, coff, comp_capacity):
    """out [comp_capacity, D] fp64 (rows at or past cu_comp[-1] are zero) and the
    window weights per row (dict c -> (entries, w [len, D]))."""
    kv, score, ape = _f64(kv), _f64(score), _f64(ape)
    D = kv.shape[1] // coff
    out = torch.zeros(comp_capacity, D, dtype=F64)
    weights = {}
    for c, t0, b in _rows(cu_seqlens, cu_comp, ratio):
        ent = window(t0, b, ratio, ratio, coff, D)
        s = torch.stack([score[t, off:off + D] + ape[r, off:off + D] for t, off, r in ent])
        v = torch.stack([kv[t, off:off + D] for t, off, r in ent])
        w = torch.softmax(s, dim=0)                 # over the window, per dim
        out[c] = (w * v).sum(dim=0)
        weights[c] = (ent, w)
    return out, weights


def compressor_backward(kv, score, ape, dout, cu_seqlens, cu_comp, ratio, coff, comp_capacity):
    """Returns dict(out, dkv [T, coff*D], dscore [T, coff*D], dape [ratio, coff*D])."""
    kv, dout = _f64(kv), _f64(dout)
    D = kv.shape[1] // coff
    out, weights = compressor_forward(kv, score, ape, cu_seqlens, cu_comp, ratio, coff,
                                      comp_capacity)
    dkv = torch.zeros_like(kv)
    dscore = torch.zeros_like(kv)
    dape = torch.zeros(ratio, coff * D, dtype=F64)
    for c, (ent, w) in weights.items():
        g = dout[c]
        for i, (t, off, r) in enumerate(ent):
            v = kv[t, off:off + D]
            ds = w[i] * g * (v - out[c])
            dkv[t, off:off + D] = w[i] * g
            dscore[t, off:off + D] = ds
            dape[r, off:off + D] += ds
    return dict(out=out, dkv=dkv, dscore=dscore, dape=dape)


def consumed_mask(tokens, cu_seqlens, ratio, coff, head_dim):
    """bool [tokens, coff] : True where (token, column half) feeds some window."""
    cu = [int(x) for x in cu_seqlens.tolist()]
    m = torch.zeros(tokens, coff, dtype=torch.bool)
    for n in range(len(cu) - 1):
        nb = (cu[n + 1] - cu[n]) // ratio
        for b in range(nb):
            for t, off, r in window(cu[n], b, ratio, ratio, coff, head_dim):
                m[t, off // head_dim] = True
    return m
