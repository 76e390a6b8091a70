"""fp64 CPU oracle of the DSA lightning indexer, its top-k selection and the
sparse KL loss that trains it.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module: only
the tests, the smoke check and the CPU-baseline leg of the benchmark do.  It
shares no code with the CUDA kernels.

Source: "[2/2] Add TileLang fused DSA kernels support with THD and CP & Clean up"
(Megatron-LM #5049): file table (fused indexer forward kernel with logits
cleaning, fused indexer backward, top-k / SparseMLA / streaming sparse-KL hooks),
review thread (the indexer's `use_relu` switch; IndexerFunction.backward returns
gradients for q, k and the weights; run_fused_qk_topk returns (topk_indices,
topk_length), -1 sentinels or a compact prefix of length topk_length; top-k slots
sorted by key index; the KL target normalisation "including all-invalid/empty
rows").  The page names these steps but prints no formula; what follows is the
reading taken, written out with plain fp64 loops and products.

Indexer logits, per query token t and key token s (one shared key per token,
H index heads per query):

    I[t, s] = sum_h w[t, h] * act(<q[t, h], k[s]>),   act = ReLU (use_relu) or identity

for the keys t may see: s <= t within t's sequence (THD: cu_seqlens); every
other entry is "cleaned" to -inf.

Top-k: the min(topk, n_t) keys of largest I[t, .] among the n_t keys t sees, ties
broken toward the smaller key index, listed in ascending key order and padded
with -1; topk_length[t] = min(topk, n_t) (the compact-prefix form); the scores
are I[t, idx] (-inf in padded slots).

Indexer backward of L = sum_{t, j valid} g[t, j] * I[t, idx[t, j]]:

    dz[t, h, j] = g[t, j] * w[t, h] * act'(z),   z = <q[t, h], k[idx[t, j]]>
    dq[t, h]  = sum_j dz[t, h, j] k[idx[t, j]]
    dk[s]    += sum_h dz[t, h, j] q[t, h]      for s = idx[t, j]
    dw[t, h]  = sum_j g[t, j] act(z)

Sparse KL loss (the indexer's training signal): with the sparse attention's
probabilities P[t, h, j] = exp(scale <q_a[t, h], kv[idx[t, j]]> - lse[t, h]) over
the token's valid slots, the target is p[t, j] = (1/H) sum_h P[t, h, j] (each
head's row sums to 1, so p does), the indexer's distribution is
r[t, .] = softmax of the scores over the valid slots, and

    loss[t] = sum_j p[t, j] (ln p[t, j] - ln r[t, j])      (0 ln 0 = 0; 0 for a
                                                           token with no slot)
    d loss[t] / d score[t, j] = r[t, j] - p[t, j]          (0 for -1 slots)
"""
from __future__ import annotations

import torch

F64 = torch.float64
NEG_INF = float("-inf")


def _f64(x):
    return x.detach().to("cpu", F64)


def visible_keys(T, cu_seqlens=None):
    """[T, T] bool: key s visible to query t (s <= t, same sequence)."""
    t = torch.arange(T)[:, None]
    s = torch.arange(T)[None, :]
    vis = s <= t
    if cu_seqlens is not None:
        seq = torch.full((T,), -1, dtype=torch.long)
        cu = [int(x) for x in cu_seqlens.tolist()]
        for n in range(len(cu) - 1):
            seq[cu[n]:cu[n + 1]] = n
        vis = vis & (seq[:, None] == seq[None, :]) & (seq[:, None] >= 0)
    return vis


def indexer_logits(q, k, w, cu_seqlens=None, use_relu=True):
    """q [T,H,D], k [T,D], w [T,H] -> I [T,T] fp64 with -inf where not visible."""
    q, k, w = _f64(q), _f64(k), _f64(w)
    T, H, _ = q.shape
    out = torch.zeros(T, T, dtype=F64)
    for h in range(H):
        z = q[:, h, :] @ k.T                       # [T, T]
        if use_relu:
            z = torch.clamp(z, min=0.0)
        out += w[:, h:h + 1] * z
    vis = visible_keys(T, cu_seqlens)
    return torch.where(vis, out, torch.full_like(out, NEG_INF))


def indexer_logits_rows(q, k, w, rows, cu_seqlens=None, use_relu=True):
    """Rows `rows` of indexer_logits only ([len(rows), T]): the same sums for
    the listed query tokens (each row is independent of the others)."""
    q, k, w = _f64(q), _f64(k), _f64(w)
    T, H, _ = q.shape
    rows = [int(r) for r in rows]
    out = torch.zeros(len(rows), T, dtype=F64)
    for n, t in enumerate(rows):
        z = q[t] @ k.T                              # [H, T]
        if use_relu:
            z = torch.clamp(z, min=0.0)
        out[n] = (w[t][:, None] * z).sum(0)
    vis = visible_keys(T, cu_seqlens)[rows]
    return torch.where(vis, out, torch.full_like(out, NEG_INF)), vis


def topk_select(logits, topk, visible):
    """Per row: the min(topk, n) visible keys of largest logit, ties toward the
    smaller index, in ascending index order.  Returns idx int32 [T, topk] (-1
    padded), length int32 [T], scores fp64 [T, topk] (-inf padded)."""
    T = logits.shape[0]
    idx = torch.full((T, topk), -1, dtype=torch.int32)
    length = torch.zeros(T, dtype=torch.int32)
    scores = torch.full((T, topk), NEG_INF, dtype=F64)
    for t in range(T):
        cand = [s for s in range(logits.shape[1]) if visible[t, s]]
        # order: larger logit first, then smaller key index
        cand.sort(key=lambda s: (-float(logits[t, s]), s))
        pick = sorted(cand[:topk])
        n = len(pick)
        length[t] = n
        if n:
            idx[t, :n] = torch.tensor(pick, dtype=torch.int32)
            scores[t, :n] = logits[t, pick]
    return idx, length, scores


def indexer_backward(q, k, w, idx, grad, use_relu=True, tokens=None):
    """Gradients of L = sum_{t, j valid} grad[t, j] * I[t, idx[t, j]].  With
    `tokens`, only those query tokens contribute (dq and dw of other tokens
    stay zero, dk holds only their share)."""
    q, k, w, grad = _f64(q), _f64(k), _f64(w), _f64(grad)
    T, H, D = q.shape
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dw = torch.zeros_like(w)
    for t in (range(T) if tokens is None else tokens):
        sel = [(j, int(s)) for j, s in enumerate(idx[t].tolist()) if 0 <= s < k.shape[0]]
        if not sel:
            continue
        js = torch.tensor([j for j, _ in sel])
        ss = torch.tensor([s for _, s in sel])
        ks = k[ss]                                 # [n, D]
        g = grad[t, js]                            # [n]
        z = q[t] @ ks.T                            # [H, n]
        act = torch.clamp(z, min=0.0) if use_relu else z
        der = (z > 0).to(F64) if use_relu else torch.ones_like(z)
        dz = g[None, :] * w[t][:, None] * der      # [H, n]
        dq[t] = dz @ ks
        dk.index_add_(0, ss, dz.T @ q[t])
        dw[t] = act @ g
    return dict(dq=dq, dk=dk, dw=dw)


def indexer_dk_rows(q, k, w, idx, grad, rows, use_relu=True):
    """dk of a few key rows only: the contributions of every token whose list
    names the row (equal to indexer_backward(...)["dk"][rows])."""
    rows = [int(r) for r in rows]
    want = torch.tensor(rows, dtype=idx.dtype)
    hit = (idx[:, :, None] == want[None, None, :]).any(dim=1).any(dim=1)
    toks = torch.nonzero(hit).flatten().tolist()
    return indexer_backward(q, k, w, idx, grad, use_relu, tokens=toks)["dk"][rows]


def attention_target(q, kv, idx, scale, tokens=None):
    """p [T, K] fp64: the sparse attention probabilities of each slot averaged
    over the heads (0 in -1 slots), from the exact fp64 softmax of every head.
    With `tokens`, only those rows are computed (the others stay zero)."""
    q, kv = _f64(q), _f64(kv)
    T, H, _ = q.shape
    p = torch.zeros(idx.shape, dtype=F64)
    for t in (range(T) if tokens is None else tokens):
        js = [j for j, s in enumerate(idx[t].tolist()) if 0 <= s < kv.shape[0]]
        if not js:
            continue
        ss = idx[t, js].to(torch.long)
        s = scale * (q[t] @ kv[ss].T)              # [H, n]
        prob = torch.softmax(s, dim=1)
        p[t, js] = prob.mean(dim=0)
    return p


def sparse_kl(target, scores, idx):
    """loss [T] and d loss / d scores [T, K] for the KL of the target from the
    softmax of the scores over each token's valid slots."""
    target, scores = _f64(target), _f64(scores)
    T, K = scores.shape
    loss = torch.zeros(T, dtype=F64)
    grad = torch.zeros(T, K, dtype=F64)
    for t in range(T):
        js = [j for j in range(K) if int(idx[t, j]) >= 0]
        if not js:
            continue
        r = torch.softmax(scores[t, js], dim=0)
        p = target[t, js]
        terms = torch.where(p > 0, p * (torch.log(torch.where(p > 0, p, torch.ones_like(p)))
                                        - torch.log(r)), torch.zeros_like(p))
        loss[t] = terms.sum()
        grad[t, js] = r - p
    return loss, grad
