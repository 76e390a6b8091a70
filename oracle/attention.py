"""fp64 CPU oracle for softmax attention: forward with row log-sum-exp, and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module: only
the tests, the smoke check and the CPU-baseline leg of the benchmark do.  It
shares no code with the CUDA kernels.

What is computed, per batch b and query head h (kv head g = h // (Hq/Hkv), the
head mapping of the GQA backward in "[Example] Introduce split+sum template, and
optimize atomic_add performance for bwd examples" (tile-ai/tilelang #940), review
comment "Guard dK atomics on tail blocks", where dK is indexed by bx // groups):

    s_ij   = scale * <q_i, k_j>              for allowed (i, j), else -inf
    lse_i  = ln sum_j exp(s_ij)              (natural log, scale included)
    p_ij   = exp(s_ij - lse_i)
    o_i    = sum_j p_ij v_j
    delta_i = <do_i, o_i>                    (the "bwd preprocess" stage of #940)
    dp_ij  = <do_i, v_j>
    ds_ij  = p_ij (dp_ij - delta_i)
    dv_j   = sum_i p_ij do_i
    dk_j   = scale sum_i ds_ij q_i
    dq_i   = scale sum_j ds_ij k_j

The pages name the stages (preprocess -> backward -> postprocess, #940 code-graph
section) but do not print these formulas; they are the textbook derivative of
softmax attention, written out here with plain fp64 matrix products and no
blocking, fusion or online rescaling.  GQA sums dK/dV over the query heads of a
group.  Allowed pairs: every (i, j) when non-causal; j <= i when causal
(top-left aligned, equal lengths); THD packing restricts pairs to one sequence
("[2/2] Add TileLang fused DSA kernels support with THD and CP" (Megatron-LM
#5049), packed-THD discussion).  A row with no allowed key gets lse = -inf,
o = 0 and zero gradients.  THD rows at or past cu_seqlens[-1] are padding: their
O and gradients are exact zeros and their LSE is -inf (the exact-zero contract of
"CSA: add fused Compressor forward+backward CuTe-DSL kernels" (cudnn-frontend
#427), backward zero-write commit, tokens beyond cu_seqlens[-1]).

Sparse (SparseMLA style, Megatron-LM #5049, support envelope and -1 sentinel
discussion): one KV head of 576 = 512 + 64 dims; token t attends the keys listed
in idx[t] (int32, -1 = empty slot); keys use all 576 dims, values the first 512.
dKV[:, :576] collects scale * ds^T q and dKV[:, :512] additionally p^T do.
"""
from __future__ import annotations

import torch

F64 = torch.float64
NEG_INF = float("-inf")


def _f64(x):
    return x.detach().to("cpu", F64)


# ----------------------------------------------------------------------------
# One (query rows x key rows) block with an explicit boolean mask
# ----------------------------------------------------------------------------
def head_forward(q, k, v, scale, allowed):
    """q [Sq,D], k [Sk,D], v [Sk,Dv], allowed [Sq,Sk] bool -> o [Sq,Dv], lse [Sq]."""
    s = scale * (q @ k.T)
    s = torch.where(allowed, s, torch.full_like(s, NEG_INF))
    if s.shape[1] == 0:                             # no key at all: the empty sum
        m = torch.full((s.shape[0], 1), NEG_INF, dtype=s.dtype)
    else:
        m = s.max(dim=1, keepdim=True).values
    has = torch.isfinite(m)
    m_safe = torch.where(has, m, torch.zeros_like(m))
    e = torch.exp(s - m_safe)                       # exp(-inf) = 0 for masked pairs
    z = e.sum(dim=1, keepdim=True)
    lse = torch.where(has, m_safe + torch.log(z), torch.full_like(m, NEG_INF))
    p = torch.where(has, e / torch.where(has, z, torch.ones_like(z)), torch.zeros_like(e))
    o = p @ v
    return o, lse.squeeze(1), p


def head_backward(q, k, v, do, scale, allowed):
    """Full forward + backward of one block; returns a dict of fp64 tensors."""
    o, lse, p = head_forward(q, k, v, scale, allowed)
    delta = (do * o).sum(dim=1)                     # [Sq]
    dp = do @ v.T                                   # [Sq,Sk]
    ds = p * (dp - delta[:, None])
    dv = p.T @ do
    dk = scale * (ds.T @ q)
    dq = scale * (ds @ k)
    return dict(o=o, lse=lse, p=p, dp=dp, ds=ds, delta=delta, dq=dq, dk=dk, dv=dv)


def causal_mask(sq: int, sk: int):
    i = torch.arange(sq)[:, None]
    j = torch.arange(sk)[None, :]
    return j <= i


def full_mask(sq: int, sk: int):
    return torch.ones(sq, sk, dtype=torch.bool)


# ----------------------------------------------------------------------------
# Dense BSHD
# ----------------------------------------------------------------------------
def _group(hq: int, hkv: int) -> int:
    if hq % hkv:
        raise ValueError("heads_q must be a multiple of heads_kv")
    return hq // hkv


def dense_forward(q, k, v, scale, causal, heads=None):
    """q [B,S,Hq,D], k/v [B,S,Hkv,D] -> o [B,S,Hq,D] fp64, lse [B,Hq,S] fp64.

    ``heads`` optionally restricts the computation to a list of (b, h) pairs;
    other entries stay NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    grp = _group(Hq, Hkv)
    o = torch.full((B, S, Hq, v.shape[3]), float("nan"), dtype=F64)
    lse = torch.full((B, Hq, S), float("nan"), dtype=F64)
    mask = causal_mask(S, Sk) if causal else full_mask(S, Sk)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in pairs:
        g = h // grp
        ob, lb, _ = head_forward(q[b, :, h], k[b, :, g], v[b, :, g], scale, mask)
        o[b, :, h] = ob
        lse[b, h] = lb
    return o, lse


def dense_backward(q, k, v, do, scale, causal, kv_heads=None):
    """Returns dict(o, lse, delta, dq, dk, dv) in fp64.

    ``kv_heads`` optionally restricts the work to a list of (b, g) kv-head units
    (each unit is independent: its query heads, their dQ and its own dK/dV);
    entries outside the listed units stay NaN."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, S, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    grp = _group(Hq, Hkv)
    nan = float("nan")
    out = dict(o=torch.full_like(do, nan), lse=torch.full((B, Hq, S), nan, dtype=F64),
               delta=torch.full((B, Hq, S), nan, dtype=F64), dq=torch.full_like(q, nan),
               dk=torch.full_like(k, nan), dv=torch.full_like(v, nan))
    mask = causal_mask(S, Sk) if causal else full_mask(S, Sk)
    units = kv_heads if kv_heads is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for b, g in units:
        dk = torch.zeros_like(k[b, :, g])
        dv = torch.zeros_like(v[b, :, g])
        for h in range(g * grp, (g + 1) * grp):
            r = head_backward(q[b, :, h], k[b, :, g], v[b, :, g], do[b, :, h], scale, mask)
            out["o"][b, :, h] = r["o"]
            out["lse"][b, h] = r["lse"]
            out["delta"][b, h] = r["delta"]
            out["dq"][b, :, h] = r["dq"]
            dk += r["dk"]
            dv += r["dv"]
        out["dk"][b, :, g] = dk
        out["dv"][b, :, g] = dv
    return out


# ----------------------------------------------------------------------------
# THD packed variable length
# ----------------------------------------------------------------------------
def thd_backward(q, k, v, do, cu_seqlens, scale, causal, seqs=None):
    """q/do [cap,Hq,D], k/v [cap,Hkv,D], cu_seqlens int32 [n+1].

    Returns dict(o, lse [Hq,cap], delta [Hq,cap], dq, dk, dv) in fp64.  Rows at
    or past cu_seqlens[-1] come out as exact zeros (lse -inf, delta 0).
    ``seqs`` optionally restricts the work to some sequences (others stay NaN
    except the padding rows)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cap, Hq, D = q.shape
    Hkv = k.shape[1]
    grp = _group(Hq, Hkv)
    cu = [int(x) for x in cu_seqlens.tolist()]
    nan = float("nan")
    out = dict(o=torch.full_like(do, nan), lse=torch.full((Hq, cap), nan, dtype=F64),
               delta=torch.full((Hq, cap), nan, dtype=F64), dq=torch.full_like(q, nan),
               dk=torch.full_like(k, nan), dv=torch.full_like(v, nan))
    end = cu[-1]
    for key in ("o", "dq", "dk", "dv"):
        out[key][end:] = 0.0
    out["lse"][:, end:] = NEG_INF
    out["delta"][:, end:] = 0.0
    todo = seqs if seqs is not None else range(len(cu) - 1)
    for n in todo:
        a, e = cu[n], cu[n + 1]
        L = e - a
        if L == 0:
            continue
        mask = causal_mask(L, L) if causal else full_mask(L, L)
        for g in range(Hkv):
            dk = torch.zeros(L, D, dtype=F64)
            dv = torch.zeros(L, v.shape[2], dtype=F64)
            for h in range(g * grp, (g + 1) * grp):
                r = head_backward(q[a:e, h], k[a:e, g], v[a:e, g], do[a:e, h], scale, mask)
                out["o"][a:e, h] = r["o"]
                out["lse"][h, a:e] = r["lse"]
                out["delta"][h, a:e] = r["delta"]
                out["dq"][a:e, h] = r["dq"]
                dk += r["dk"]
                dv += r["dv"]
            out["dk"][a:e, g] = dk
            out["dv"][a:e, g] = dv
    return out


# ----------------------------------------------------------------------------
# Top-k sparse, one shared KV head (keys 576 dims, values the first 512)
# ----------------------------------------------------------------------------
def sparse_valid(idx_row):
    """Selected key rows of one token: entries >= 0 (-1 marks an empty slot)."""
    return idx_row[idx_row >= 0].to(torch.long)


def sparse_token(q_t, kv, idx_row, do_t, scale, dv_dims=512):
    """One token: q_t [H,576], kv [T,576], idx_row [K], do_t [H,512] (or None).

    Returns dict(o [H,512], lse [H], and when do_t is given delta, dq [H,576],
    rows (selected key rows), dkv_rows [n,576])."""
    sel = sparse_valid(idx_row)
    kt = kv[sel]                                    # [n,576]
    vt = kt[:, :dv_dims]                            # [n,512]
    allowed = torch.ones(q_t.shape[0], sel.numel(), dtype=torch.bool)
    if do_t is None:
        o, lse, _ = head_forward(q_t, kt, vt, scale, allowed)
        return dict(o=o, lse=lse, rows=sel)
    r = head_backward(q_t, kt, vt, do_t, scale, allowed)
    dkv_rows = r["dk"].clone()
    dkv_rows[:, :dv_dims] += r["dv"]
    return dict(o=r["o"], lse=r["lse"], delta=r["delta"], dq=r["dq"], rows=sel,
                dkv_rows=dkv_rows)


def sparse_forward(q, kv, idx, scale, tokens=None, dv_dims=512):
    q, kv = _f64(q), _f64(kv)
    T, H, _ = q.shape
    o = torch.full((T, H, dv_dims), float("nan"), dtype=F64)
    lse = torch.full((T, H), float("nan"), dtype=F64)
    for t in (tokens if tokens is not None else range(T)):
        r = sparse_token(q[t], kv, idx[t], None, scale, dv_dims)
        o[t], lse[t] = r["o"], r["lse"]
    return o, lse


def sparse_backward(q, kv, idx, do, scale, dv_dims=512):
    """Full sparse forward + backward; dkv [T,576] accumulates over all tokens."""
    q, kv, do = _f64(q), _f64(kv), _f64(do)
    T, H, _ = q.shape
    o = torch.zeros(T, H, dv_dims, dtype=F64)
    lse = torch.zeros(T, H, dtype=F64)
    delta = torch.zeros(T, H, dtype=F64)
    dq = torch.zeros_like(q)
    dkv = torch.zeros_like(kv)
    for t in range(T):
        r = sparse_token(q[t], kv, idx[t], do[t], scale, dv_dims)
        o[t], lse[t], delta[t], dq[t] = r["o"], r["lse"], r["delta"], r["dq"]
        dkv.index_add_(0, r["rows"], r["dkv_rows"])
    return dict(o=o, lse=lse, delta=delta, dq=dq, dkv=dkv)


def sparse_dkv_rows(q, kv, idx, do, scale, rows, dv_dims=512):
    """dKV for a few key rows only: sums the contributions of every token whose
    index list holds the row (exact, independent of the other rows).  Equal to
    ``sparse_backward(...)["dkv"][rows]``; a row that no token names is zero."""
    q, kv, do = _f64(q), _f64(kv), _f64(do)
    rows = [int(r) for r in rows]
    want = torch.tensor(rows, dtype=idx.dtype)
    hit = (idx[:, :, None] == want[None, None, :]).any(dim=1)      # [T, len(rows)]
    out = torch.zeros(len(rows), kv.shape[1], dtype=F64)
    tok = torch.nonzero(hit.any(dim=1)).flatten().tolist()
    for t in tok:
        r = sparse_token(q[t], kv, idx[t], do[t], scale, dv_dims)
        sel = r["rows"].tolist()
        pos = {key: n for n, key in enumerate(sel)}
        for c, key in enumerate(rows):
            if key in pos:
                out[c] += r["dkv_rows"][pos[key]]
    return out
