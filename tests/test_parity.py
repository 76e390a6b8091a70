"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared in full; the full-size workloads are compared on
sampled independent units (a (batch, kv-head) group, a sequence, a token, a
key row) that the oracle computes on their own, with the kernels launched at
full size exactly as the benchmark launches them."""
import functools

import pytest
import torch

import oracle
import softmax_attention_backward_gb300 as A
from softmax_attention_backward_gb300 import workloads as W
from _util import assert_close, assert_lse, workload_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
MODES = [A.ATTN_DQ_ATOMIC, A.ATTN_DQ_SPLIT]


def _gpu(*ts):
    return [t.to(DEV) for t in ts]


def _err_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _check_err(err, expect=0):
    torch.cuda.synchronize()
    assert int(err.item()) == expect, f"device error word {int(err.item()):#x}"


def run_dense(q, k, v, do, causal, scale, mode, cu=None, max_seqlen=None):
    err = _err_word()
    gq, gk, gv, gdo = _gpu(q, k, v, do)
    gcu = cu.to(DEV) if cu is not None else None
    o, lse = A.attn_fwd(gq, gk, gv, causal=causal, scale=scale, cu_seqlens=gcu,
                        max_seqlen=max_seqlen, error_word=err)
    dq, dk, dv = A.dense_backward(gq, gk, gv, o, lse, gdo, mode=mode, causal=causal, scale=scale,
                                  cu_seqlens=gcu, max_seqlen=max_seqlen, error_word=err)
    _check_err(err)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def compare_dense(got, ref, units, hq, hkv):
    grp = hq // hkv
    for b, g in units:
        hs = slice(g * grp, (g + 1) * grp)
        assert_close(f"o[{b},{g}]", got["o"][b, :, hs], ref["o"][b, :, hs])
        assert_lse(f"lse[{b},{g}]", got["lse"][b, hs], ref["lse"][b, hs])
        assert_close(f"dq[{b},{g}]", got["dq"][b, :, hs], ref["dq"][b, :, hs])
        assert_close(f"dk[{b},{g}]", got["dk"][b, :, g], ref["dk"][b, :, g])
        assert_close(f"dv[{b},{g}]", got["dv"][b, :, g], ref["dv"][b, :, g])


# ----------------------------------------------------------------------------
# Dense BSHD
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("mode", MODES)
def test_mha_s128_d64_full(mode):
    w, x = workload_inputs("mha_s128_d64")
    got = run_dense(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, mode)
    ref = oracle.dense_backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
    compare_dense(got, ref, [(0, 0), (0, 1)], 2, 2)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,S,hq,hkv,D,causal", [
    (2, 200, 4, 2, 64, True),      # ragged tail, GQA 2:1
    (1, 129, 2, 2, 128, False),    # one row past a tile
    (2, 333, 8, 2, 128, True),     # several tiles + tail, GQA 4:1
    (1, 1, 2, 1, 64, True),        # a single row
    (1, 384, 3, 1, 64, False),     # three query heads per kv head
])
def test_dense_small_full(mode, B, S, hq, hkv, D, causal):
    q, k, v, do = W.dense_inputs(B, S, hq, hkv, D, seed=100 + S)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, causal, scale, mode)
    ref = oracle.dense_backward(q, k, v, do, scale, causal)
    compare_dense(got, ref, [(b, g) for b in range(B) for g in range(hkv)], hq, hkv)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,S,hq,hkv,D,causal", [
    (5, 1000, 10, 5, 64, True),     # persistent grids over 5*5 kv heads, ragged last tile
    (4, 3000, 6, 2, 128, True),     # persistent backward, 3:1 groups, ragged last tile
    (3, 1500, 16, 2, 128, False),   # 8:1 groups, no mask: every K/V tile meets every query tile
    (2, 2100, 16, 2, 128, True),    # 8:1 groups under the causal mask
])
def test_dense_persistent_odd_shapes_sampled(mode, B, S, hq, hkv, D, causal):
    """More items than SMs with batch * heads and tile counts that are not
    powers of two: the item decoding of the persistent grids (division by
    invariant integers) on the paths the small cases do not take, and large
    GQA groups (the head_dim 128 backward walks a group's query heads
    innermost)."""
    q, k, v, do = W.dense_inputs(B, S, hq, hkv, D, seed=200 + S)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, causal, scale, mode)
    units = [(0, 0), (B - 1, hkv - 1), (B // 2, hkv // 2)]
    ref = oracle.dense_backward(q, k, v, do, scale, causal, kv_heads=units)
    compare_dense(got, ref, units, hq, hkv)


def _random_dense_cases(n=8, seed=2026):
    """Seeded shapes: batch 1-3, ragged lengths 1-700, 1-8 kv heads with 1-4 query
    heads each, D in {64, 128}, causal or not."""
    g = torch.Generator().manual_seed(seed)
    r = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    cases = []
    for _ in range(n):
        hkv = r(1, 8)
        cases.append((r(1, 3), r(1, 700), hkv * r(1, 4), hkv, (64, 128)[r(0, 1)], bool(r(0, 1))))
    return cases


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("B,S,hq,hkv,D,causal", _random_dense_cases())
def test_dense_random_shapes(mode, B, S, hq, hkv, D, causal):
    q, k, v, do = W.dense_inputs(B, S, hq, hkv, D, seed=300 + S)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, causal, scale, mode)
    units = sorted({(0, 0), (B - 1, hkv - 1)})
    ref = oracle.dense_backward(q, k, v, do, scale, causal, kv_heads=units)
    compare_dense(got, ref, units, hq, hkv)


@pytest.mark.parametrize("mode", MODES)
def test_mha_causal_b8_h32_s1024_d64_sampled(mode):
    w, x = workload_inputs("mha_causal_b8_h32_s1024_d64")
    got = run_dense(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, mode)
    units = [(0, 0), (3, 17), (7, 31)]
    ref = oracle.dense_backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal, kv_heads=units)
    compare_dense(got, ref, units, w.heads_q, w.heads_kv)


@pytest.mark.parametrize("mode", MODES)
def test_gqa_causal_b4_h32x8_s4096_d128_sampled(mode):
    w, x = workload_inputs("gqa_causal_b4_h32x8_s4096_d128")
    got = run_dense(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, mode)
    units = [(0, 0), (1, 3), (2, 5), (3, 7)]
    ref = oracle.dense_backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal, kv_heads=units)
    compare_dense(got, ref, units, w.heads_q, w.heads_kv)


# ----------------------------------------------------------------------------
# THD packed variable length
# ----------------------------------------------------------------------------
def compare_thd(got, ref, cu, seqs, hq, hkv):
    cu = cu.tolist()
    for n in seqs:
        s = slice(cu[n], cu[n + 1])
        assert_close(f"o[seq {n}]", got["o"][s], ref["o"][s])
        assert_lse(f"lse[seq {n}]", got["lse"][:, s], ref["lse"][:, s])
        for key in ("dq", "dk", "dv"):
            assert_close(f"{key}[seq {n}]", got[key][s], ref[key][s])
    end = cu[-1]
    for key in ("o", "dq", "dk", "dv"):
        pad = got[key][end:]
        assert (pad == 0).all(), f"{key}: padding rows are not exact zeros"
    assert torch.isneginf(got["lse"][:, end:]).all()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("D", [64, 128])
def test_thd_small_full(mode, D):
    lens = [1, 130, 77, 256, 3]
    cap = 600
    cu = W.cu_seqlens_from(lens)
    q, k, v, do = W.thd_inputs(cap, 4, 2, D, seed=7)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, True, scale, mode, cu=cu, max_seqlen=max(lens))
    ref = oracle.thd_backward(q, k, v, do, cu, scale, True)
    compare_thd(got, ref, cu, range(len(lens)), 4, 2)


def _random_thd_cases(n=4, seed=2030):
    """Seeded THD problems: 1-6 sequences of 0-400 rows (an empty one in about
    half the cases), 0-100 padding rows, 1-4 kv heads with 1-3 query heads each,
    D in {64, 128}, causal or not."""
    g = torch.Generator().manual_seed(seed)
    r = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    cases = []
    for _ in range(n):
        lens = [r(0, 400) for _ in range(r(1, 6))]
        if r(0, 1):
            lens[r(0, len(lens) - 1)] = 0
        if sum(lens) == 0:
            lens[0] = 1
        hkv = r(1, 4)
        cases.append((tuple(lens), r(0, 100), hkv * r(1, 3), hkv, (64, 128)[r(0, 1)], bool(r(0, 1))))
    return cases


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("lens,pad,hq,hkv,D,causal", _random_thd_cases())
def test_thd_random_lengths(mode, lens, pad, hq, hkv, D, causal):
    cap = sum(lens) + pad
    cu = W.cu_seqlens_from(lens)
    q, k, v, do = W.thd_inputs(cap, hq, hkv, D, seed=400 + cap)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, causal, scale, mode, cu=cu, max_seqlen=max(lens))
    ref = oracle.thd_backward(q, k, v, do, cu, scale, causal)
    compare_thd(got, ref, cu, [n for n in range(len(lens)) if lens[n] > 0], hq, hkv)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("D", [64, 128])
def test_thd_many_sequences_descending_work_list(mode, D):
    """A causal pack of 24 sequences of 0-256 rows (two empty), 8 query heads
    over 4 kv heads: both grids are persistent (288 forward and 192 backward
    slots over 152 CTAs) and walk the descending-work item list of at most 32
    sequences, whose levels mix sequences of different lengths.  Full parity,
    padding rows exact zeros."""
    g = torch.Generator().manual_seed(90 + D)
    lens = [int(x) for x in torch.randint(1, 257, (24,), generator=g)]
    lens[5] = lens[17] = 0
    lens[9] = 256
    cap = sum(lens) + 40
    cu = W.cu_seqlens_from(lens)
    q, k, v, do = W.thd_inputs(cap, 8, 4, D, seed=91 + D)
    scale = D ** -0.5
    got = run_dense(q, k, v, do, True, scale, mode, cu=cu, max_seqlen=256)
    ref = oracle.thd_backward(q, k, v, do, cu, scale, True)
    compare_thd(got, ref, cu, [n for n in range(len(lens)) if lens[n] > 0], 8, 4)


@pytest.mark.parametrize("mode", MODES)
def test_thd_varlen_causal_h16_d128_sampled(mode):
    w, x = workload_inputs("thd_varlen_causal_h16_d128")
    got = run_dense(x["q"], x["k"], x["v"], x["do"], w.causal, w.scale, mode, cu=x["cu_seqlens"],
                    max_seqlen=max(w.lengths))
    seqs = [0, 1]                     # the longest (3670 rows) and the shortest (1053)
    ref = oracle.thd_backward(x["q"], x["k"], x["v"], x["do"], x["cu_seqlens"], w.scale, w.causal,
                              seqs=seqs)
    compare_thd(got, ref, x["cu_seqlens"], seqs, w.heads_q, w.heads_kv)


# ----------------------------------------------------------------------------
# Top-k sparse
# ----------------------------------------------------------------------------
def run_sparse(q, kv, idx, do, scale, deterministic=False):
    err = _err_word()
    gq, gkv, gidx, gdo = _gpu(q, kv, idx, do)
    o, lse = A.sparse_attn_fwd(gq, gkv, gidx, scale=scale, error_word=err)
    bwd = A.sparse_attn_bwd_deterministic if deterministic else A.sparse_attn_bwd
    dq, dkv = bwd(gq, gkv, gidx, o, gdo, lse, scale=scale, error_word=err)
    _check_err(err)
    return dict(o=o, lse=lse, dq=dq, dkv=dkv, gpu=(gq, gkv, gidx, gdo))


@pytest.mark.parametrize("T,H,K", [(600, 64, 256), (300, 16, 100), (200, 128, 64), (150, 32, 33)])
def test_sparse_small_full(T, H, K):
    q, kv, do, idx = W.sparse_inputs(T, H, K, seed=20 + H)
    scale = 576 ** -0.5
    got = run_sparse(q, kv, idx, do, scale)
    ref = oracle.sparse_backward(q, kv, idx, do, scale)
    assert_close("o", got["o"], ref["o"])
    assert_lse("lse", got["lse"], ref["lse"])
    assert_close("dq", got["dq"], ref["dq"])
    assert_close("dkv", got["dkv"], ref["dkv"])


@pytest.mark.parametrize("T,H,K", [(600, 64, 256), (300, 16, 100), (200, 128, 64), (150, 32, 33)])
def test_sparse_deterministic_small_full(T, H, K):
    """Ordered dKV: parity with the oracle, dKV bitwise equal over repeated
    runs, dQ bitwise equal to the atomic path (the same kernel computes it)."""
    q, kv, do, idx = W.sparse_inputs(T, H, K, seed=20 + H)
    scale = 576 ** -0.5
    got = run_sparse(q, kv, idx, do, scale, deterministic=True)
    ref = oracle.sparse_backward(q, kv, idx, do, scale)
    assert_close("dq", got["dq"], ref["dq"])
    assert_close("dkv", got["dkv"], ref["dkv"])
    gq, gkv, gidx, gdo = got["gpu"]
    for _ in range(3):
        dq2, dkv2 = A.sparse_attn_bwd_deterministic(gq, gkv, gidx, got["o"], gdo, got["lse"],
                                                    scale=scale)
        assert torch.equal(dkv2, got["dkv"]) and torch.equal(dq2, got["dq"])
    dq_at, _ = A.sparse_attn_bwd(gq, gkv, gidx, got["o"], gdo, got["lse"], scale=scale)
    assert torch.equal(dq_at, got["dq"])


@pytest.mark.parametrize("deterministic", [False, True])
def test_sparse_empty_lists_and_scattered_sentinels(deterministic):
    """Tokens whose whole list is -1 (o = 0, lse = -inf, dq = 0), the -1
    sentinel scattered through every list instead of trailing, and more slots
    than tokens (topk 130 over 70 tokens: three chunks, the last ragged)."""
    T, H, K = 70, 32, 130
    q, kv, do, idx = W.sparse_inputs(T, H, K, seed=61)
    idx[[5, 33, 69]] = -1
    g = torch.Generator().manual_seed(62)
    idx = torch.stack([row[torch.randperm(K, generator=g)] for row in idx])
    scale = 576 ** -0.5
    got = run_sparse(q, kv, idx, do, scale, deterministic)
    ref = oracle.sparse_backward(q, kv, idx, do, scale)
    assert_close("o", got["o"], ref["o"])
    assert_lse("lse", got["lse"], ref["lse"])
    assert_close("dq", got["dq"], ref["dq"])
    assert_close("dkv", got["dkv"], ref["dkv"])
    for t in (5, 33, 69):
        assert torch.isneginf(got["lse"][t]).all()
        assert (got["o"][t] == 0).all() and (got["dq"][t] == 0).all()


def test_sparse_deterministic_item_walk_with_empty_and_short_lists():
    """The deterministic main kernel runs 152 CTAs, each walking its items (a
    token and a 64-head block) in order: 500 tokens x 2 head blocks gives each
    CTA six or seven items, among them tokens with no valid slot (every 7th:
    dq = 0, skipped by every role) and tokens whose valid slots end in the
    first, second or third of the four chunks (top-k 200, the last chunk
    ragged).  Parity with the oracle, dKV bitwise equal over repeats, dQ
    bitwise equal to the atomic path."""
    T, H, K = 500, 128, 200
    q, kv, do, _ = W.sparse_inputs(T, H, 1, seed=71)
    idx = _random_index_lists(T, K, seed=72)
    idx[::7] = -1
    for t, last in ((3, 10), (4, 70), (9, 130), (10, 64), (11, 63)):
        idx[t, last + 1:] = -1
    scale = 576 ** -0.5
    got = run_sparse(q, kv, idx, do, scale, deterministic=True)
    ref = oracle.sparse_backward(q, kv, idx, do, scale)
    assert_close("dq", got["dq"], ref["dq"])
    assert_close("dkv", got["dkv"], ref["dkv"])
    assert (got["dq"][::7] == 0).all()
    gq, gkv, gidx, gdo = got["gpu"]
    for _ in range(2):
        dq2, dkv2 = A.sparse_attn_bwd_deterministic(gq, gkv, gidx, got["o"], gdo, got["lse"],
                                                    scale=scale)
        assert torch.equal(dkv2, got["dkv"]) and torch.equal(dq2, got["dq"])
    dq_at, dkv_at = A.sparse_attn_bwd(gq, gkv, gidx, got["o"], gdo, got["lse"], scale=scale)
    assert torch.equal(dq_at, got["dq"])
    assert_close("dkv (atomic)", dkv_at, ref["dkv"])


def _random_sparse_cases(n=4, seed=2030):
    """Seeded top-k problems: 1-300 tokens, heads in {16, 32, 64, 128}, top-k 1-300."""
    g = torch.Generator().manual_seed(seed)
    r = lambda lo, hi: int(torch.randint(lo, hi + 1, (1,), generator=g))
    return [(r(1, 300), (16, 32, 64, 128)[r(0, 3)], r(1, 300), r(0, 10 ** 6)) for _ in range(n)]


def _random_index_lists(T, K, seed):
    """int32 [T, K]: each token names min(K, T) distinct rows drawn from all T
    (not only a causal window), drops about a fifth of them to -1, and lists
    its slots in random order."""
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((T, K), -1, dtype=torch.int32)
    n = min(K, T)
    for t in range(T):
        sel = torch.randperm(T, generator=g)[:n].to(torch.int32)
        sel[torch.rand(n, generator=g) < 0.2] = -1
        row = torch.full((K,), -1, dtype=torch.int32)
        row[:n] = sel
        idx[t] = row[torch.randperm(K, generator=g)]
    return idx


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("T,H,K,seed", _random_sparse_cases())
def test_sparse_random_shapes(deterministic, T, H, K, seed):
    q, kv, do, _ = W.sparse_inputs(T, H, 1, seed=seed)
    idx = _random_index_lists(T, K, seed)
    scale = 576 ** -0.5
    got = run_sparse(q, kv, idx, do, scale, deterministic)
    ref = oracle.sparse_backward(q, kv, idx, do, scale)
    assert_close("o", got["o"], ref["o"])
    assert_lse("lse", got["lse"], ref["lse"])
    assert_close("dq", got["dq"], ref["dq"])
    assert_close("dkv", got["dkv"], ref["dkv"])


# Key rows compared at full size: rows below 2048 are named by every token after
# them (row 0 by about 4900 tokens), the last rows by a few dozen or one.
C5_ROWS = (0, 1, 1000, 2047, 4000, 4096, 8100, 8150, 8191)


@functools.lru_cache(maxsize=1)
def _c5_dkv_reference():
    w, x = workload_inputs("sparse_topk2048_t8192_h64")
    return oracle.sparse_dkv_rows(x["q"], x["kv"], x["idx"], x["do"], w.scale, C5_ROWS)


def test_sparse_deterministic_topk2048_t8192_h64_sampled():
    w, x = workload_inputs("sparse_topk2048_t8192_h64")
    got = run_sparse(x["q"], x["kv"], x["idx"], x["do"], w.scale, deterministic=True)
    q, kv, idx, do = (x[n].double() if n != "idx" else x[n] for n in ("q", "kv", "idx", "do"))
    for t in (0, 2048, 8191):
        r = oracle.sparse_token(q[t], kv, idx[t], do[t], w.scale)
        assert_close(f"dq[{t}]", got["dq"][t], r["dq"])
    ref = _c5_dkv_reference()
    for c, j in enumerate(C5_ROWS):
        assert_close(f"dkv[{j}]", got["dkv"][j], ref[c])
    gq, gkv, gidx, gdo = got["gpu"]
    _, dkv2 = A.sparse_attn_bwd_deterministic(gq, gkv, gidx, got["o"], gdo, got["lse"],
                                              scale=w.scale)
    assert torch.equal(dkv2, got["dkv"])


def test_sparse_topk2048_t8192_h64_sampled():
    w, x = workload_inputs("sparse_topk2048_t8192_h64")
    got = run_sparse(x["q"], x["kv"], x["idx"], x["do"], w.scale)
    q, kv, idx, do = (x[n].double() if n != "idx" else x[n] for n in ("q", "kv", "idx", "do"))
    for t in (0, 1, 2047, 2048, 5000, 8191):
        r = oracle.sparse_token(q[t], kv, idx[t], do[t], w.scale)
        assert_close(f"o[{t}]", got["o"][t], r["o"])
        assert_lse(f"lse[{t}]", got["lse"][t], r["lse"])
        assert_close(f"dq[{t}]", got["dq"][t], r["dq"])
    ref = _c5_dkv_reference()
    for c, j in enumerate(C5_ROWS):
        assert_close(f"dkv[{j}]", got["dkv"][j], ref[c])


@pytest.mark.parametrize("mode", MODES)
def test_thd_varlen_causal_h16_d64_persistent_sampled(mode):
    """The c4 lengths at D = 64: 2112 forward items, so the forward and the
    backward both run their persistent grids over THD sequences."""
    lens = W.varlen_lengths(3)
    cap = 32768
    cu = W.cu_seqlens_from(lens)
    q, k, v, do = W.thd_inputs(cap, 16, 16, 64, seed=31)
    got = run_dense(q, k, v, do, True, 0.125, mode, cu=cu, max_seqlen=max(lens))
    seqs = [1, 3]
    ref = oracle.thd_backward(q, k, v, do, cu, 0.125, True, seqs=seqs)
    compare_thd(got, ref, cu, seqs, 16, 16)
