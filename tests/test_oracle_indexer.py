"""Pins of the DSA indexer / top-k / sparse-KL oracle (CPU, no GPU): closed forms
(identity activation = one GEMM with the weighted query; keys a query cannot see;
zero loss when the scores are the log target), linearity and homogeneity, library
sorting for the top-k, brute-force THD masks, and central finite differences.

Source: "[2/2] Add TileLang fused DSA kernels support with THD and CP & Clean up"
(Megatron-LM #5049): file table and review thread (indexer forward with logits
cleaning and use_relu, backward gradients of q, k and the weights, top-k indices
with -1 sentinels or a compact prefix, streaming sparse-KL)."""
import math

import pytest
import torch

from oracle import dsa_indexer as X
from softmax_attention_backward_gb300 import workloads as W

F64 = torch.float64


def rnd(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64)


def test_identity_activation_is_one_gemm():
    T, H, D = 9, 4, 5
    q, k, w = rnd(T, H, D, seed=1), rnd(T, D, seed=2), rnd(T, H, seed=3)
    I = X.indexer_logits(q, k, w, use_relu=False)
    qw = (w[:, :, None] * q).sum(1)                 # sum_h w_h q_h
    ref = qw @ k.T
    vis = torch.arange(T)[None, :] <= torch.arange(T)[:, None]
    torch.testing.assert_close(I[vis], ref[vis], rtol=0, atol=1e-12)
    assert torch.isneginf(I[~vis]).all()


def test_relu_linearity_and_homogeneity():
    T, H, D = 8, 3, 4
    q, k, w1, w2 = rnd(T, H, D, seed=4), rnd(T, D, seed=5), rnd(T, H, seed=6), rnd(T, H, seed=7)
    vis = X.visible_keys(T)
    a = X.indexer_logits(q, k, w1)[vis]
    b = X.indexer_logits(q, k, w2)[vis]
    torch.testing.assert_close(X.indexer_logits(q, k, w1 + w2)[vis], a + b, rtol=0, atol=1e-12)
    torch.testing.assert_close(X.indexer_logits(2.5 * q, k, w1)[vis], 2.5 * a, rtol=0, atol=1e-12)
    # keys opposite to every query give zero under ReLU and a negative sum without it
    kk = -q[:, 0, :].clone()
    qq = q[:, :1, :].expand(T, H, D).clone()
    pos = torch.ones(T, H, dtype=F64)
    I = X.indexer_logits(qq, kk, pos)
    for t in range(T):
        assert I[t, t] == 0.0
        assert X.indexer_logits(qq, kk, pos, use_relu=False)[t, t] < 0


def test_single_term_hand_value():
    # one head; token 1 has w = 2: I[1, 0] = 2 relu(<(1, 2), (3, -1)>) = 2, I[1, 1] = 2 relu(-3) = 0
    q = torch.tensor([[[0.0, 1.0]], [[1.0, 2.0]]], dtype=F64)
    k = torch.tensor([[3.0, -1.0], [-1.0, -1.0]], dtype=F64)
    w = torch.tensor([[1.0], [2.0]], dtype=F64)
    I = X.indexer_logits(q, k, w)
    assert I[0, 0] == 0.0 and math.isinf(I[0, 1]) and I[0, 1] < 0      # relu(-1) = 0; future key
    assert I[1, 0] == 2.0 and I[1, 1] == 0.0                           # 2*relu(1), 2*relu(-3)


def test_thd_mask_is_block_causal():
    cu = W.cu_seqlens_from([3, 0, 4])
    vis = X.visible_keys(9, cu)             # tokens 7, 8 are padding
    for t in range(9):
        for s in range(9):
            want = (t < 3 and s <= t) or (3 <= t < 7 and 3 <= s <= t)
            assert bool(vis[t, s]) == want, (t, s)


def test_topk_against_library_sort_and_ties():
    T, K = 40, 7
    g = torch.Generator().manual_seed(8)
    logits = torch.randint(-3, 4, (T, T), generator=g).to(F64)   # many ties
    vis = X.visible_keys(T)
    logits = torch.where(vis, logits, torch.full_like(logits, float("-inf")))
    idx, length, scores = X.topk_select(logits, K, vis)
    for t in range(T):
        n = min(K, t + 1)
        assert int(length[t]) == n
        row = idx[t, :n]
        assert (idx[t, n:] == -1).all() and torch.isneginf(scores[t, n:]).all()
        assert (row[1:] > row[:-1]).all()                          # ascending key order
        # library stable sort of (-logit, index) over the visible keys
        vals = logits[t, :t + 1]
        order = sorted(range(t + 1), key=lambda s: (-float(vals[s]), s))[:n]
        assert sorted(order) == row.tolist()
        torch.testing.assert_close(scores[t, :n], logits[t, row.long()], rtol=0, atol=0)
    # continuous values: equal to torch.topk's set
    logits2 = torch.where(vis, rnd(T, T, seed=9), torch.full((T, T), float("-inf"), dtype=F64))
    idx2, _, _ = X.topk_select(logits2, K, vis)
    for t in range(K, T):
        ref = torch.topk(logits2[t, :t + 1], K).indices.sort().values
        assert idx2[t].tolist() == ref.tolist()


def _fd(f, x, h=1e-6):
    g = torch.zeros_like(x)
    xf, gf = x.view(-1), g.view(-1)
    for i in range(xf.numel()):
        keep = xf[i].item()
        xf[i] = keep + h
        up = f()
        xf[i] = keep - h
        dn = f()
        xf[i] = keep
        gf[i] = (up - dn) / (2 * h)
    return g


@pytest.mark.parametrize("use_relu", [True, False])
def test_indexer_backward_finite_differences(use_relu):
    T, H, D, K = 7, 3, 4, 4
    q, k, w = rnd(T, H, D, seed=10), rnd(T, D, seed=11), rnd(T, H, seed=12)
    idx = W.topk_indices(T, K, seed=13)
    idx[3, 1] = -1                                                  # a mid-list sentinel
    grad = rnd(T, K, seed=14)

    def L():
        I = X.indexer_logits(q, k, w, use_relu=use_relu)
        tot = 0.0
        for t in range(T):
            for j in range(K):
                s = int(idx[t, j])
                if s >= 0:
                    tot += float(grad[t, j] * I[t, s])
        return tot

    r = X.indexer_backward(q, k, w, idx, grad, use_relu=use_relu)
    for name, x in (("dq", q), ("dk", k), ("dw", w)):
        fd = _fd(L, x)
        err = (r[name] - fd).abs().max().item()
        assert err < 1e-6 * max(1.0, fd.abs().max().item()), (name, err)


def test_attention_target_and_kl():
    T, H, Dq, K = 10, 3, 6, 5
    q, kv = rnd(T, H, Dq, seed=15), rnd(T, Dq, seed=16)
    idx = W.topk_indices(T, K, seed=17)
    idx[[2, 6], :] = -1                                           # tokens with no slot
    p = X.attention_target(q, kv, idx, 0.4)
    valid = idx >= 0
    for t in range(T):
        if valid[t].any():
            assert abs(p[t].sum().item() - 1.0) < 1e-12
    assert (p[~valid] == 0).all()
    # one head and one slot: the target is 1 there
    p1 = X.attention_target(q[:, :1], kv, W.topk_indices(T, 1, seed=3), 0.4)
    assert (p1[:, 0] == 1.0).all()
    # scores equal to ln target: zero loss and zero gradient; KL is never negative
    scores = torch.where(valid, torch.log(torch.where(valid, p, torch.ones_like(p))),
                         torch.zeros_like(p))
    loss, grad = X.sparse_kl(p, scores, idx)
    assert loss.abs().max() < 1e-12 and grad.abs().max() < 1e-12
    s2 = rnd(T, K, seed=18)
    loss2, grad2 = X.sparse_kl(p, s2, idx)
    assert (loss2 >= -1e-15).all() and loss2[[2, 6]].eq(0).all()
    assert (grad2[~valid] == 0).all()
    for t in range(T):                                             # the gradient sums to 0
        assert abs(grad2[t].sum().item()) < 1e-12

    def L():
        return X.sparse_kl(p, s2, idx)[0].sum().item()
    fd = _fd(L, s2)
    assert (fd - grad2).abs().max() < 1e-6


def test_row_and_token_restricted_variants_match_the_full_ones():
    T, H, D, K = 12, 3, 4, 5
    q, k, w = rnd(T, H, D, seed=20), rnd(T, D, seed=21), rnd(T, H, seed=22)
    cu = W.cu_seqlens_from([5, 6])
    full = X.indexer_logits(q, k, w, cu_seqlens=cu)
    rows = [0, 4, 7, 11]
    part, vis = X.indexer_logits_rows(q, k, w, rows, cu_seqlens=cu)
    assert torch.equal(vis, X.visible_keys(T, cu)[rows])
    fin = torch.isfinite(full[rows])
    assert torch.equal(fin, torch.isfinite(part))
    torch.testing.assert_close(part[fin], full[rows][fin], rtol=0, atol=1e-12)
    idx = W.topk_indices(T, K, seed=23)
    grad = rnd(T, K, seed=24)
    r = X.indexer_backward(q, k, w, idx, grad)
    for kr in ([0], [1, 2, 9], [11]):
        torch.testing.assert_close(X.indexer_dk_rows(q, k, w, idx, grad, kr), r["dk"][kr],
                                   rtol=0, atol=1e-12)
    sub = X.indexer_backward(q, k, w, idx, grad, tokens=[3, 8])
    for t in (3, 8):
        torch.testing.assert_close(sub["dq"][t], r["dq"][t], rtol=0, atol=1e-12)
        torch.testing.assert_close(sub["dw"][t], r["dw"][t], rtol=0, atol=1e-12)
    assert (sub["dq"][[0, 1, 2]] == 0).all()
    qa, kv = rnd(T, 2, 6, seed=25), rnd(T, 6, seed=26)
    pt = X.attention_target(qa, kv, idx, 0.3)
    ps = X.attention_target(qa, kv, idx, 0.3, tokens=[2, 10])
    torch.testing.assert_close(ps[[2, 10]], pt[[2, 10]], rtol=0, atol=0)
    assert (ps[[0, 1, 3]] == 0).all()
