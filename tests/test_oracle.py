"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties the oracle to an independent fact: central finite differences of
the scalar loss <O, dO>, torch's own scaled_dot_product_attention with autograd
(a library routine the oracle does not call), logsumexp, mathematical identities,
brute-force masks built by loops, closed forms and a hand-worked example.
"""
import json
import math
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
from softmax_attention_backward_gb300 import workloads

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64)


# ----------------------------------------------------------------------------
# Finite differences of L = <O, dO>
# ----------------------------------------------------------------------------
def _fd_grad(loss_fn, x, h=1e-6):
    g = torch.zeros_like(x)
    flat = x.view(-1)
    gf = g.view(-1)
    for n in range(flat.numel()):
        old = flat[n].item()
        flat[n] = old + h
        lp = loss_fn()
        flat[n] = old - h
        lm = loss_fn()
        flat[n] = old
        gf[n] = (lp - lm) / (2 * h)
    return g


def _assert_rel(a, b, tol):
    err = (a - b).abs().max().item()
    ref = max(b.abs().max().item(), 1e-12)
    assert err <= tol * ref, f"max err {err} vs ref scale {ref}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2)])
def test_dense_backward_matches_finite_differences(causal, hq, hkv):
    B, S, D = 1, 5, 3
    q, k, v, do = rnd(B, S, hq, D, seed=1), rnd(B, S, hkv, D, seed=2), rnd(B, S, hkv, D, seed=3), \
        rnd(B, S, hq, D, seed=4)
    scale = 0.7

    def loss():
        o, _ = oracle.dense_forward(q, k, v, scale, causal)
        return (o * do).sum().item()

    r = oracle.dense_backward(q, k, v, do, scale, causal)
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        _assert_rel(r[name], _fd_grad(loss, x), 1e-6)


def test_thd_backward_matches_finite_differences():
    cap, H, D = 7, 2, 3
    cu = torch.tensor([0, 2, 5], dtype=torch.int32)
    q, k, v, do = rnd(cap, H, D, seed=5), rnd(cap, H, D, seed=6), rnd(cap, H, D, seed=7), \
        rnd(cap, H, D, seed=8)
    scale = 0.9

    def loss():
        r = oracle.thd_backward(q, k, v, do, cu, scale, True)
        return (r["o"] * do).sum().item()

    r = oracle.thd_backward(q, k, v, do, cu, scale, True)
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        _assert_rel(r[name], _fd_grad(loss, x), 1e-6)


def test_sparse_backward_matches_finite_differences():
    T, H, Dk, Dv, K = 6, 2, 5, 3, 3
    q, kv, do = rnd(T, H, Dk, seed=9), rnd(T, Dk, seed=10), rnd(T, H, Dv, seed=11)
    idx = torch.tensor([[0, -1, -1], [0, 1, -1], [0, 2, -1], [1, 2, 3], [0, 3, 4], [2, 4, 5]],
                       dtype=torch.int32)
    scale = 0.6

    def loss():
        o, _ = oracle.sparse_forward(q, kv, idx, scale, dv_dims=Dv)
        return (o * do).sum().item()

    r = oracle.sparse_backward(q, kv, idx, do, scale, dv_dims=Dv)
    _assert_rel(r["dq"], _fd_grad(loss, q), 1e-6)
    _assert_rel(r["dkv"], _fd_grad(loss, kv), 1e-6)


# ----------------------------------------------------------------------------
# Library routine: scaled_dot_product_attention + autograd in fp64
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal,hq,hkv,S,D", [(False, 2, 2, 37, 16), (True, 4, 4, 33, 8),
                                              (True, 8, 2, 29, 16), (False, 6, 3, 17, 24)])
def test_dense_matches_sdpa_autograd(causal, hq, hkv, S, D):
    B = 2
    q, k, v, do = rnd(B, S, hq, D, seed=12), rnd(B, S, hkv, D, seed=13), \
        rnd(B, S, hkv, D, seed=14), rnd(B, S, hq, D, seed=15)
    scale = 1.0 / math.sqrt(D)
    qt, kt, vt = (x.transpose(1, 2).clone().requires_grad_(True) for x in (q, k, v))
    o_ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale,
                                           enable_gqa=(hq != hkv))
    o_ref.backward(do.transpose(1, 2))
    r = oracle.dense_backward(q, k, v, do, scale, causal)
    tol = 1e-10
    _assert_rel(r["o"], o_ref.detach().transpose(1, 2), tol)
    _assert_rel(r["dq"], qt.grad.transpose(1, 2), tol)
    _assert_rel(r["dk"], kt.grad.transpose(1, 2), tol)
    _assert_rel(r["dv"], vt.grad.transpose(1, 2), tol)
    # LSE against logsumexp of the masked logits (library routine)
    s = scale * torch.einsum("bihd,bjhd->bhij", q, k.repeat_interleave(hq // hkv, dim=2))
    if causal:
        s = s.masked_fill(~oracle.causal_mask(S, S), float("-inf"))
    _assert_rel(r["lse"], torch.logsumexp(s, dim=-1), 1e-12)


def test_sparse_matches_sdpa_with_index_mask():
    T, H, Dk, Dv, K = 40, 4, 12, 8, 6
    q, kv, do = rnd(T, H, Dk, seed=16), rnd(T, Dk, seed=17), rnd(T, H, Dv, seed=18)
    idx = workloads.topk_indices(T, K, seed=5)
    scale = 0.3
    mask = torch.zeros(T, T, dtype=torch.bool)
    for t in range(T):
        for j in idx[t].tolist():
            if j >= 0:
                mask[t, j] = True
    qt = q.transpose(0, 1).clone().requires_grad_(True)        # [H,T,Dk]
    kvt = kv.clone().requires_grad_(True)
    kk = kvt[None].expand(H, T, Dk)
    vv = kvt[None, :, :Dv].expand(H, T, Dv)
    o_ref = F.scaled_dot_product_attention(qt, kk, vv, attn_mask=mask[None], scale=scale)
    o_ref.backward(do.transpose(0, 1))
    r = oracle.sparse_backward(q, kv, idx, do, scale, dv_dims=Dv)
    _assert_rel(r["o"], o_ref.detach().transpose(0, 1), 1e-10)
    _assert_rel(r["dq"], qt.grad.transpose(0, 1), 1e-10)
    _assert_rel(r["dkv"], kvt.grad, 1e-10)


# ----------------------------------------------------------------------------
# Identities
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one_and_delta_identity(causal):
    S, D = 23, 7
    q, k, v, do = rnd(S, D, seed=19), rnd(S, D, seed=20), rnd(S, D, seed=21), rnd(S, D, seed=22)
    mask = oracle.causal_mask(S, S) if causal else oracle.full_mask(S, S)
    r = oracle.head_backward(q, k, v, do, 0.5, mask)
    assert (r["p"].sum(dim=1) - 1).abs().max().item() < 1e-12
    # rowsum(P o dP) == rowsum(dO o O)
    assert ((r["p"] * r["dp"]).sum(dim=1) - r["delta"]).abs().max().item() < 1e-12
    # masked pairs carry exactly zero probability and zero dS
    assert (r["p"][~mask] == 0).all() and (r["ds"][~mask] == 0).all()
    # sum_j ds_ij == 0 for every row (softmax Jacobian annihilates constants)
    assert r["ds"].sum(dim=1).abs().max().item() < 1e-12


def test_lse_is_log_of_explicit_sum():
    S, D = 9, 4
    q, k = rnd(S, D, seed=23), rnd(S, D, seed=24)
    mask = oracle.causal_mask(S, S)
    _, lse, _ = oracle.head_forward(q, k, k, 1.3, mask)
    for i in range(S):
        vals = [1.3 * float(q[i] @ k[j]) for j in range(i + 1)]
        m = max(vals)
        ref = m + math.log(sum(math.exp(x - m) for x in vals))
        assert abs(lse[i].item() - ref) < 1e-12


# ----------------------------------------------------------------------------
# Brute-force masks and structural equivalences
# ----------------------------------------------------------------------------
def test_causal_equals_loop_built_bias():
    S, D = 6, 3
    q, k, v = rnd(S, D, seed=25), rnd(S, D, seed=26), rnd(S, D, seed=27)
    o, lse, _ = oracle.head_forward(q, k, v, 1.0, oracle.causal_mask(S, S))
    # pure Python softmax with a -inf bias built entry by entry
    for i in range(S):
        logits = []
        for j in range(S):
            bias = 0.0 if j <= i else float("-inf")
            logits.append(float(q[i] @ k[j]) + bias)
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        z = sum(w)
        for d in range(D):
            ref = sum(w[j] * float(v[j, d]) for j in range(S)) / z
            assert abs(o[i, d].item() - ref) < 1e-12
        assert abs(lse[i].item() - (m + math.log(z))) < 1e-12


def test_gqa_equals_repeated_mha():
    B, S, hq, hkv, D = 2, 11, 6, 2, 5
    q, k, v, do = rnd(B, S, hq, D, seed=28), rnd(B, S, hkv, D, seed=29), \
        rnd(B, S, hkv, D, seed=30), rnd(B, S, hq, D, seed=31)
    g = oracle.dense_backward(q, k, v, do, 0.4, True)
    rep = hq // hkv
    m = oracle.dense_backward(q, k.repeat_interleave(rep, dim=2), v.repeat_interleave(rep, dim=2),
                              do, 0.4, True)
    torch.testing.assert_close(g["o"], m["o"], rtol=0, atol=1e-13)
    torch.testing.assert_close(g["dq"], m["dq"], rtol=0, atol=1e-13)
    torch.testing.assert_close(g["dk"], m["dk"].view(B, S, hkv, rep, D).sum(3), rtol=0, atol=1e-13)
    torch.testing.assert_close(g["dv"], m["dv"].view(B, S, hkv, rep, D).sum(3), rtol=0, atol=1e-13)


def test_thd_equals_independent_sequences_and_zero_padding():
    lens = [3, 1, 5]
    cap, H, D = 12, 2, 4
    cu = workloads.cu_seqlens_from(lens)
    q, k, v, do = rnd(cap, H, D, seed=32), rnd(cap, H, D, seed=33), rnd(cap, H, D, seed=34), \
        rnd(cap, H, D, seed=35)
    r = oracle.thd_backward(q, k, v, do, cu, 0.8, True)
    a = 0
    for L in lens:
        s = slice(a, a + L)
        d = oracle.dense_backward(q[None, s], k[None, s], v[None, s], do[None, s], 0.8, True)
        for key in ("o", "dq", "dk", "dv"):
            torch.testing.assert_close(r[key][s], d[key][0], rtol=0, atol=1e-13)
        torch.testing.assert_close(r["lse"][:, s], d["lse"][0], rtol=0, atol=1e-13)
        a += L
    for key in ("o", "dq", "dk", "dv"):
        assert (r[key][a:] == 0).all()
    assert torch.isneginf(r["lse"][:, a:]).all()


def test_sparse_full_index_set_equals_dense_causal():
    T, H, Dk, Dv = 9, 3, 10, 6
    q, kv, do = rnd(T, H, Dk, seed=36), rnd(T, Dk, seed=37), rnd(T, H, Dv, seed=38)
    idx = workloads.topk_indices(T, T, seed=0)          # every key of [0, t]
    assert (idx[T - 1] == torch.arange(T)).all()
    s = oracle.sparse_backward(q, kv, idx, do, 0.5, dv_dims=Dv)
    k = kv[None, :, None, :]                             # one shared kv head
    v = kv[None, :, None, :Dv]
    d = oracle.dense_backward(q[None], k, v, do[None], 0.5, True)
    torch.testing.assert_close(s["o"], d["o"][0], rtol=0, atol=1e-13)
    torch.testing.assert_close(s["dq"], d["dq"][0], rtol=0, atol=1e-13)
    dkv = d["dk"][0, :, 0].clone()
    dkv[:, :Dv] += d["dv"][0, :, 0]
    torch.testing.assert_close(s["dkv"], dkv, rtol=0, atol=1e-12)


def test_sparse_single_index_closed_form_and_unselected_rows():
    T, H, Dk, Dv = 5, 2, 6, 4
    q, kv, do = rnd(T, H, Dk, seed=39), rnd(T, Dk, seed=40), rnd(T, H, Dv, seed=41)
    idx = torch.tensor([[0, -1], [0, -1], [1, -1], [3, -1], [2, -1]], dtype=torch.int32)
    r = oracle.sparse_backward(q, kv, idx, do, 0.5, dv_dims=Dv)
    for t in range(T):
        j = int(idx[t, 0])
        torch.testing.assert_close(r["o"][t], kv[j, :Dv].expand(H, Dv), rtol=0, atol=1e-14)
        torch.testing.assert_close(r["lse"][t], 0.5 * (q[t] @ kv[j]), rtol=0, atol=1e-13)
    assert r["dq"].abs().max().item() < 1e-14
    # dV of a singly-attended row is the sum of the dO rows that picked it; dK part is 0
    for j in range(T):
        ts = [t for t in range(T) if int(idx[t, 0]) == j]
        ref = sum((do[t].sum(0) for t in ts), torch.zeros(Dv, dtype=F64))
        torch.testing.assert_close(r["dkv"][j, :Dv], ref, rtol=0, atol=1e-13)
        assert r["dkv"][j, Dv:].abs().max().item() < 1e-13
    # poisoning a row that nobody selects changes nothing
    kv2 = kv.clone()
    kv2[4] = float("nan")
    r2 = oracle.sparse_backward(q, kv2, idx, do, 0.5, dv_dims=Dv)
    torch.testing.assert_close(r2["o"], r["o"], rtol=0, atol=0)
    torch.testing.assert_close(r2["dq"], r["dq"], rtol=0, atol=0)


def test_sparse_empty_index_list_and_slot_order():
    """A token whose list holds no valid slot: the empty sum gives lse = -inf,
    o = 0 and dq = 0, and the token adds nothing to dKV.  The -1 sentinel may
    sit anywhere in a list: permuting each list's slots changes nothing."""
    T, H, Dk, Dv, K = 12, 3, 8, 5, 6
    q, kv, do = rnd(T, H, Dk, seed=57), rnd(T, Dk, seed=58), rnd(T, H, Dv, seed=59)
    idx = workloads.topk_indices(T, K, seed=9)
    idx[[4, 11]] = -1
    r = oracle.sparse_backward(q, kv, idx, do, 0.5, dv_dims=Dv)
    for t in (4, 11):
        assert torch.isneginf(r["lse"][t]).all()
        assert (r["o"][t] == 0).all() and (r["dq"][t] == 0).all() and (r["delta"][t] == 0).all()
    assert torch.isfinite(r["dkv"]).all()
    q2, do2 = q.clone(), do.clone()
    q2[[4, 11]], do2[[4, 11]] = 7.0, -3.0
    r2 = oracle.sparse_backward(q2, kv, idx, do2, 0.5, dv_dims=Dv)
    torch.testing.assert_close(r2["dkv"], r["dkv"], rtol=0, atol=0)
    g = torch.Generator().manual_seed(60)
    perm = torch.stack([row[torch.randperm(K, generator=g)] for row in idx])
    assert not torch.equal(perm, idx)
    r3 = oracle.sparse_backward(q, kv, perm, do, 0.5, dv_dims=Dv)
    for key in ("o", "dq", "dkv"):
        torch.testing.assert_close(r3[key], r[key], rtol=0, atol=1e-12)
    torch.testing.assert_close(r3["lse"], r["lse"], rtol=0, atol=1e-12)


def test_sparse_token_and_valid_against_full():
    """sparse_valid keeps exactly the slots >= 0 in list order; sparse_token's per-token
    outputs equal the rows of the finite-difference-pinned sparse_backward, and its dkv
    rows, scattered to their key rows, add up to the full dKV."""
    T, H, Dk, Dv, K = 16, 2, 8, 5, 6
    q, kv, do = rnd(T, H, Dk, seed=71), rnd(T, Dk, seed=72), rnd(T, H, Dv, seed=73)
    idx = workloads.topk_indices(T, K, seed=11)
    idx[9, 2] = -1
    full = oracle.sparse_backward(q, kv, idx, do, 0.5, dv_dims=Dv)
    acc = torch.zeros_like(full["dkv"])
    for t in range(T):
        sel = oracle.sparse_valid(idx[t])
        assert sel.tolist() == [int(x) for x in idx[t].tolist() if x >= 0]
        r = oracle.sparse_token(q[t], kv, idx[t], do[t], 0.5, Dv)
        assert torch.equal(r["rows"], sel)
        for key in ("o", "lse", "dq", "delta"):
            torch.testing.assert_close(r[key], full[key][t], rtol=0, atol=1e-13)
        for n, row in enumerate(sel.tolist()):
            acc[row] += r["dkv_rows"][n]
    torch.testing.assert_close(acc, full["dkv"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("T,H,Dk,Dv,K,seed", [(30, 2, 8, 5, 7, 6), (24, 2, 576, 512, 32, 8)])
def test_sparse_dkv_rows_matches_full(T, H, Dk, Dv, K, seed):
    """sparse_dkv_rows against the finite-difference-pinned sparse_backward, on row
    sets holding a row every token names (row 0 with K >= T), a row no token names
    (every occurrence of row 3 replaced by a -1 sentinel mid-list), heavily and
    lightly named rows, a repeated row and the last row."""
    q, kv, do = rnd(T, H, Dk, seed=42 + seed), rnd(T, Dk, seed=43 + seed), rnd(T, H, Dv, seed=44 + seed)
    idx = workloads.topk_indices(T, K, seed=seed)
    idx[idx == 3] = -1
    mid = (idx[:, :-1] == -1) & (idx[:, 1:] >= 0)
    assert mid.any()                                # a -1 slot sits before a valid one
    full = oracle.sparse_backward(q, kv, idx, do, 0.5, dv_dims=Dv)["dkv"]
    if K >= T:
        assert (idx[:, 0] == 0).all()               # row 0 is named by every token
    for rows in ([0], [3], [0, 3, 7, T - 1], [T - 1, 1, 1, 2]):
        part = oracle.sparse_dkv_rows(q, kv, idx, do, 0.5, rows, dv_dims=Dv)
        torch.testing.assert_close(part, full[rows], rtol=0, atol=1e-12)
    assert (oracle.sparse_dkv_rows(q, kv, idx, do, 0.5, [3], dv_dims=Dv) == 0).all()
    assert full[0].abs().max() > 0


# ----------------------------------------------------------------------------
# Closed forms and the hand-worked example
# ----------------------------------------------------------------------------
def test_single_key_closed_form():
    q, k, v, do = rnd(1, 1, 3, 4, seed=45), rnd(1, 1, 3, 4, seed=46), rnd(1, 1, 3, 4, seed=47), \
        rnd(1, 1, 3, 4, seed=48)
    r = oracle.dense_backward(q, k, v, do, 0.5, False)
    # one key per head (S = 1): O = V, dQ = dK = 0, dV = dO
    torch.testing.assert_close(r["o"], v, rtol=0, atol=1e-15)
    assert r["dq"].abs().max() < 1e-15 and r["dk"].abs().max() < 1e-15
    torch.testing.assert_close(r["dv"], do, rtol=0, atol=1e-15)


def test_zero_query_is_cumulative_mean():
    S, D = 8, 3
    v = rnd(1, S, 1, D, seed=49)
    k = rnd(1, S, 1, D, seed=50)
    q = torch.zeros(1, S, 1, D, dtype=F64)
    o, lse = oracle.dense_forward(q, k, v, 1.0, True)
    for i in range(S):
        torch.testing.assert_close(o[0, i, 0], v[0, :i + 1, 0].mean(0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i].item() - math.log(i + 1)) < 1e-14


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_2x2.json")) as f:
        ex = json.load(f)
    q = torch.tensor(ex["inputs"]["q"], dtype=F64).view(1, 2, 1, 2)
    k = torch.tensor(ex["inputs"]["k"], dtype=F64).view(1, 2, 1, 2)
    v = torch.tensor(ex["inputs"]["v"], dtype=F64).view(1, 2, 1, 2)
    do = torch.tensor(ex["inputs"]["do"], dtype=F64).view(1, 2, 1, 2)
    for case in ("non_causal", "causal"):
        exp = ex[case]
        r = oracle.dense_backward(q, k, v, do, ex["inputs"]["scale"], case == "causal")
        for key in ("o", "dq", "dk", "dv"):
            ref = torch.tensor(eval(exp[key], {"ln": math.log}), dtype=F64).view(1, 2, 1, 2)
            torch.testing.assert_close(r[key], ref, rtol=0, atol=1e-15)
        lse = torch.tensor(eval(exp["lse"], {"ln": math.log}), dtype=F64)
        torch.testing.assert_close(r["lse"][0, 0], lse, rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------
# Planted mistakes: each plausible slip in the formulas must fail a pin above
# ----------------------------------------------------------------------------
def _mutant_backward(q, k, v, do, scale, allowed, slip):
    o, lse, p = oracle.head_forward(q, k, v, scale, allowed)
    delta = (do * o).sum(dim=1)
    dp = do @ v.T
    if slip == "drop_delta":
        ds = p * dp
    elif slip == "sign":
        ds = p * (delta[:, None] - dp)
    else:
        ds = p * (dp - delta[:, None])
    dv = p.T @ do
    dk = (ds.T @ q) if slip == "no_scale_dk" else scale * (ds.T @ q)
    dq = scale * (ds.T @ k) if slip == "transpose_dq" else scale * (ds @ k)
    return dq, dk, dv


@pytest.mark.parametrize("slip", ["drop_delta", "sign", "no_scale_dk", "transpose_dq"])
def test_finite_differences_catch_planted_slips(slip):
    S, D = 5, 5
    q, k, v, do = rnd(S, D, seed=51), rnd(S, D, seed=52), rnd(S, D, seed=53), rnd(S, D, seed=54)
    mask = oracle.causal_mask(S, S)
    scale = 0.7

    def loss():
        o, _, _ = oracle.head_forward(q, k, v, scale, mask)
        return (o * do).sum().item()

    dq, dk, dv = _mutant_backward(q, k, v, do, scale, mask, slip)
    fd = {"dq": _fd_grad(loss, q), "dk": _fd_grad(loss, k), "dv": _fd_grad(loss, v)}
    errs = [(a - fd[n]).abs().max().item() for n, a in (("dq", dq), ("dk", dk), ("dv", dv))]
    assert max(errs) > 1e-3


# ----------------------------------------------------------------------------
# Workload recipe
# ----------------------------------------------------------------------------
def test_workload_recipe():
    w = workloads.get_workload("thd_varlen_causal_h16_d128")
    assert all(512 <= n <= 8192 for n in w.lengths) and sum(w.lengths) <= w.capacity
    idx = workloads.topk_indices(3000, 2048, seed=4)
    assert (idx[100, :101] == torch.arange(101)).all() and (idx[100, 101:] == -1).all()
    row = idx[2999]
    assert (row >= 0).all() and (row[1:] > row[:-1]).all() and int(row.max()) <= 2999
