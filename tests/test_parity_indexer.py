"""GPU parity of the DSA indexer kernels (through the C ABI) against the fp64
oracle: indexer logits (dense causal and THD, ReLU or not, ragged token counts),
the top-k selection (bit-exact: the oracle's selection rule applied to the
kernel's own fp32 logits, since floating point decides which keys are kept),
the indexer backward, and the sparse KL loss of the attention target; full
small cases and sampled rows / tokens / key rows at the 8192-token workload."""
import functools

import pytest
import torch

import softmax_attention_backward_gb300 as A
from oracle import dsa_indexer as X
from softmax_attention_backward_gb300 import workloads as W
from _util import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
F32_REL, F32_ATOL = 1e-3, 1e-3     # fp32 results computed from exact bf16 products


def close32(name, got, ref, rel=F32_REL, atol=F32_ATOL):
    g = got.detach().double().cpu()
    assert torch.isfinite(g).all(), f"{name}: non-finite values"
    err = (g - ref).abs().max().item() if ref.numel() else 0.0
    lim = rel * (ref.abs().max().item() if ref.numel() else 0.0) + atol
    assert err <= lim, f"{name}: max err {err:.3e} > {lim:.3e}"


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def check_logits(got, ref):
    g = got.double().cpu()
    fin = torch.isfinite(ref)
    assert torch.equal(torch.isneginf(g), ~fin), "cleaned (-inf) pattern differs"
    close32("logits", g[fin], ref[fin])


def check_topk(gl, vis, K, idx, length, scores):
    """The kernel's selection equals the oracle's rule on the kernel's logits."""
    ridx, rlen, rsc = X.topk_select(gl.double(), K, vis)
    assert torch.equal(length.cpu(), rlen)
    assert torch.equal(idx.cpu(), ridx)
    torch.testing.assert_close(scores.double().cpu(), rsc, rtol=0, atol=0)


CASES = [  # T, H, lens (None: one dense causal sequence), use_relu, K
    (300, 64, None, True, 64),
    (129, 16, None, False, 200),
    (517, 32, [100, 0, 77, 250], True, 96),
    (256, 64, [256], True, 256),
]


@pytest.mark.parametrize("T,H,lens,relu,K", CASES)
def test_indexer_logits_topk_small_full(T, H, lens, relu, K):
    x = W.indexer_inputs(T, H, seed=T + H, topk=K)
    cu = W.cu_seqlens_from(lens) if lens else None
    q, k, w = (x[n].to(DEV) for n in ("q", "k", "w"))
    gcu = cu.to(DEV) if cu is not None else None
    err = _err()
    logits = A.dsa_indexer_fwd(q, k, w, use_relu=relu, cu_seqlens=gcu, error_word=err)
    ref = X.indexer_logits(x["q"], x["k"], x["w"], cu_seqlens=cu, use_relu=relu)
    gl = logits[:, :T].cpu()
    check_logits(gl, ref)
    idx, length, scores = A.dsa_topk(logits, K, heads=H, cu_seqlens=gcu, error_word=err)
    check_topk(gl, X.visible_keys(T, cu), K, idx, length, scores)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_topk_heavy_ties_and_signed_zeros(seed):
    """Logits of five integer levels, zeros of both signs: the threshold class
    holds many keys, of which only the first (smallest indices) are taken, and
    -0.0 ties with +0.0 as equal values do."""
    T, K = 700, 128
    g = torch.Generator().manual_seed(seed)
    lg = torch.randint(-2, 3, (T, T), generator=g).float()
    neg = (lg == 0) & (torch.rand(T, T, generator=g) < 0.5)
    lg[neg] = -0.0
    logits = torch.full((T, A.logits_ld(T)), float("-inf"))
    logits[:, :T] = lg
    idx, length, scores = A.dsa_topk(logits.to(DEV), K)
    torch.cuda.synchronize()
    check_topk(lg, X.visible_keys(T), K, idx, length, scores)


@pytest.mark.parametrize("T,H,K,relu", [(300, 64, 64, True), (200, 16, 250, False),
                                        (150, 32, 33, True)])
def test_indexer_backward_small_full(T, H, K, relu):
    x = W.indexer_inputs(T, H, seed=7 * T + H, topk=K)
    idx = W.topk_indices(T, K, seed=T)
    idx[5] = -1                                              # a token with no slot
    q, k, w, g = (x[n].to(DEV) for n in ("q", "k", "w", "grad"))
    err = _err()
    dq, dk, dw = A.dsa_indexer_bwd(q, k, w, idx.to(DEV), g, use_relu=relu, error_word=err)
    ref = X.indexer_backward(x["q"], x["k"], x["w"], idx, x["grad"], use_relu=relu)
    assert_close("dq", dq, ref["dq"])
    assert_close("dk", dk, ref["dk"])
    close32("dw", dw, ref["dw"])
    assert (dq[5] == 0).all() and (dw[5] == 0).all()
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_indexer_backward_flags_bad_index():
    x = W.indexer_inputs(64, 16, seed=3, topk=8)
    idx = W.topk_indices(64, 8, seed=3)
    idx[10, 2] = 64                                          # out of range: skipped, flagged
    q, k, w, g = (x[n].to(DEV) for n in ("q", "k", "w", "grad"))
    err = _err()
    dq, dk, dw = A.dsa_indexer_bwd(q, k, w, idx.to(DEV), g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x1
    clean = idx.clone()
    clean[10, 2] = -1
    ref = X.indexer_backward(x["q"], x["k"], x["w"], clean, x["grad"])
    assert_close("dq", dq, ref["dq"])
    assert_close("dk", dk, ref["dk"])


@pytest.mark.parametrize("T,H,K", [(200, 64, 64), (90, 16, 100), (120, 128, 40)])
def test_sparse_kl_small_full(T, H, K):
    qa, kv, _, idx = W.sparse_inputs(T, H, K, seed=T + H)
    idx[7] = -1                                              # a token with no slot
    scale = 576 ** -0.5
    g = torch.Generator().manual_seed(T)
    scores = torch.randn(T, K, generator=g, dtype=torch.float32) * 3
    gq, gkv, gidx = qa.to(DEV), kv.to(DEV), idx.to(DEV)
    err = _err()
    _, lse = A.sparse_attn_fwd(gq, gkv, gidx, scale=scale, error_word=err)
    loss, grad, target = A.dsa_sparse_kl(gq, gkv, lse, gidx, scores.to(DEV), scale=scale,
                                         want_target=True, error_word=err)
    p = X.attention_target(qa, kv, idx, scale)
    rl, rg = X.sparse_kl(p, scores.double(), idx)
    close32("target", target, p, rel=1e-3, atol=1e-6)
    close32("grad", grad, rg, rel=1e-3, atol=1e-6)
    close32("loss", loss, rl, rel=1e-3, atol=1e-5)
    assert loss[7].item() == 0 and (grad[7] == 0).all()
    torch.cuda.synchronize()
    assert int(err.item()) == 0


# ----------------------------------------------------------------------------
# The 8192-token workload: sampled rows, tokens and key rows
# ----------------------------------------------------------------------------
@functools.lru_cache(maxsize=1)
def _full():
    c = W.INDEXER_WORKLOAD
    x = W.indexer_inputs(c["tokens"], c["heads"], c["seed"], topk=c["topk"])
    return c, x


def test_indexer_t8192_h64_top2048_sampled():
    c, x = _full()
    T, K = c["tokens"], c["topk"]
    q, k, w, g = (x[n].to(DEV) for n in ("q", "k", "w", "grad"))
    err = _err()
    logits = A.dsa_indexer_fwd(q, k, w, error_word=err)
    idx, length, scores = A.dsa_topk(logits, K, heads=c["heads"], error_word=err)
    rows = [0, 1, 127, 128, 2047, 2048, 5000, 8191]
    ref, vis = X.indexer_logits_rows(x["q"], x["k"], x["w"], rows)
    gl = logits[rows, :T].cpu()
    check_logits(gl, ref)
    check_topk(gl, vis, K, idx[rows], length[rows], scores[rows])
    # backward with the kernel's own selection
    dq, dk, dw = A.dsa_indexer_bwd(q, k, w, idx, g, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    cidx = idx.cpu()
    toks = [0, 2048, 8191]
    rb = X.indexer_backward(x["q"], x["k"], x["w"], cidx, x["grad"], tokens=toks)
    for t in toks:
        assert_close(f"dq[{t}]", dq[t], rb["dq"][t])
        close32(f"dw[{t}]", dw[t], rb["dw"][t])
    krows = [0, 1000, 8191]
    rk = X.indexer_dk_rows(x["q"], x["k"], x["w"], cidx, x["grad"], krows)
    for n, s in enumerate(krows):
        assert_close(f"dk[{s}]", dk[s], rk[n])


def test_sparse_kl_topk2048_t8192_h64_sampled():
    from _util import workload_inputs
    w_, x = workload_inputs("sparse_topk2048_t8192_h64")
    gq, gkv, gidx = x["q"].to(DEV), x["kv"].to(DEV), x["idx"].to(DEV)
    g = torch.Generator().manual_seed(9)
    scores = torch.randn(x["idx"].shape, generator=g, dtype=torch.float32) * 3
    _, lse = A.sparse_attn_fwd(gq, gkv, gidx, scale=w_.scale)
    loss, grad, target = A.dsa_sparse_kl(gq, gkv, lse, gidx, scores.to(DEV), scale=w_.scale,
                                         want_target=True)
    toks = [0, 1, 2047, 2048, 5000, 8191]
    p = X.attention_target(x["q"], x["kv"], x["idx"], w_.scale, tokens=toks)
    rl, rg = X.sparse_kl(p[toks], scores[toks].double(), x["idx"][toks])
    close32("target", target[toks], p[toks], rel=1e-3, atol=1e-6)
    close32("grad", grad[toks], rg, rel=1e-3, atol=1e-6)
    close32("loss", loss[toks], rl, rel=1e-3, atol=1e-5)


def test_outputs_fully_written_over_nan_canaries():
    """Every element of every output is written: the buffers start as NaN (or
    0x7f7f7f7f for the integer ones) and must end up equal to a run on zeroed
    buffers."""
    T, H, K = 333, 32, 100
    x = W.indexer_inputs(T, H, seed=77, topk=K)
    q, k, w, g = (x[n].to(DEV) for n in ("q", "k", "w", "grad"))
    ld = A.logits_ld(T)

    def run(fill_f, fill_i):
        logits = torch.full((T, ld), fill_f, dtype=torch.float32, device=DEV)
        A.dsa_indexer_fwd(q, k, w, logits=logits)
        idx = torch.full((T, K), fill_i, dtype=torch.int32, device=DEV)
        length = torch.full((T,), fill_i, dtype=torch.int32, device=DEV)
        scores = torch.full((T, K), fill_f, dtype=torch.float32, device=DEV)
        A.dsa_topk(logits, K, heads=H, idx=idx, length=length, scores=scores)
        dq = torch.full_like(q, fill_f)
        dk = torch.full_like(k, fill_f)
        dw = torch.full_like(w, fill_f)
        A.dsa_indexer_bwd(q, k, w, idx, g, dq=dq, dk=dk, dw=dw)
        torch.cuda.synchronize()
        return logits[:, :T], idx, length, scores, dq, dk, dw

    a = run(float("nan"), 0x7F7F7F7F)
    b = run(0.0, 0)
    for n, x1, x2 in zip(("logits", "idx", "length", "scores", "dq", "dk", "dw"), a, b):
        if n == "dk":
            # summed with fp32 atomics: every element written (finite), equal up to the
            # order of the additions
            assert torch.isfinite(x1.float()).all(), "dk: an element was left unwritten"
            torch.testing.assert_close(x1.float(), x2.float(), rtol=2e-2, atol=2e-2)
        else:
            assert torch.equal(x1, x2), f"{n}: an element was left unwritten"


def test_sparse_kl_outputs_fully_written():
    T, H, K = 100, 64, 80
    qa, kv, _, idx = W.sparse_inputs(T, H, K, seed=5)
    gq, gkv, gidx = qa.to(DEV), kv.to(DEV), idx.to(DEV)
    _, lse = A.sparse_attn_fwd(gq, gkv, gidx)
    sc = torch.randn(T, K, generator=torch.Generator().manual_seed(1)).to(DEV)
    outs = []
    for fill in (float("nan"), 0.0):
        loss = torch.full((T,), fill, device=DEV)
        grad = torch.full((T, K), fill, device=DEV)
        tgt = torch.full((T, K), fill, device=DEV)
        A.dsa_sparse_kl(gq, gkv, lse, gidx, sc, loss=loss, grad=grad, target=tgt)
        torch.cuda.synchronize()
        outs.append((loss, grad, tgt))
    for x1, x2 in zip(*outs):
        assert torch.equal(x1, x2)


def test_indexer_chain_in_a_cuda_graph():
    """logits -> top-k -> sparse attention -> KL -> indexer backward captured in
    one CUDA graph: replays reproduce the eager results, and a replay after new
    inputs are copied into the captured buffers follows them (no host reads,
    no allocation inside the calls)."""
    T, H, K, HA = 256, 64, 64, 16
    x = W.indexer_inputs(T, H, seed=3, topk=K)
    qa, kv, _, _ = W.sparse_inputs(T, HA, 1, seed=4)
    q, k, w = (x[n].to(DEV) for n in ("q", "k", "w"))
    gqa, gkv = qa.to(DEV), kv.to(DEV)
    logits = torch.empty(T, A.logits_ld(T), device=DEV)
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    length = torch.empty(T, dtype=torch.int32, device=DEV)
    scores = torch.empty(T, K, device=DEV)
    o = torch.empty(T, HA, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(T, HA, device=DEV)
    loss = torch.empty(T, device=DEV)
    grad = torch.empty(T, K, device=DEV)
    dq, dk, dw = torch.empty_like(q), torch.empty_like(k), torch.empty_like(w)
    ws = torch.empty(T * 128 * 4, dtype=torch.uint8, device=DEV)

    def chain(stream=None):
        A.dsa_indexer_fwd(q, k, w, logits=logits, stream=stream)
        A.dsa_topk(logits, K, heads=H, idx=idx, length=length, scores=scores, stream=stream)
        A.sparse_attn_fwd(gqa, gkv, idx, out=o, lse=lse, stream=stream)
        A.dsa_sparse_kl(gqa, gkv, lse, idx, scores, loss=loss, grad=grad, stream=stream)
        A.dsa_indexer_bwd(q, k, w, idx, grad, workspace=ws, dq=dq, dk=dk, dw=dw, stream=stream)

    chain()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (logits, idx, loss, grad, dq, dw)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            chain(stream=s)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    for n, e, t in zip(("logits", "idx", "loss", "grad", "dq", "dw"), eager,
                       (logits, idx, loss, grad, dq, dw)):
        if n in ("logits", "idx"):
            assert torch.equal(e, t), n
        else:
            torch.testing.assert_close(t, e, rtol=1e-5, atol=1e-6)
    # new query weights: the replay follows them
    x2 = W.indexer_inputs(T, H, seed=8, topk=K)
    w.copy_(x2["w"].to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    ref = X.indexer_logits(x["q"], x["k"], x2["w"])
    check_logits(logits[:, :T].cpu(), ref)
