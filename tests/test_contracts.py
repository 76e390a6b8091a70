"""GPU tests of the buffer, determinism, graph and error contracts of the C ABI.

- ATTN_DQ_SPLIT gradients are bitwise identical run to run (head_dim 64:
  disjoint partial stores + fixed-order sum; head_dim 128: partials added in
  K/V tile order behind per-query-tile tickets), and independent of the
  workspace contents.
- Every output element is written: buffers pre-filled with NaN come out
  finite, and THD padding rows come out as exact zeros (the exact-zero
  contract of cudnn-frontend #427 for tokens past cu_seqlens[-1]).
- The launch sequence can be captured in a CUDA graph and replayed with new
  device-side cu_seqlens contents.
- Problems only the device sees are reported through the error word.
"""
import pytest
import torch

import oracle
import softmax_attention_backward_gb300 as A
from softmax_attention_backward_gb300 import workloads as W
from _util import assert_close, assert_lse

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _dense(B=2, S=333, hq=8, hkv=2, D=64, seed=3):
    return [t.to(DEV) for t in W.dense_inputs(B, S, hq, hkv, D, seed=seed)]


@pytest.mark.parametrize("D", [64, 128])
def test_split_mode_is_bitwise_deterministic(D):
    q, k, v, do = _dense(D=D)
    o, lse = A.attn_fwd(q, k, v, causal=True)
    runs = []
    for i in range(5):
        n = A.attn_bwd_workspace_size(q, k, mode=A.ATTN_DQ_SPLIT, causal=True)
        ws = torch.full((n,), 0xFF if i % 2 else 0x7F, dtype=torch.uint8, device=DEV)  # NaN-ish junk
        runs.append(A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_SPLIT, causal=True,
                                     workspace=ws))
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [True, False])
def test_split_mode_d128_ordered_accumulation_is_bitwise_deterministic(causal):
    # head_dim 128 adds the dQ partials of a query tile in K/V tile order behind
    # a ticket; at this size the K/V tiles of one (batch, kv head) run on many
    # CTAs at once, so the tickets are contended
    q, k, v, do = _dense(B=2, S=2048, hq=8, hkv=2, D=128, seed=11)
    o, lse = A.attn_fwd(q, k, v, causal=causal)
    n = A.attn_bwd_workspace_size(q, k, mode=A.ATTN_DQ_SPLIT, causal=causal)
    runs = []
    for i in range(3):
        ws = torch.full((n,), 0xFF if i % 2 else 0x7F, dtype=torch.uint8, device=DEV)
        runs.append(A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_SPLIT, causal=causal,
                                     workspace=ws))
    for r in runs[1:]:
        for x, y in zip(runs[0], r):
            assert torch.equal(x, y)
    # and the same gradients as the unordered accumulation, up to addition order
    ref = A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_ATOMIC, causal=causal)
    for name, x, y in zip(("dq", "dk", "dv"), runs[0], ref):
        assert_close(name, x, y.double().cpu())


def test_split_mode_d128_thd_is_bitwise_deterministic():
    lens = [1500, 1, 700, 2100, 0, 300]
    cap = sum(lens) + 64
    q, k, v, do = (t.to(DEV) for t in W.thd_inputs(cap, 8, 2, 128, seed=12))
    cu = W.cu_seqlens_from(lens).to(DEV)
    kw = dict(causal=True, cu_seqlens=cu, max_seqlen=max(lens))
    o, lse = A.attn_fwd(q, k, v, **kw)
    n = A.attn_bwd_workspace_size(q, k, mode=A.ATTN_DQ_SPLIT, **kw)
    runs = []
    for i in range(3):
        ws = torch.full((n,), 0xFF if i % 2 else 0x7F, dtype=torch.uint8, device=DEV)
        runs.append(A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_SPLIT, workspace=ws,
                                     **kw))
    for r in runs[1:]:
        for x, y in zip(runs[0], r):
            assert torch.equal(x, y)
    ref = oracle.thd_backward(*(t.cpu() for t in (q, k, v, do)), cu.cpu(), 128 ** -0.5, True,
                              seqs=[0, 2])
    for key, t in zip(("dq", "dk", "dv"), runs[0]):
        for s0, s1 in ((0, 1500), (1501, 2201)):
            assert_close(f"{key} rows {s0}..{s1}", t[s0:s1], ref[key][s0:s1])


def test_outputs_fully_written_dense():
    q, k, v, do = _dense(B=1, S=200, hq=4, hkv=4, D=128)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 4, 200), float("nan"), dtype=torch.float32, device=DEV)
    A.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for mode in (A.ATTN_DQ_ATOMIC, A.ATTN_DQ_SPLIT):
        dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
        n = A.attn_bwd_workspace_size(q, k, mode=mode, causal=True)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)
        delta = A.attn_bwd_preprocess(q, k, o, do, mode=mode, workspace=ws, causal=True)
        A.attn_bwd(q, k, v, do, lse, delta, mode=mode, workspace=ws, causal=True, dk=dk, dv=dv)
        A.attn_bwd_postprocess(q, k, dk, dv, mode=mode, workspace=ws, causal=True, dq=dq)
        for t in (dq, dk, dv):
            assert torch.isfinite(t).all()


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("D", [64, 128])
def test_thd_padding_rows_exact_zero_in_nan_buffers(mode, D):
    """Padding rows of every output exact zeros in NaN-filled buffers: at head_dim
    64 the postprocess writes those of dq, dk and dv, at head_dim 128 attn_bwd
    writes those of dk and dv (a warp of the main kernel) and the postprocess
    those of dq."""
    lens = [5, 130, 64]
    cap = 256
    cu = W.cu_seqlens_from(lens).to(DEV)
    q, k, v, do = (t.to(DEV) for t in W.thd_inputs(cap, 4, 2, D, seed=12))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((4, cap), float("nan"), dtype=torch.float32, device=DEV)
    A.attn_fwd(q, k, v, causal=True, cu_seqlens=cu, max_seqlen=130, out=o, lse=lse)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    n = A.attn_bwd_workspace_size(q, k, mode=mode, causal=True, cu_seqlens=cu, max_seqlen=130)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=DEV)
    kw = dict(mode=mode, causal=True, cu_seqlens=cu, max_seqlen=130, workspace=ws)
    delta = torch.full((4, cap), float("nan"), dtype=torch.float32, device=DEV)
    A.attn_bwd_preprocess(q, k, o, do, delta=delta, **kw)
    # Delta = rowsum(dO * O) on the valid rows, exact zeros on the padding rows
    end = sum(lens)
    want = (do.double() * o.double()).sum(-1).t()[:, :end]
    assert torch.allclose(delta[:, :end].double(), want, rtol=1e-4, atol=1e-4)
    assert (delta[:, end:] == 0).all()
    A.attn_bwd(q, k, v, do, lse, delta, dk=dk, dv=dv, **kw)
    A.attn_bwd_postprocess(q, k, dk, dv, dq=dq, **kw)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t).all()
        assert (t[end:] == 0).all()
    assert torch.isneginf(lse[:, end:]).all() and torch.isfinite(lse[:, :end]).all()
    ref = oracle.thd_backward(*(t.cpu() for t in (q, k, v, do)), cu.cpu(), D ** -0.5, True)
    assert_close("dq", dq, ref["dq"])
    assert_close("dk", dk, ref["dk"])


def test_graph_capture_and_replay_with_new_cu_seqlens():
    cap, H, D = 512, 4, 64
    q, k, v, do = (t.to(DEV) for t in W.thd_inputs(cap, H, H, D, seed=21))
    cu = W.cu_seqlens_from([100, 200, 50]).to(DEV)
    max_seqlen = 300
    o = torch.empty_like(q)
    lse = torch.empty(H, cap, dtype=torch.float32, device=DEV)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    n = A.attn_bwd_workspace_size(q, k, mode=A.ATTN_DQ_SPLIT, causal=True, cu_seqlens=cu,
                                  max_seqlen=max_seqlen)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    kw = dict(causal=True, cu_seqlens=cu, max_seqlen=max_seqlen)

    def step():
        A.attn_fwd(q, k, v, out=o, lse=lse, **kw)
        delta = A.attn_bwd_preprocess(q, k, o, do, mode=A.ATTN_DQ_SPLIT, workspace=ws, **kw)
        A.attn_bwd(q, k, v, do, lse, delta, mode=A.ATTN_DQ_SPLIT, workspace=ws, dk=dk, dv=dv, **kw)
        A.attn_bwd_postprocess(q, k, dk, dv, mode=A.ATTN_DQ_SPLIT, workspace=ws, dq=dq, **kw)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for lens in ([100, 200, 50], [300, 1, 120], [17, 0, 260]):
        cu.copy_(W.cu_seqlens_from(lens).to(DEV))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.thd_backward(*(t.cpu() for t in (q, k, v, do)), cu.cpu(), 0.125, True)
        end = sum(lens)
        assert_close(f"o {lens}", o[:end], ref["o"][:end])
        assert_lse(f"lse {lens}", lse[:, :end], ref["lse"][:, :end])
        for key, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert_close(f"{key} {lens}", t, ref[key])


def test_sparse_out_of_range_index_is_flagged_and_skipped():
    T, H, K = 80, 16, 24
    q, kv, do, idx = W.sparse_inputs(T, H, K, seed=31)
    bad = idx.clone()
    bad[50, 3] = T + 7           # out of range
    bad[60, 0] = -5              # below the -1 sentinel
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = A.sparse_attn_fwd(q.to(DEV), kv.to(DEV), bad.to(DEV), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x1
    cleaned = bad.clone()
    cleaned[(cleaned < -1) | (cleaned >= T)] = -1
    ref_o, ref_lse = oracle.sparse_forward(q, kv, cleaned, 576 ** -0.5)
    assert_close("o", o, ref_o)
    assert_lse("lse", lse, ref_lse)
    # both backward paths skip the bad slots (the deterministic one in its
    # chunk counts and its slab adds alike) and flag them
    ref = oracle.sparse_backward(q, kv, cleaned, do, 576 ** -0.5)
    for bwd in (A.sparse_attn_bwd, A.sparse_attn_bwd_deterministic):
        err.zero_()
        dq, dkv = bwd(q.to(DEV), kv.to(DEV), bad.to(DEV), o, do.to(DEV), lse, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) & 0x1
        assert_close("dq", dq, ref["dq"])
        assert_close("dkv", dkv, ref["dkv"])


def test_split_mode_flags_sequence_longer_than_max_seqlen():
    cap, H, D = 384, 2, 64
    q, k, v, do = (t.to(DEV) for t in W.thd_inputs(cap, H, H, D, seed=41))
    cu = W.cu_seqlens_from([300, 20]).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, lse = A.attn_fwd(q, k, v, causal=True, cu_seqlens=cu, max_seqlen=128)
    A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_SPLIT, causal=True, cu_seqlens=cu,
                     max_seqlen=128, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x4


def test_binding_rejects_bad_tensors():
    q, k, v, _ = _dense(B=1, S=64, hq=2, hkv=2, D=64)
    with pytest.raises(A.AttnError, match="unsupported"):
        A.attn_fwd(q[..., :32].contiguous(), k[..., :32].contiguous(), v[..., :32].contiguous())
    with pytest.raises(ValueError, match="contiguous"):
        A.attn_fwd(q.transpose(1, 2), k, v)
    with pytest.raises(TypeError):
        A.attn_fwd(q.float(), k, v)


def test_sparse_outputs_fully_written():
    T, H, K = 96, 32, 40
    q, kv, do, idx = (t.to(DEV) for t in W.sparse_inputs(T, H, K, seed=51))
    o = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
    A.sparse_attn_fwd(q, kv, idx, out=o, lse=lse)
    dq, dkv = torch.full_like(q, float("nan")), torch.full_like(kv, float("nan"))
    ws = torch.full((A.sparse_attn_bwd_workspace_size(q, idx),), 0xFF, dtype=torch.uint8, device=DEV)
    A.sparse_attn_bwd(q, kv, idx, o, do, lse, workspace=ws, dq=dq, dkv=dkv)
    for t in (o, lse, dq, dkv):
        assert torch.isfinite(t).all()
    # deterministic path: 0xFF-filled workspace (its slabs are cleared by the call)
    # and NaN outputs, every slot still written,
    # key rows that no token names get exact zeros
    dq2, dkv2 = torch.full_like(q, float("nan")), torch.full_like(kv, float("nan"))
    ws2 = torch.full((A.sparse_attn_bwd_deterministic_workspace_size(q, idx),), 0xFF,
                     dtype=torch.uint8, device=DEV)
    A.sparse_attn_bwd_deterministic(q, kv, idx, o, do, lse, workspace=ws2, dq=dq2, dkv=dkv2)
    assert torch.isfinite(dq2).all() and torch.isfinite(dkv2).all()
    named = torch.zeros(T, dtype=torch.bool, device=DEV)
    named[idx[idx >= 0].long()] = True
    assert (dkv2[~named] == 0).all()
    assert torch.equal(dq2, dq)


def test_bounded_wait_runs_out_sets_timeout_and_returns():
    """The library's bounded mbarrier wait, made to run out (a barrier nothing
    completes, 2 ms limit): the error word gets the timeout bit, the other role
    stops on the abort flag, the CTA frees its TMEM and returns, and the context
    stays usable for a regular call afterwards."""
    res, err = A.attn_wait_selftest(2000)
    assert res == 7, f"self-test result bits {res:#x}"
    assert err & 0x2
    q, k, v, do = (t.to(DEV) for t in W.dense_inputs(1, 64, 2, 2, 64, seed=1))
    o, lse = A.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
