"""GPU parity of the CSA compressor kernels (through the C ABI) against the fp64
oracle: ragged THD packs (segments shorter than ratio, empty segments, static
capacity padding of tokens and compressed rows), every (ratio, coff) the kernels
instantiate, head_dim 64 to 512, the page's four benchmark shapes in full, the
exact zeros of never-read slots over NaN-filled outputs, bitwise repeatability,
and the device error bit of an inconsistent row layout."""
import pytest
import torch

import softmax_attention_backward_gb300 as A
from oracle import csa_compressor as C
from softmax_attention_backward_gb300 import workloads as W
from _util import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
DAPE_REL, DAPE_ATOL = 1e-3, 1e-4      # dape is fp32 end to end


def _gpu(x):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}


def run(x, ratio, coff, nan_outputs=True):
    g = _gpu(x)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((x["comp_capacity"], x["kv"].shape[1] // coff), float("nan"),
                     dtype=torch.bfloat16, device=DEV) if nan_outputs else None
    out = A.csa_compressor_fwd(g["kv"], g["score"], g["ape"], g["cu_seqlens"],
                               g["cu_seqlens_comp"], ratio=ratio, coff=coff,
                               comp_capacity=x["comp_capacity"], out=out, error_word=err)
    nan = (lambda t: torch.full_like(t, float("nan"))) if nan_outputs else (lambda t: None)
    dkv, dscore, dape = A.csa_compressor_bwd(g["kv"], g["score"], g["ape"], g["dout"],
                                             g["cu_seqlens"], g["cu_seqlens_comp"], ratio=ratio,
                                             coff=coff, dkv=nan(g["kv"]), dscore=nan(g["score"]),
                                             dape=nan(g["ape"]), error_word=err)
    torch.cuda.synchronize()
    return dict(out=out, dkv=dkv, dscore=dscore, dape=dape, err=int(err.item()), gpu=g)


def compare(got, x, ratio, coff):
    ref = C.compressor_backward(x["kv"], x["score"], x["ape"], x["dout"], x["cu_seqlens"],
                                x["cu_seqlens_comp"], ratio, coff, x["comp_capacity"])
    assert got["err"] == 0
    assert_close("out", got["out"], ref["out"])
    assert_close("dkv", got["dkv"], ref["dkv"])
    assert_close("dscore", got["dscore"], ref["dscore"])
    d = got["dape"].double().cpu()
    assert torch.isfinite(d).all()
    err = (d - ref["dape"]).abs().max().item()
    assert err <= DAPE_REL * ref["dape"].abs().max().item() + DAPE_ATOL, f"dape err {err:.3e}"
    # never-read slots and padding rows are exact zeros (the outputs started as NaN)
    D = x["kv"].shape[1] // coff
    used = C.consumed_mask(x["kv"].shape[0], x["cu_seqlens"], ratio, coff, D)
    cols = used.repeat_interleave(D, dim=1)
    for key in ("dkv", "dscore"):
        assert (got[key].cpu()[~cols] == 0).all(), f"{key}: unread slots are not exact zeros"
    end = int(x["cu_seqlens_comp"][-1])
    assert (got["out"].cpu()[end:] == 0).all()
    return ref


CASES = [  # lengths, D, ratio, coff, pad_tokens, pad_rows
    ([37, 3, 0, 64, 9], 64, 4, 2, 5, 3),
    ([130, 1, 77], 128, 4, 1, 0, 0),
    ([50, 50, 7], 192, 2, 2, 11, 2),
    ([17, 40], 64, 2, 1, 3, 1),
    ([100, 3, 64], 128, 8, 2, 0, 4),
    ([90], 256, 8, 1, 2, 0),
    ([1000, 5, 333], 512, 4, 2, 7, 5),
]


@pytest.mark.parametrize("lengths,D,ratio,coff,pad_t,pad_r", CASES)
def test_csa_small_full(lengths, D, ratio, coff, pad_t, pad_r):
    x = W.csa_inputs(lengths, D, ratio, coff, seed=sum(lengths) + D, pad_tokens=pad_t,
                     pad_rows=pad_r)
    compare(run(x, ratio, coff), x, ratio, coff)


def test_csa_no_compressed_rows():
    # every segment shorter than ratio: no output rows, all gradients exact zeros
    x = W.csa_inputs([3, 1, 2], 64, 4, 2, seed=3, pad_tokens=4)
    x["dout"] = x["dout"][:0]
    x["comp_capacity"] = 0
    got = run(x, 4, 2)
    assert got["err"] == 0 and got["out"].numel() == 0
    assert (got["dkv"] == 0).all() and (got["dscore"] == 0).all() and (got["dape"] == 0).all()


@pytest.mark.parametrize("name", list(W.CSA_WORKLOADS))
def test_csa_benchmark_shapes_full(name):
    c = W.CSA_WORKLOADS[name]
    x = W.csa_inputs(c["lengths"], c["head_dim"], c["ratio"], c["coff"], c["seed"])
    got = run(x, c["ratio"], c["coff"])
    compare(got, x, c["ratio"], c["coff"])
    # bitwise run-to-run: disjoint stores and the fixed-order dape sums
    g = got["gpu"]
    for _ in range(2):
        dkv, dscore, dape = A.csa_compressor_bwd(g["kv"], g["score"], g["ape"], g["dout"],
                                                 g["cu_seqlens"], g["cu_seqlens_comp"],
                                                 ratio=c["ratio"], coff=c["coff"])
        assert torch.equal(dkv, got["dkv"]) and torch.equal(dscore, got["dscore"])
        assert torch.equal(dape, got["dape"])


def test_csa_inconsistent_layout_is_flagged():
    x = W.csa_inputs([40, 24], 64, 4, 2, seed=8, pad_rows=2)
    x["cu_seqlens_comp"] = torch.tensor([0, 9, 15], dtype=torch.int32)   # 10 rows for 40 tokens
    got = run(x, 4, 2)
    assert got["err"] & 0x8
    # the rejected segment's rows are zero, its tokens' gradients exact zeros
    assert (got["out"][:9].cpu() == 0).all()
    assert (got["dkv"][:40].cpu() == 0).all() and (got["dscore"][:40].cpu() == 0).all()
    # the consistent segment is still right
    sub = W.csa_inputs([24], 64, 4, 2, seed=1)
    sub.update(kv=x["kv"][40:64], score=x["score"][40:64], ape=x["ape"], dout=x["dout"][9:15],
               comp_capacity=6)
    ref = C.compressor_backward(sub["kv"], sub["score"], sub["ape"], sub["dout"],
                                sub["cu_seqlens"], sub["cu_seqlens_comp"], 4, 2, 6)
    assert_close("out[seg 1]", got["out"][9:15], ref["out"])
    assert_close("dkv[seg 1]", got["dkv"][40:64], ref["dkv"])


def test_csa_graph_replay_follows_device_side_lengths():
    """Forward and backward captured in a CUDA graph over a static capacity;
    replaying after new cu_seqlens / cu_seqlens_comp contents are copied into
    the captured buffers gives the oracle's result for the new layout (the
    library never reads the lengths on the host)."""
    cap_t, cap_c, D = 160, 40, 128
    first, second = [64, 30, 17], [9, 100, 40]
    x = W.csa_inputs([cap_t], D, 4, 2, seed=11)
    g = {n: x[n].to(DEV) for n in ("kv", "score", "ape")}
    dout = torch.randn(cap_c, D, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).to(DEV)
    cu = W.cu_seqlens_from(first).to(DEV)
    cc = W.cu_seqlens_from([n // 4 for n in first]).to(DEV)
    out = torch.empty(cap_c, D, dtype=torch.bfloat16, device=DEV)
    dkv, dsc = torch.empty_like(g["kv"]), torch.empty_like(g["score"])
    dape = torch.empty_like(g["ape"])
    n = A.csa_compressor_bwd_workspace_size(g["kv"], cu, cc, comp_capacity=cap_c)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)

    def step(stream=None):
        A.csa_compressor_fwd(g["kv"], g["score"], g["ape"], cu, cc, comp_capacity=cap_c, out=out,
                             stream=stream)
        A.csa_compressor_bwd(g["kv"], g["score"], g["ape"], dout, cu, cc, workspace=ws, dkv=dkv,
                             dscore=dsc, dape=dape, stream=stream)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(stream=s)
    torch.cuda.synchronize()
    for lens in (second, first):
        cu.copy_(W.cu_seqlens_from(lens).to(DEV))
        cc.copy_(W.cu_seqlens_from([m // 4 for m in lens]).to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        ref = C.compressor_backward(x["kv"], x["score"], x["ape"], dout.cpu(),
                                    W.cu_seqlens_from(lens),
                                    W.cu_seqlens_from([m // 4 for m in lens]), 4, 2, cap_c)
        assert_close("out", out, ref["out"])
        assert_close("dkv", dkv, ref["dkv"])
        assert_close("dscore", dsc, ref["dscore"])
        err = (dape.double().cpu() - ref["dape"]).abs().max().item()
        assert err <= DAPE_REL * ref["dape"].abs().max().item() + DAPE_ATOL
