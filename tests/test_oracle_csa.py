"""Pins of the CSA compressor oracle (CPU, no GPU): central finite differences of
<out, dout>, closed forms, a hand-worked example, the zero-sum of each window's
score gradient, brute-force window membership and the zero-written slots.

Source: "CSA: add fused Compressor forward+backward CuTe-DSL kernels (ported from
Megatron-LM)" (cudnn-frontend #427): PR description and backward zero-write commit."""
import json
import math
import os

import pytest
import torch

from oracle import csa_compressor as C
from softmax_attention_backward_gb300 import workloads as W

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _case(lens, D, ratio, coff, pad=3, seed=0):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens) + pad
    kv = torch.randn(T, coff * D, generator=g, dtype=F64)
    score = torch.randn(T, coff * D, generator=g, dtype=F64)
    ape = torch.randn(ratio, coff * D, generator=g, dtype=F64)
    cu = W.cu_seqlens_from(lens)
    cc = W.cu_seqlens_from([n // ratio for n in lens])
    cap = int(cc[-1]) + 2
    dout = torch.randn(cap, D, generator=g, dtype=F64)
    return kv, score, ape, dout, cu, cc, cap


def _loss(kv, score, ape, dout, cu, cc, ratio, coff, cap):
    out, _ = C.compressor_forward(kv, score, ape, cu, cc, ratio, coff, cap)
    return (out * dout).sum().item()


def _fd(fn, x, h=1e-6):
    g = torch.zeros_like(x)
    flat, gf = x.view(-1), g.view(-1)
    for i in range(flat.numel()):
        keep = flat[i].item()
        flat[i] = keep + h
        up = fn()
        flat[i] = keep - h
        dn = fn()
        flat[i] = keep
        gf[i] = (up - dn) / (2 * h)
    return g


@pytest.mark.parametrize("lens,D,ratio,coff", [([9, 3, 0, 6], 3, 2, 2), ([7, 1, 8], 2, 4, 2),
                                               ([5, 4], 3, 2, 1), ([12], 2, 4, 1)])
def test_finite_differences(lens, D, ratio, coff):
    kv, score, ape, dout, cu, cc, cap = _case(lens, D, ratio, coff, seed=len(lens) + D)
    r = C.compressor_backward(kv, score, ape, dout, cu, cc, ratio, coff, cap)
    f = lambda: _loss(kv, score, ape, dout, cu, cc, ratio, coff, cap)
    for name, x in (("dkv", kv), ("dscore", score), ("dape", ape)):
        fd = _fd(f, x)
        err = (r[name] - fd).abs().max().item()
        assert err <= 1e-6 * max(1.0, fd.abs().max().item()), (name, err)


def test_ratio_one_is_identity():
    # one token per window: softmax of one entry is 1, so out = kv and no score gradient
    kv, score, ape, dout, cu, cc, cap = _case([5, 3], 4, 1, 1, pad=2, seed=3)
    r = C.compressor_backward(kv, score, ape, dout, cu, cc, 1, 1, cap)
    torch.testing.assert_close(r["out"][:8], kv[:8], rtol=0, atol=1e-15)
    assert (r["out"][8:] == 0).all()
    torch.testing.assert_close(r["dkv"][:8], dout[:8], rtol=0, atol=1e-15)
    assert r["dscore"].abs().max() < 1e-15 and r["dape"].abs().max() < 1e-15


def test_uniform_scores_give_window_means():
    lens, D, ratio = [8, 5], 3, 2
    kv, _, _, dout, cu, cc, cap = _case(lens, D, ratio, 2, seed=4)
    zero = torch.zeros_like(kv)
    out, _ = C.compressor_forward(kv, zero, torch.zeros(ratio, 2 * D, dtype=F64), cu, cc, ratio,
                                  2, cap)
    # segment 0, block 0: mean of its own tokens' second halves
    torch.testing.assert_close(out[0], kv[0:2, D:].mean(0), rtol=0, atol=1e-15)
    # block 2: own second halves of tokens 4, 5 and previous first halves of tokens 2, 3
    ref = torch.cat([kv[4:6, D:], kv[2:4, :D]]).mean(0)
    torch.testing.assert_close(out[2], ref, rtol=0, atol=1e-15)
    # segment 1 starts a new window: its first row only sees its own tokens 8, 9
    torch.testing.assert_close(out[4], kv[8:10, D:].mean(0), rtol=0, atol=1e-15)


def test_window_score_gradients_sum_to_zero():
    # sum over a window of w*(kv - out) is zero, so the ape gradient summed over
    # the positions of both halves vanishes per dim
    kv, score, ape, dout, cu, cc, cap = _case([9, 7, 4], 5, 2, 2, seed=5)
    r = C.compressor_backward(kv, score, ape, dout, cu, cc, 2, 2, cap)
    D = 5
    tot = r["dape"][:, :D].sum(0) + r["dape"][:, D:].sum(0)
    assert tot.abs().max() < 1e-12
    # shifting every score of a dim by a constant leaves the output unchanged
    shift = score.clone()
    shift[:, 1] += 3.0
    shift[:, D + 1] += 3.0
    out2, _ = C.compressor_forward(kv, shift, ape, cu, cc, 2, 2, cap)
    torch.testing.assert_close(out2, r["out"], rtol=0, atol=1e-12)


def _frac(expr):
    env = {"ln": math.log}
    return float(eval(expr.replace("/", "/"), env)) if isinstance(expr, str) else float(expr)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "csa_hand_worked.json")) as f:
        ex = json.load(f)
    i = ex["inputs"]
    t = lambda a: torch.tensor([[_frac(x) for x in row] for row in a], dtype=F64)
    r = C.compressor_backward(t(i["kv"]), t(i["score"]), t(i["ape"]), t(i["dout"]),
                              torch.tensor(i["cu_seqlens"], dtype=torch.int32),
                              torch.tensor(i["cu_comp"], dtype=torch.int32), i["ratio"], i["coff"], 2)
    e = ex["expected"]
    torch.testing.assert_close(r["out"][:, 0], torch.tensor([_frac(x) for x in e["out"]],
                                                            dtype=F64), rtol=0, atol=1e-14)
    for key in ("dkv", "dscore", "dape"):
        torch.testing.assert_close(r[key], t(e[key]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("coff", [1, 2])
def test_consumed_slots_brute_force_and_zero_writes(coff):
    lens, D, ratio = [11, 2, 0, 8, 6], 2, 4
    kv, score, ape, dout, cu, cc, cap = _case(lens, D, ratio, coff, pad=5, seed=6)
    T = kv.shape[0]
    # brute force: (token, half) is read iff some row's window names it
    want = torch.zeros(T, coff, dtype=torch.bool)
    start = 0
    for n in lens:
        nb = n // ratio
        for t in range(start, start + nb * ratio):
            b = (t - start) // ratio
            if coff == 1:
                want[t, 0] = True
            else:
                want[t, 1] = True                    # own block
                want[t, 0] = b + 1 < nb              # next block's prev part
        start += n
    got = C.consumed_mask(T, cu, ratio, coff, D)
    assert torch.equal(got, want)
    r = C.compressor_backward(kv, score, ape, dout, cu, cc, ratio, coff, cap)
    cols = want.repeat_interleave(D, dim=1)
    assert (r["dkv"][~cols] == 0).all() and (r["dscore"][~cols] == 0).all()
    assert (r["dkv"][cols] != 0).all()
    # unread inputs do not matter: poison them
    kv2, sc2 = kv.clone(), score.clone()
    kv2[~cols], sc2[~cols] = 1e6, -1e6
    r2 = C.compressor_backward(kv2, sc2, ape, dout, cu, cc, ratio, coff, cap)
    for key in ("out", "dape"):
        torch.testing.assert_close(r2[key], r[key], rtol=0, atol=0)
    assert (r["out"][int(cc[-1]):] == 0).all()


def test_inconsistent_compressed_lengths_are_rejected():
    kv, score, ape, dout, cu, cc, cap = _case([8], 2, 4, 2, seed=7)
    with pytest.raises(ValueError):
        C.compressor_forward(kv, score, ape, cu, torch.tensor([0, 3], dtype=torch.int32), 4, 2, 4)


def _mutant_window(slip):
    orig = C.window

    def win(n_tok0, b, r_count, ratio, coff, head_dim):
        ent = orig(n_tok0, b, r_count, ratio, coff, head_dim)
        t0 = n_tok0 + b * ratio
        if slip == "leak" and b == 0 and coff == 2 and t0 >= ratio:
            ent = ent + [(t0 - ratio + r, 0, r) for r in range(r_count)]
        if slip == "swap_halves":
            ent = [(t, head_dim - off, r) for t, off, r in ent]
        if slip == "ape_shift":
            ent = [(t, off, (r + 1) % ratio) for t, off, r in ent]
        return ent
    return win


@pytest.mark.parametrize("slip", ["leak", "swap_halves", "ape_shift"])
def test_planted_window_slips_fail_a_pin(monkeypatch, slip):
    monkeypatch.setattr(C, "window", _mutant_window(slip))
    failed = 0
    for pin in (test_hand_worked_example, test_uniform_scores_give_window_means):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1
