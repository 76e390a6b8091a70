"""attn_bwd_fixed_scratch: the backward for callers that cannot allocate
device memory (its Delta and dQ accumulator sit in a static array the library
owns).  Checked through the C ABI against the regular workspace-based backward
and against the fp64 oracle, on two calls in a row so that leftovers of the
first call in the shared array cannot leak into the second.  This file is
collected last on purpose."""
import pytest
import torch

import oracle
import softmax_attention_backward_gb300 as A
from softmax_attention_backward_gb300 import workloads as W
from _util import assert_close

pytestmark = pytest.mark.gpu


def _regular(q, k, v, o, lse, do, causal, scale, cu=None, max_seqlen=None):
    return A.dense_backward(q, k, v, o, lse, do, mode=A.ATTN_DQ_ATOMIC, causal=causal,
                            scale=scale, cu_seqlens=cu, max_seqlen=max_seqlen)


@pytest.mark.parametrize("B,S,hq,hkv,D,causal", [(1, 128, 2, 2, 64, False),
                                                 (2, 300, 4, 2, 128, True)])
def test_fixed_scratch_matches_workspace_backward_twice(B, S, hq, hkv, D, causal):
    dev = torch.device("cuda:0")
    scale = D ** -0.5
    for call, seed in enumerate((5, 6)):
        q, k, v, do = (t.to(dev) for t in W.dense_inputs(B, S, hq, hkv, D, seed=seed))
        o, lse = A.attn_fwd(q, k, v, causal=causal, scale=scale)
        ref = _regular(q, k, v, o, lse, do, causal, scale)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        got = A.attn_bwd_fixed_scratch(q, k, v, o, do, lse, causal=causal, scale=scale,
                                       error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_close(f"call {call} {name}", g, r.double().cpu())
        # and directly against the fp64 oracle on the same inputs
        o64 = oracle.dense_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, causal)
        for name, g in zip(("dq", "dk", "dv"), got):
            assert_close(f"call {call} {name} vs oracle", g, o64[name])


def test_fixed_scratch_thd_and_capacity_limit():
    dev = torch.device("cuda:0")
    lens = [70, 1, 200]
    cu = W.cu_seqlens_from(lens).to(dev)
    q, k, v, do = (t.to(dev) for t in W.thd_inputs(300, 4, 4, 64, seed=9))
    o, lse = A.attn_fwd(q, k, v, causal=True, cu_seqlens=cu, max_seqlen=200)
    ref = _regular(q, k, v, o, lse, do, True, 0.125, cu, 200)
    for _ in range(2):
        got = A.attn_bwd_fixed_scratch(q, k, v, o, do, lse, causal=True, cu_seqlens=cu,
                                       max_seqlen=200)
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_close(name, g, r.double().cpu())
    # a problem larger than the fixed array is refused before anything runs
    big = torch.empty(1, 8192, 8, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="scratch"):
        A.attn_bwd_fixed_scratch(big, big, big, big, big,
                                 torch.empty(1, 8, 8192, dtype=torch.float32, device=dev))
    p = A._problem(big, big, False, None, None, None, None)
    ptr = A._ptr(big)
    code = A.lib().attn_bwd_fixed_scratch(A.ctypes.byref(p), ptr, ptr, ptr, ptr, ptr, ptr, ptr,
                                          ptr, ptr, A._stream(None))
    assert code == 2          # ATTN_ERR_UNSUPPORTED: exceeds ATTN_FIXED_SCRATCH_BYTES
