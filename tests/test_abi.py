"""Host-only checks of the C ABI: the library builds and loads, exports every
function declared in include/*.h, and rejects invalid calls before touching
the GPU (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

import softmax_attention_backward_gb300 as A
from softmax_attention_backward_gb300 import build as B

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def L():
    B.build()
    return A.lib()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\(", text,
                                 flags=re.M)))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert set(names) == set(A.EXPORTED_SYMBOLS), names
    for n in names:
        assert getattr(L, n) is not None


def test_status_strings_and_version(L):
    assert A.attn_status_string(0) == "ok"
    assert "aligned" in A.attn_status_string(3)
    assert A.attn_status_string(99) == "unknown status"
    assert A.attn_version() >= 100


def _problem(**kw):
    p = A._Problem()
    p.batch, p.seqlen, p.heads_q, p.heads_kv, p.head_dim = 1, 128, 2, 2, 64
    p.causal, p.scale = 0, 0.125
    p.cu_seqlens, p.num_seqs, p.capacity, p.max_seqlen, p.error_word = None, 0, 0, 0, None
    for k, v in kw.items():
        setattr(p, k, v)
    return p


FAKE = 0x10000   # 16-byte aligned; never dereferenced (validation fails first or nothing runs)


def _fwd(L, p, ptrs=(FAKE,) * 5):
    return L.attn_fwd(ctypes.byref(p), *[ctypes.c_void_p(x) for x in ptrs], None)


def test_dense_validation(L):
    assert _fwd(L, _problem(head_dim=96)) == 2                     # unsupported dim
    assert _fwd(L, _problem(heads_q=3, heads_kv=2)) == 1           # group mismatch
    assert _fwd(L, _problem(heads_kv=0)) == 1
    assert _fwd(L, _problem(scale=float("nan"))) == 1
    assert _fwd(L, _problem(), (FAKE, 0, FAKE, FAKE, FAKE)) == 1   # null k
    assert _fwd(L, _problem(), (FAKE, FAKE + 8, FAKE, FAKE, FAKE)) == 3
    assert _fwd(L, _problem(seqlen=0)) == 0                         # empty: nothing enqueued
    assert _fwd(L, _problem(batch=0)) == 0
    assert L.attn_fwd(None, *[ctypes.c_void_p(FAKE)] * 5, None) == 1


def test_thd_validation_and_workspace(L):
    thd = dict(cu_seqlens=FAKE, num_seqs=4, capacity=32768, max_seqlen=3670, head_dim=128,
               heads_q=16, heads_kv=16)
    assert _fwd(L, _problem(**dict(thd, num_seqs=0))) == 1
    assert _fwd(L, _problem(**dict(thd, cu_seqlens=FAKE + 2))) == 3
    assert _fwd(L, _problem(**dict(thd, capacity=0))) == 0
    p = _problem(**thd)
    per = 32768 * 16 * 128 * 4
    assert L.attn_bwd_workspace_size(ctypes.byref(p), 0) == per
    # SPLIT, head_dim 128: one accumulator + an int32 order ticket per (head,
    # query tile slot); THD slots: 32768 / 128 + one per sequence
    assert L.attn_bwd_workspace_size(ctypes.byref(p), 1) == per + 16 * (256 + 4) * 4
    # SPLIT, head_dim 64: one slab per K/V tile of the longest sequence
    p64 = _problem(**dict(thd, head_dim=64))
    assert L.attn_bwd_workspace_size(ctypes.byref(p64), 1) == per // 2 * ((3670 + 127) // 128)
    # workspace missing / too small is rejected before any launch
    args = [ctypes.c_void_p(FAKE)] * 8           # q k v dout lse delta dk dv
    assert L.attn_bwd(ctypes.byref(p), 0, *args, None, 0, None) == 5
    assert L.attn_bwd(ctypes.byref(p), 0, *args, ctypes.c_void_p(FAKE), 16, None) == 5
    assert L.attn_bwd(ctypes.byref(p), 7, *args, ctypes.c_void_p(FAKE), per, None) == 1
    assert L.attn_bwd_preprocess(ctypes.byref(p), 0, *args[:3], None, 0, None) == 5
    assert L.attn_bwd_postprocess(ctypes.byref(p), 0, None, 0, *args[:3], None) == 5
    assert L.attn_bwd_postprocess(ctypes.byref(p), 1, ctypes.c_void_p(FAKE), per, *args[:3],
                                  None) == 5


def test_dense_workspace_sizes(L):
    p = _problem(batch=4, seqlen=4096, heads_q=32, heads_kv=8, head_dim=128, causal=1)
    per = 4 * 4096 * 32 * 128 * 4
    assert L.attn_bwd_workspace_size(ctypes.byref(p), 0) == per
    assert L.attn_bwd_workspace_size(ctypes.byref(p), 1) == per + 4 * 32 * 32 * 4
    p64 = _problem(batch=4, seqlen=4096, heads_q=32, heads_kv=8, head_dim=64, causal=1)
    assert L.attn_bwd_workspace_size(ctypes.byref(p64), 1) == per // 2 * 32
    assert L.attn_bwd_workspace_size(ctypes.byref(_problem(head_dim=80)), 0) == 0


def _sparse(**kw):
    p = A._SparseProblem()
    p.tokens, p.heads, p.dim_qk, p.dim_v, p.topk, p.scale, p.error_word = 8192, 64, 576, 512, \
        2048, 1 / 24, None
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_sparse_validation(L):
    f = lambda p, ptrs=(FAKE,) * 5: L.sparse_attn_fwd(ctypes.byref(p),
                                                      *[ctypes.c_void_p(x) for x in ptrs], None)
    assert f(_sparse(dim_qk=512)) == 2
    assert f(_sparse(dim_v=256)) == 2
    assert f(_sparse(heads=48)) == 2
    assert f(_sparse(tokens=-1)) == 1
    assert f(_sparse(), (FAKE, FAKE, FAKE + 2, FAKE, FAKE)) == 3     # idx not 4-byte aligned
    assert f(_sparse(tokens=0)) == 0
    p = _sparse()
    ws = L.sparse_attn_bwd_workspace_size(ctypes.byref(p))
    assert ws == 8192 * 576 * 4 + 8192 * 64 * 4 + 8192 * 4    # accumulator, Delta, chunk counts
    args = [ctypes.c_void_p(FAKE)] * 8          # q kv idx o dout lse dq dkv
    assert L.sparse_attn_bwd(ctypes.byref(p), *args, ctypes.c_void_p(FAKE), ws - 1, None) == 5


def test_sparse_deterministic_workspace_and_validation(L):
    """Workspace of the deterministic sparse backward: one fp32 [tokens, 576]
    dKV slab per CTA of its main kernel (152, or one per (token, 64-head
    block) item when there are fewer), Delta and the chunk counts; each piece
    256-byte aligned.  Calls with a short workspace or bad shapes are refused
    before any launch."""
    a256 = lambda x: (x + 255) // 256 * 256
    p = _sparse()
    ws = L.sparse_attn_bwd_deterministic_workspace_size(ctypes.byref(p))
    assert ws == 152 * 8192 * 576 * 4 + 8192 * 64 * 4 + 8192 * 4
    # 128 heads: two head blocks per token; few items: one slab per item
    p2 = _sparse(tokens=50, heads=128, topk=64)
    assert L.sparse_attn_bwd_deterministic_workspace_size(ctypes.byref(p2)) == (
        a256(100 * 50 * 576 * 4) + a256(50 * 128 * 4) + a256(50 * 4))
    p3 = _sparse(tokens=100, heads=128, topk=64)
    assert L.sparse_attn_bwd_deterministic_workspace_size(ctypes.byref(p3)) == (
        a256(152 * 100 * 576 * 4) + a256(100 * 128 * 4) + a256(100 * 4))
    assert L.sparse_attn_bwd_deterministic_workspace_size(ctypes.byref(_sparse(heads=48))) == 0
    args = [ctypes.c_void_p(FAKE)] * 8          # q kv idx o dout lse dq dkv
    f = lambda q, *rest: L.sparse_attn_bwd_deterministic(ctypes.byref(q), *rest)
    assert f(p, *args, ctypes.c_void_p(FAKE), ws - 1, None) == 5
    assert f(_sparse(dim_v=256), *args, ctypes.c_void_p(FAKE), ws, None) == 2
    assert f(_sparse(tokens=0), *args, ctypes.c_void_p(FAKE), 0, None) == 0


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(A, "_LIB", None)
    monkeypatch.setattr(A, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        A.lib()


def _csa(**kw):
    p = A._CsaProblem()
    p.tokens, p.comp_capacity, p.num_seqs, p.head_dim, p.ratio, p.coff = 64, 16, 2, 128, 4, 2
    p.cu_seqlens, p.cu_seqlens_comp, p.error_word = FAKE, FAKE + 64, None
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _csa_fwd(L, p, ptrs=(FAKE,) * 4):
    return L.csa_compressor_fwd(ctypes.byref(p), *[ctypes.c_void_p(x) for x in ptrs], None)


def test_csa_compressor_validation(L):
    assert L.csa_compressor_fwd(None, *[ctypes.c_void_p(FAKE)] * 4, None) == 1
    assert _csa_fwd(L, _csa(coff=3)) == 2                       # coff outside {1, 2}
    assert _csa_fwd(L, _csa(ratio=3)) == 2                      # ratio outside {2, 4, 8}
    assert _csa_fwd(L, _csa(head_dim=100)) == 2                 # not a multiple of 64
    assert _csa_fwd(L, _csa(head_dim=2048)) == 2                # above 1024
    assert _csa_fwd(L, _csa(num_seqs=0)) == 1
    assert _csa_fwd(L, _csa(tokens=-1)) == 1
    assert _csa_fwd(L, _csa(cu_seqlens=None)) == 1
    assert _csa_fwd(L, _csa(cu_seqlens=FAKE + 2)) == 3           # int32 array misaligned
    assert _csa_fwd(L, _csa(tokens=1 << 22, head_dim=512)) == 2  # flat offsets past int32
    assert _csa_fwd(L, _csa(), (FAKE, 0, FAKE, FAKE)) == 1        # null score with tokens
    assert _csa_fwd(L, _csa(), (FAKE, FAKE + 8, FAKE, FAKE)) == 3
    assert _csa_fwd(L, _csa(comp_capacity=0)) == 0              # nothing to write
    # workspace: one fp32 slab of ratio * coff * head_dim per row group
    n = L.csa_compressor_bwd_workspace_size(ctypes.byref(_csa()))
    assert n > 0 and n % (4 * 2 * 128 * 4) == 0
    assert L.csa_compressor_bwd_workspace_size(ctypes.byref(_csa(coff=3))) == 0
    args = [ctypes.c_void_p(FAKE)] * 7
    assert L.csa_compressor_bwd(ctypes.byref(_csa()), *args, ctypes.c_void_p(FAKE), n - 4,
                                None) == 5
    assert L.csa_compressor_bwd(ctypes.byref(_csa()), *args, None, n, None) == 5


def test_wait_selftest_validation(L):
    v = ctypes.c_void_p(FAKE)
    assert L.attn_wait_selftest(None, 1000, v, None) == 1
    assert L.attn_wait_selftest(v, 0, v, None) == 1
    assert L.attn_wait_selftest(v, 2000000, v, None) == 1
