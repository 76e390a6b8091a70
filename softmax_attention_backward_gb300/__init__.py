"""GB300 softmax-attention training kernels: thin Python binding of libattn.so.

Every function here only marshals torch tensors (device memory and the current
stream) into the C ABI declared in include/attn.h; all arithmetic runs in the
library's CUDA kernels.  There is no CPU or eager fallback: if the library is
missing or a call fails, an exception is raised.

Entry points (same names as the C ABI):
  attn_fwd, attn_bwd_workspace_size, attn_bwd_preprocess, attn_bwd, attn_bwd_postprocess,
  sparse_attn_fwd, sparse_attn_bwd_workspace_size, sparse_attn_bwd,
  sparse_attn_bwd_deterministic_workspace_size, sparse_attn_bwd_deterministic,
  attn_bwd_fixed_scratch, attn_status_string, attn_version   (include/attn.h)
  dsa_indexer_fwd, dsa_topk, dsa_indexer_bwd_workspace_size, dsa_indexer_bwd, dsa_sparse_kl,
  csa_compressor_fwd, csa_compressor_bwd_workspace_size, csa_compressor_bwd  (include/dsa.h)
"""
from __future__ import annotations

import ctypes
import math
import os
import warnings

import torch

__all__ = [
    "ATTN_DQ_ATOMIC", "ATTN_DQ_SPLIT", "AttnError", "lib", "attn_fwd", "attn_bwd_workspace_size",
    "attn_bwd_preprocess", "attn_bwd", "attn_bwd_postprocess", "sparse_attn_fwd", "sparse_attn_bwd_workspace_size",
    "sparse_attn_bwd", "sparse_attn_bwd_deterministic_workspace_size", "sparse_attn_bwd_deterministic",
    "attn_status_string", "attn_version", "dense_backward",
    "SPARSE_DIM_QK", "SPARSE_DIM_V", "EXPORTED_SYMBOLS", "attn_bwd_fixed_scratch",
    "FIXED_SCRATCH_BYTES", "csa_compressor_fwd", "csa_compressor_bwd_workspace_size",
    "csa_compressor_bwd", "dsa_indexer_fwd", "dsa_topk", "dsa_indexer_bwd_workspace_size",
    "dsa_indexer_bwd", "dsa_sparse_kl", "INDEXER_HEAD_DIM", "attn_wait_selftest",
]

ATTN_DQ_ATOMIC = 0
ATTN_DQ_SPLIT = 1
SPARSE_DIM_QK = 576
SPARSE_DIM_V = 512
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")

EXPORTED_SYMBOLS = (
    "attn_fwd", "attn_bwd_workspace_size", "attn_bwd_preprocess", "attn_bwd", "attn_bwd_postprocess",
    "sparse_attn_fwd", "sparse_attn_bwd_workspace_size", "sparse_attn_bwd",
    "sparse_attn_bwd_deterministic_workspace_size", "sparse_attn_bwd_deterministic",
    "attn_status_string", "attn_version", "attn_bwd_fixed_scratch",
    "csa_compressor_fwd", "csa_compressor_bwd_workspace_size", "csa_compressor_bwd",
    "dsa_indexer_fwd", "dsa_topk", "dsa_indexer_bwd_workspace_size", "dsa_indexer_bwd",
    "dsa_sparse_kl", "attn_wait_selftest",
)
INDEXER_HEAD_DIM = 128
FIXED_SCRATCH_BYTES = 16 << 20


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {attn_status_string(code)} (status {code})")
        self.code = code


class _Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("heads_q", ctypes.c_int),
        ("heads_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("causal", ctypes.c_int),
        ("scale", ctypes.c_float), ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
        ("capacity", ctypes.c_int), ("max_seqlen", ctypes.c_int), ("error_word", ctypes.c_void_p),
    ]


class _SparseProblem(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int), ("heads", ctypes.c_int), ("dim_qk", ctypes.c_int),
        ("dim_v", ctypes.c_int), ("topk", ctypes.c_int), ("scale", ctypes.c_float),
        ("error_word", ctypes.c_void_p),
    ]


class _CsaProblem(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int), ("comp_capacity", ctypes.c_int), ("num_seqs", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("ratio", ctypes.c_int), ("coff", ctypes.c_int),
        ("cu_seqlens", ctypes.c_void_p), ("cu_seqlens_comp", ctypes.c_void_p),
        ("error_word", ctypes.c_void_p),
    ]


class _IndexerProblem(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("topk", ctypes.c_int), ("use_relu", ctypes.c_int), ("logits_ld", ctypes.c_int),
        ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
        ("error_word", ctypes.c_void_p),
    ]


_LIB = None


def lib() -> ctypes.CDLL:
    """Loads libattn.so (built by __graft_entry__.build() or build.py)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m softmax_attention_backward_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        P = ctypes.POINTER(_Problem)
        SP = ctypes.POINTER(_SparseProblem)
        L.attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp]
        L.attn_bwd_workspace_size.argtypes = [P, i32]
        L.attn_bwd_workspace_size.restype = sz
        L.attn_bwd_preprocess.argtypes = [P, i32, vp, vp, vp, vp, sz, vp]
        L.attn_bwd.argtypes = [P, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_bwd_postprocess.argtypes = [P, i32, vp, sz, vp, vp, vp, vp]
        L.sparse_attn_fwd.argtypes = [SP, vp, vp, vp, vp, vp, vp]
        L.sparse_attn_bwd_workspace_size.argtypes = [SP]
        L.sparse_attn_bwd_workspace_size.restype = sz
        L.sparse_attn_bwd.argtypes = [SP, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.sparse_attn_bwd_deterministic_workspace_size.argtypes = [SP]
        L.sparse_attn_bwd_deterministic_workspace_size.restype = sz
        L.sparse_attn_bwd_deterministic.argtypes = [SP, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_bwd_fixed_scratch.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        CP = ctypes.POINTER(_CsaProblem)
        L.csa_compressor_fwd.argtypes = [CP, vp, vp, vp, vp, vp]
        L.csa_compressor_bwd_workspace_size.argtypes = [CP]
        L.csa_compressor_bwd_workspace_size.restype = sz
        L.csa_compressor_bwd.argtypes = [CP, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        IP = ctypes.POINTER(_IndexerProblem)
        L.dsa_indexer_fwd.argtypes = [IP, vp, vp, vp, vp, vp]
        L.dsa_topk.argtypes = [IP, vp, vp, vp, vp, vp]
        L.dsa_indexer_bwd_workspace_size.argtypes = [IP]
        L.dsa_indexer_bwd_workspace_size.restype = sz
        L.dsa_indexer_bwd.argtypes = [IP, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.dsa_sparse_kl.argtypes = [SP, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.attn_wait_selftest.argtypes = [vp, ctypes.c_uint, vp, vp]
        L.attn_wait_selftest.restype = i32
        L.attn_status_string.argtypes = [i32]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_version.argtypes = []
        for name in ("attn_fwd", "attn_bwd_preprocess", "attn_bwd", "attn_bwd_postprocess",
                     "sparse_attn_fwd", "sparse_attn_bwd", "attn_bwd_fixed_scratch",
                     "csa_compressor_fwd", "csa_compressor_bwd", "dsa_indexer_fwd", "dsa_topk",
                     "dsa_indexer_bwd", "dsa_sparse_kl"):
            getattr(L, name).restype = i32
        _LIB = L
    return _LIB


def attn_status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def attn_version() -> int:
    return int(lib().attn_version())


def attn_wait_selftest(limit_us=1000, *, device=None, stream=None):
    """Runs the bounded-wait self-test; returns (result bits, error word)
    after synchronizing (7 and ATTN_DEVERR_TIMEOUT when the mechanism works)."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    res = torch.full((1,), -1, dtype=torch.int32, device=dev)
    _check("attn_wait_selftest", lib().attn_wait_selftest(_ptr(err), int(limit_us), _ptr(res),
                                                          _stream(stream)))
    torch.cuda.synchronize(dev)
    return int(res.item()), int(err.item())


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != 0:
        raise AttnError(fn, code)


def _need(t, name, dtype, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _nondeterministic(what: str, instead: str):
    if torch.are_deterministic_algorithms_enabled():
        msg = f"{what} accumulates with fp32 atomics and is not bitwise reproducible"
        if torch.is_deterministic_algorithms_warn_only_enabled():
            warnings.warn(msg, RuntimeWarning, stacklevel=3)
        else:
            raise RuntimeError(f"{msg}; use {instead}")


def _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word):
    p = _Problem()
    if cu_seqlens is None:
        if q.dim() != 4:
            raise ValueError("dense q must be [batch, seqlen, heads, head_dim]")
        p.batch, p.seqlen, p.heads_q, p.head_dim = q.shape
        p.heads_kv = k.shape[2]
        p.cu_seqlens = None
        p.num_seqs = 0
        p.capacity = 0
        p.max_seqlen = q.shape[1]
    else:
        if q.dim() != 3:
            raise ValueError("THD q must be [capacity, heads, head_dim]")
        _need(cu_seqlens, "cu_seqlens", torch.int32, q.device)
        p.batch, p.seqlen = 1, 0
        p.capacity, p.heads_q, p.head_dim = q.shape
        p.heads_kv = k.shape[1]
        p.cu_seqlens = cu_seqlens.data_ptr()
        p.num_seqs = cu_seqlens.numel() - 1
        if max_seqlen is None:
            # Deriving it from cu_seqlens would read device memory on the host: a
            # hidden synchronisation, and a stale value under graph capture.
            raise ValueError("THD calls need max_seqlen, an upper bound on every "
                             "sequence length (the host never reads cu_seqlens)")
        p.max_seqlen = int(max_seqlen)
    p.causal = 1 if causal else 0
    p.scale = float(scale if scale is not None else 1.0 / math.sqrt(p.head_dim))
    p.error_word = None if error_word is None else error_word.data_ptr()
    return p


def _lse_shape(q, cu_seqlens):
    if cu_seqlens is None:
        return (q.shape[0], q.shape[2], q.shape[1])
    return (q.shape[1], q.shape[0])


# ----------------------------------------------------------------------------
# dense / THD
# ----------------------------------------------------------------------------
def attn_fwd(q, k, v, *, causal=False, scale=None, cu_seqlens=None, max_seqlen=None, out=None,
             lse=None, error_word=None, stream=None):
    """Returns (o, lse).  Dense: q [B,S,Hq,D], k/v [B,S,Hkv,D], lse [B,Hq,S].
    THD: q [cap,Hq,D], k/v [cap,Hkv,D], cu_seqlens int32 [n+1], lse [Hq,cap]."""
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, torch.bfloat16, dev)
    o = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty(_lse_shape(q, cu_seqlens), dtype=torch.float32,
                                                  device=dev)
    _need(o, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word)
    _check("attn_fwd", lib().attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(lse), _stream(stream)))
    return o, lse


def attn_bwd_workspace_size(q, k, *, mode=ATTN_DQ_ATOMIC, causal=False, cu_seqlens=None,
                            max_seqlen=None, scale=None) -> int:
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, None)
    return int(lib().attn_bwd_workspace_size(ctypes.byref(p), int(mode)))


def attn_bwd_preprocess(q, k, o, dout, *, mode=ATTN_DQ_ATOMIC, workspace=None, causal=False,
                        scale=None, cu_seqlens=None, max_seqlen=None, delta=None,
                        error_word=None, stream=None):
    """Returns delta = rowsum(dO * O) (fp32, layout of lse); clears the atomic
    dQ accumulator inside `workspace` (a uint8 CUDA tensor)."""
    dev = q.device
    _need(o, "o", torch.bfloat16, dev)
    _need(dout, "dout", torch.bfloat16, dev)
    delta = delta if delta is not None else torch.empty(_lse_shape(q, cu_seqlens),
                                                        dtype=torch.float32, device=dev)
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel())
    _check("attn_bwd_preprocess",
           lib().attn_bwd_preprocess(ctypes.byref(p), int(mode), _ptr(o), _ptr(dout), _ptr(delta),
                                     ws_ptr, ws_bytes, _stream(stream)))
    return delta


def attn_bwd(q, k, v, dout, lse, delta, *, mode=ATTN_DQ_ATOMIC, workspace, causal=False,
             scale=None, cu_seqlens=None, max_seqlen=None, dk=None, dv=None, error_word=None,
             stream=None):
    """Main backward pass: returns (dk, dv) bf16 and leaves dQ (fp32) in the
    workspace.  Call attn_bwd_preprocess before and attn_bwd_postprocess after,
    with the same workspace and mode."""
    if int(mode) == ATTN_DQ_ATOMIC:
        _nondeterministic("attn_bwd(dq_mode=ATTN_DQ_ATOMIC)", "dq_mode=ATTN_DQ_SPLIT")
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _need(t, n, torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    _need(delta, "delta", torch.float32, dev)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word)
    _check("attn_bwd",
           lib().attn_bwd(ctypes.byref(p), int(mode), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                          _ptr(lse), _ptr(delta), _ptr(dk), _ptr(dv), _ptr(workspace),
                          workspace.numel(), _stream(stream)))
    return dk, dv


def attn_bwd_postprocess(q, k, dk, dv, *, mode=ATTN_DQ_ATOMIC, workspace, causal=False, scale=None,
                         cu_seqlens=None, max_seqlen=None, dq=None, error_word=None, stream=None):
    """Writes dq (bf16) from the workspace of attn_bwd; returns dq."""
    dq = dq if dq is not None else torch.empty_like(q)
    _need(dq, "dq", torch.bfloat16, q.device)
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word)
    _check("attn_bwd_postprocess",
           lib().attn_bwd_postprocess(ctypes.byref(p), int(mode), _ptr(workspace),
                                      workspace.numel(), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _stream(stream)))
    return dq


def dense_backward(q, k, v, o, lse, dout, *, mode=ATTN_DQ_ATOMIC, causal=False, scale=None,
                   cu_seqlens=None, max_seqlen=None, workspace=None, error_word=None,
                   stream=None):
    """Preprocess + backward with a workspace allocated here when not given."""
    if workspace is None:
        n = attn_bwd_workspace_size(q, k, mode=mode, causal=causal, cu_seqlens=cu_seqlens,
                                    max_seqlen=max_seqlen)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    kw = dict(mode=mode, causal=causal, scale=scale, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen,
              error_word=error_word, stream=stream)
    delta = attn_bwd_preprocess(q, k, o, dout, workspace=workspace, **kw)
    dk, dv = attn_bwd(q, k, v, dout, lse, delta, workspace=workspace, **kw)
    dq = attn_bwd_postprocess(q, k, dk, dv, workspace=workspace, **kw)
    return dq, dk, dv


def attn_bwd_fixed_scratch(q, k, v, o, dout, lse, *, causal=False, scale=None, cu_seqlens=None,
                           max_seqlen=None, dq=None, dk=None, dv=None, error_word=None,
                           stream=None):
    """Backward for callers that cannot allocate device memory: no workspace
    argument; Delta and the fp32 dQ accumulator live in a 16 MiB array the
    library owns on each GPU.  Returns (dq, dk, dv).  Problems whose scratch
    need exceeds the array raise ValueError; calls that overlap on the GPU race
    on the shared array."""
    _nondeterministic("attn_bwd_fixed_scratch", "attn_bwd with dq_mode=ATTN_DQ_SPLIT")
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need(t, n, torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    rows = q.shape[0] if cu_seqlens is not None else q.shape[0] * q.shape[1]
    hq, d = q.shape[-2], q.shape[-1]
    need = (rows * hq * d * 4 + 255) // 256 * 256 + rows * hq * 4
    if need > FIXED_SCRATCH_BYTES:
        raise ValueError(f"attn_bwd_fixed_scratch: problem needs {need} bytes of scratch, "
                         f"more than the fixed {FIXED_SCRATCH_BYTES}")
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    p = _problem(q, k, causal, scale, cu_seqlens, max_seqlen, error_word)
    _check("attn_bwd_fixed_scratch",
           lib().attn_bwd_fixed_scratch(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                        _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                        _stream(stream)))
    return dq, dk, dv


# ----------------------------------------------------------------------------
# top-k sparse
# ----------------------------------------------------------------------------
def _sparse_problem(q, idx, scale, error_word):
    p = _SparseProblem()
    p.tokens, p.heads, p.dim_qk = q.shape
    p.dim_v = SPARSE_DIM_V
    p.topk = idx.shape[1]
    p.scale = float(scale if scale is not None else 1.0 / math.sqrt(p.dim_qk))
    p.error_word = None if error_word is None else error_word.data_ptr()
    return p


def sparse_attn_fwd(q, kv, idx, *, scale=None, out=None, lse=None, error_word=None, stream=None):
    """q [T,H,576], kv [T,576], idx int32 [T,K] -> (o [T,H,512], lse [T,H])."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(kv, "kv", torch.bfloat16, dev)
    _need(idx, "idx", torch.int32, dev)
    T, H, _ = q.shape
    o = out if out is not None else torch.empty(T, H, SPARSE_DIM_V, dtype=torch.bfloat16, device=dev)
    lse = lse if lse is not None else torch.empty(T, H, dtype=torch.float32, device=dev)
    p = _sparse_problem(q, idx, scale, error_word)
    _check("sparse_attn_fwd",
           lib().sparse_attn_fwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(o), _ptr(lse),
                                 _stream(stream)))
    return o, lse


def sparse_attn_bwd_workspace_size(q, idx, *, scale=None) -> int:
    p = _sparse_problem(q, idx, scale, None)
    return int(lib().sparse_attn_bwd_workspace_size(ctypes.byref(p)))


def sparse_attn_bwd(q, kv, idx, o, dout, lse, *, scale=None, workspace=None, dq=None, dkv=None,
                    error_word=None, stream=None):
    """Returns (dq [T,H,576], dkv [T,576]) bf16."""
    _nondeterministic("sparse_attn_bwd (dKV)", "sparse_attn_bwd_deterministic")
    dev = q.device
    for n, t in (("q", q), ("kv", kv), ("o", o), ("dout", dout)):
        _need(t, n, torch.bfloat16, dev)
    _need(idx, "idx", torch.int32, dev)
    _need(lse, "lse", torch.float32, dev)
    if workspace is None:
        n = sparse_attn_bwd_workspace_size(q, idx, scale=scale)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    dq = dq if dq is not None else torch.empty_like(q)
    dkv = dkv if dkv is not None else torch.empty_like(kv)
    p = _sparse_problem(q, idx, scale, error_word)
    _check("sparse_attn_bwd",
           lib().sparse_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx), _ptr(o),
                                 _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dkv), _ptr(workspace),
                                 workspace.numel(), _stream(stream)))
    return dq, dkv


def sparse_attn_bwd_deterministic_workspace_size(q, idx, *, scale=None) -> int:
    p = _sparse_problem(q, idx, scale, None)
    return int(lib().sparse_attn_bwd_deterministic_workspace_size(ctypes.byref(p)))


def sparse_attn_bwd_deterministic(q, kv, idx, o, dout, lse, *, scale=None, workspace=None, dq=None,
                                  dkv=None, error_word=None, stream=None):
    """Returns (dq [T,H,576], dkv [T,576]) bf16 with dkv bitwise reproducible
    (fixed per-key-row summation order; see include/attn.h for the workspace)."""
    dev = q.device
    for n, t in (("q", q), ("kv", kv), ("o", o), ("dout", dout)):
        _need(t, n, torch.bfloat16, dev)
    _need(idx, "idx", torch.int32, dev)
    _need(lse, "lse", torch.float32, dev)
    if workspace is None:
        n = sparse_attn_bwd_deterministic_workspace_size(q, idx, scale=scale)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    dq = dq if dq is not None else torch.empty_like(q)
    dkv = dkv if dkv is not None else torch.empty_like(kv)
    p = _sparse_problem(q, idx, scale, error_word)
    _check("sparse_attn_bwd_deterministic",
           lib().sparse_attn_bwd_deterministic(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(idx),
                                               _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dkv),
                                               _ptr(workspace), workspace.numel(), _stream(stream)))
    return dq, dkv


# ----------------------------------------------------------------------------
# CSA compressor gated pooling (include/dsa.h)
# ----------------------------------------------------------------------------
def _csa_problem(kv, cu_seqlens, cu_seqlens_comp, ratio, coff, comp_capacity, error_word):
    p = _CsaProblem()
    if kv.dim() != 2 or kv.shape[1] % coff:
        raise ValueError("kv must be [tokens, coff * head_dim]")
    _need(cu_seqlens, "cu_seqlens", torch.int32, kv.device)
    _need(cu_seqlens_comp, "cu_seqlens_comp", torch.int32, kv.device)
    if cu_seqlens.numel() != cu_seqlens_comp.numel():
        raise ValueError("cu_seqlens and cu_seqlens_comp must have the same length")
    p.tokens = kv.shape[0]
    p.comp_capacity = int(comp_capacity)
    p.num_seqs = cu_seqlens.numel() - 1
    p.head_dim = kv.shape[1] // coff
    p.ratio, p.coff = int(ratio), int(coff)
    p.cu_seqlens = cu_seqlens.data_ptr()
    p.cu_seqlens_comp = cu_seqlens_comp.data_ptr()
    p.error_word = None if error_word is None else error_word.data_ptr()
    return p


def csa_compressor_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, *, ratio=4, coff=2,
                       comp_capacity, out=None, error_word=None, stream=None):
    """kv/score bf16 [T, coff*D], ape fp32 [ratio, coff*D] -> out bf16 [comp_capacity, D]."""
    dev = kv.device
    _need(kv, "kv", torch.bfloat16, dev)
    _need(score, "score", torch.bfloat16, dev)
    _need(ape, "ape", torch.float32, dev)
    p = _csa_problem(kv, cu_seqlens, cu_seqlens_comp, ratio, coff, comp_capacity, error_word)
    out = out if out is not None else torch.empty(p.comp_capacity, p.head_dim,
                                                  dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _check("csa_compressor_fwd",
           lib().csa_compressor_fwd(ctypes.byref(p), _ptr(kv), _ptr(score), _ptr(ape), _ptr(out),
                                    _stream(stream)))
    return out


def csa_compressor_bwd_workspace_size(kv, cu_seqlens, cu_seqlens_comp, *, ratio=4, coff=2,
                                      comp_capacity) -> int:
    p = _csa_problem(kv, cu_seqlens, cu_seqlens_comp, ratio, coff, comp_capacity, None)
    return int(lib().csa_compressor_bwd_workspace_size(ctypes.byref(p)))


def csa_compressor_bwd(kv, score, ape, dout, cu_seqlens, cu_seqlens_comp, *, ratio=4, coff=2,
                       workspace=None, dkv=None, dscore=None, dape=None, error_word=None,
                       stream=None):
    """Returns (dkv, dscore) bf16 [T, coff*D] and dape fp32 [ratio, coff*D], all
    bitwise reproducible."""
    dev = kv.device
    for n, t in (("kv", kv), ("score", score), ("dout", dout)):
        _need(t, n, torch.bfloat16, dev)
    _need(ape, "ape", torch.float32, dev)
    p = _csa_problem(kv, cu_seqlens, cu_seqlens_comp, ratio, coff, dout.shape[0], error_word)
    if workspace is None:
        n = int(lib().csa_compressor_bwd_workspace_size(ctypes.byref(p)))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    dkv = dkv if dkv is not None else torch.empty_like(kv)
    dscore = dscore if dscore is not None else torch.empty_like(score)
    dape = dape if dape is not None else torch.empty_like(ape)
    _check("csa_compressor_bwd",
           lib().csa_compressor_bwd(ctypes.byref(p), _ptr(kv), _ptr(score), _ptr(ape), _ptr(dout),
                                    _ptr(dkv), _ptr(dscore), _ptr(dape), _ptr(workspace),
                                    workspace.numel(), _stream(stream)))
    return dkv, dscore, dape


# ----------------------------------------------------------------------------
# DSA lightning indexer, top-k and sparse KL (include/dsa.h)
# ----------------------------------------------------------------------------
def logits_ld(tokens: int) -> int:
    """Row stride of the logits buffer: tokens rounded up to a multiple of 4."""
    return (int(tokens) + 3) // 4 * 4


def _indexer_problem(q, topk, use_relu, cu_seqlens, error_word, ld=None):
    p = _IndexerProblem()
    if q.dim() != 3:
        raise ValueError("indexer q must be [tokens, heads, head_dim]")
    p.tokens, p.heads, p.head_dim = q.shape
    p.topk = int(topk)
    p.use_relu = 1 if use_relu else 0
    p.logits_ld = logits_ld(p.tokens) if ld is None else int(ld)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, q.device)
        p.cu_seqlens = cu_seqlens.data_ptr()
        p.num_seqs = cu_seqlens.numel() - 1
    else:
        p.cu_seqlens, p.num_seqs = None, 0
    p.error_word = None if error_word is None else error_word.data_ptr()
    return p


def dsa_indexer_fwd(q, k, w, *, use_relu=True, cu_seqlens=None, logits=None, error_word=None,
                    stream=None):
    """q bf16 [T,H,128], k bf16 [T,128], w fp32 [T,H] -> logits fp32 [T, logits_ld(T)]
    (columns past T unwritten; use logits[:, :T])."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", torch.bfloat16, dev)
    _need(w, "w", torch.float32, dev)
    p = _indexer_problem(q, 1, use_relu, cu_seqlens, error_word)
    if logits is None:
        logits = torch.empty(p.tokens, p.logits_ld, dtype=torch.float32, device=dev)
    _need(logits, "logits", torch.float32, dev)
    p.logits_ld = logits.shape[1]
    _check("dsa_indexer_fwd", lib().dsa_indexer_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w),
                                                    _ptr(logits), _stream(stream)))
    return logits


def dsa_topk(logits, topk, *, heads=1, cu_seqlens=None, idx=None, length=None, scores=None,
             error_word=None, stream=None):
    """logits fp32 [T, ld] -> (idx int32 [T,topk], length int32 [T], scores fp32 [T,topk])."""
    dev = logits.device
    _need(logits, "logits", torch.float32, dev)
    T = logits.shape[0]
    p = _IndexerProblem()
    p.tokens, p.heads, p.head_dim, p.topk = T, int(heads), INDEXER_HEAD_DIM, int(topk)
    p.use_relu, p.logits_ld = 1, logits.shape[1]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        p.cu_seqlens, p.num_seqs = cu_seqlens.data_ptr(), cu_seqlens.numel() - 1
    else:
        p.cu_seqlens, p.num_seqs = None, 0
    p.error_word = None if error_word is None else error_word.data_ptr()
    idx = idx if idx is not None else torch.empty(T, topk, dtype=torch.int32, device=dev)
    length = length if length is not None else torch.empty(T, dtype=torch.int32, device=dev)
    scores = scores if scores is not None else torch.empty(T, topk, dtype=torch.float32, device=dev)
    _check("dsa_topk", lib().dsa_topk(ctypes.byref(p), _ptr(logits), _ptr(idx), _ptr(length),
                                      _ptr(scores), _stream(stream)))
    return idx, length, scores


def dsa_indexer_bwd(q, k, w, idx, grad, *, use_relu=True, workspace=None, dq=None, dk=None,
                    dw=None, error_word=None, stream=None):
    """Gradients (dq bf16 [T,H,128], dk bf16 [T,128], dw fp32 [T,H]) of
    sum_j grad[t, j] * logits[t, idx[t, j]]."""
    _nondeterministic("dsa_indexer_bwd (dk)", "a reproducible reduction of dk")
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", torch.bfloat16, dev)
    _need(w, "w", torch.float32, dev)
    _need(idx, "idx", torch.int32, dev)
    _need(grad, "grad", torch.float32, dev)
    p = _indexer_problem(q, idx.shape[1], use_relu, None, error_word)
    if workspace is None:
        n = int(lib().dsa_indexer_bwd_workspace_size(ctypes.byref(p)))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dw = dw if dw is not None else torch.empty_like(w)
    _check("dsa_indexer_bwd",
           lib().dsa_indexer_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(w), _ptr(idx), _ptr(grad),
                                 _ptr(dq), _ptr(dk), _ptr(dw), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))
    return dq, dk, dw


def dsa_sparse_kl(q, kv, lse, idx, scores, *, scale=None, loss=None, grad=None, target=None,
                  want_target=False, error_word=None, stream=None):
    """Sparse KL of the attention target from softmax(scores) per token:
    returns (loss fp32 [T], grad fp32 [T,K], target fp32 [T,K] or None)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(kv, "kv", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    _need(idx, "idx", torch.int32, dev)
    _need(scores, "scores", torch.float32, dev)
    T = q.shape[0]
    p = _sparse_problem(q, idx, scale, error_word)
    loss = loss if loss is not None else torch.empty(T, dtype=torch.float32, device=dev)
    grad = grad if grad is not None else torch.empty_like(scores)
    if want_target and target is None:
        target = torch.empty_like(scores)
    _check("dsa_sparse_kl",
           lib().dsa_sparse_kl(ctypes.byref(p), _ptr(q), _ptr(kv), _ptr(lse), _ptr(idx),
                               _ptr(scores), _ptr(loss), _ptr(grad), _ptr(target), _stream(stream)))
    return loss, grad, target
