"""GB300 (sm_103a) fused exact-softmax attention backward.

Thin ctypes binding of the C ABI in ``include/fa.h`` (``libfa_gb300.so``,
built in-tree by ``attention_backward_preprocess_gb300.build``).  This module
only marshals arguments: every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback: when the library is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_ERR_SCRATCH_LIMIT = 5
FA_BF16, FA_FP16 = 0, 1

# entry points declared in include/fa.h and include/fa_selftest.h
EXPORTED = [
    "fa_bwd", "fa_bwd_workspace_bytes", "fa_bwd_with_workspace", "fa_bwd_preprocess",
    "fa_bwd_main", "fa_bwd_postprocess", "fa_bwd_workspace_layout", "fa_fwd",
    "fa_device_status", "fa_set_wait_timeout_ns", "fa_status_string",
    "fa_selftest_umma", "fa_selftest_semaphore", "fa_selftest_tmem_layout", "fa_bwd_noalloc",
    "fa_bwd_noalloc_scratch_bytes", "fa_fwd_ext", "fa_bwd_ext", "fa_bwd_stages_ext", "fa_bwd_workspace_sync_layout",
    "fa_bwd_noalloc_status",
]


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_SHAPE = [_i] * 6   # B, Sq, Sk, Hq, Hkv, D


class FaExt(ctypes.Structure):
    """fa_ext of include/fa.h: local window, ALiBi slopes, used lengths."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("alibi_slopes", ctypes.c_void_p), ("alibi_batch_stride", ctypes.c_int),
                ("seqused_q", ctypes.c_void_p), ("seqused_k", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("bias_batch_stride", ctypes.c_longlong),
                ("bias_head_stride", ctypes.c_longlong), ("bias_row_stride", ctypes.c_longlong),
                ("dbias", ctypes.c_void_p), ("dropout_p", ctypes.c_float),
                ("dropout_seed", ctypes.c_ulonglong), ("dropout_offset", ctypes.c_uint),
                ("dropout_mask", ctypes.c_void_p), ("total_q", ctypes.c_longlong),
                ("total_k", ctypes.c_longlong), ("head_dim_v", ctypes.c_int)]


def dropout_mask_shape(q, k, cu_seqlens_q=None, max_seqlen_k=None):
    """Shape of the int32 keep-flag buffer fa_fwd / fa_bwd take with dropout:
    [B, Hq, Sq, W] (dense) or [Hq, total_q, W] (varlen), W = ceil(Sk / 32)
    words of 32 keys per query row, Sk the key length (max_seqlen_k)."""
    if cu_seqlens_q is not None:
        Sk = int(max_seqlen_k)
        return (q.shape[1], q.shape[0], (Sk + 31) // 32)
    return (q.shape[0], q.shape[2], q.shape[1], (k.shape[1] + 31) // 32)


def _ext(Hq, window=None, alibi_slopes=None, seqused_q=None, seqused_k=None, bias=None,
         dbias=None, dropout=None, totals=None, head_dim_v=0):
    """A pointer to an FaExt, or None when no extension is asked for.

    ``bias``: [B or 1, Hq or 1, Sq, >= Sk] in the input dtype, last axis
    contiguous (a size-1 batch / head axis broadcasts).  ``dbias``: a
    contiguous [B, Hq, Sq, Sk] output of the input dtype (backward only).
    ``dropout``: (p, seed, offset), or (p, seed, offset, mask) with ``mask`` an
    int32 tensor of ``dropout_mask_shape(...)`` that fa_fwd fills with the keep
    flags and fa_bwd reads back; see fa_ext in include/fa.h.  ``totals``:
    (total_q, total_k), the packed row counts of a varlen call (cu_seqlens[B]),
    so that the library need not read them back (no stream synchronisation).
    ``head_dim_v``: the value head dim when it differs from q's (else 0)."""
    if (window is None and alibi_slopes is None and seqused_q is None and seqused_k is None
            and bias is None and dbias is None and dropout is None and totals is None
            and not head_dim_v):
        return None
    e = FaExt(-1, -1, None, 0, None, None, None, 0, 0, 0, None, 0.0, 0, 0, None, 0, 0, 0)
    e.head_dim_v = int(head_dim_v)
    if totals is not None:
        e.total_q, e.total_k = int(totals[0]), int(totals[1])
    if dropout is not None:
        e.dropout_p, e.dropout_seed, e.dropout_offset = (float(dropout[0]), int(dropout[1]),
                                                         int(dropout[2]))
        if len(dropout) > 3 and dropout[3] is not None:
            m = dropout[3]
            if m.dtype != torch.int32 or not m.is_contiguous():
                raise ValueError("dropout mask: a contiguous int32 tensor of dropout_mask_shape(...)")
            e.dropout_mask = m.data_ptr()
    if window is not None:
        e.window_left, e.window_right = int(window[0]), int(window[1])
    if alibi_slopes is not None:
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_contiguous():
            raise ValueError("alibi_slopes: contiguous fp32 [Hq] or [B, Hq]")
        e.alibi_slopes = alibi_slopes.data_ptr()
        e.alibi_batch_stride = Hq if alibi_slopes.dim() == 2 else 0
    for name, t in (("seqused_q", seqused_q), ("seqused_k", seqused_k)):
        if t is not None:
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(name + ": contiguous int32 [B]")
            setattr(e, name, t.data_ptr())
    if bias is not None:
        if bias.dim() != 4 or bias.stride(3) != 1:
            raise ValueError("bias: [B or 1, Hq or 1, Sq, Sk] with a contiguous last axis")
        e.bias = bias.data_ptr()
        e.bias_batch_stride = 0 if bias.shape[0] == 1 else bias.stride(0)
        e.bias_head_stride = 0 if bias.shape[1] == 1 else bias.stride(1)
        e.bias_row_stride = bias.stride(2)
    if dbias is not None:
        if not dbias.is_contiguous():
            raise ValueError("dbias: a contiguous [B, Hq, Sq, Sk] tensor")
        e.dbias = dbias.data_ptr()
    return ctypes.pointer(e)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libfa_gb300.so is not built (run attention_backward_preprocess_gb300.build."
                "build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        L.fa_bwd.argtypes = [_vp] * 9 + _SHAPE + [_f, _i, _vp, _vp, _i, _i, _vp]
        L.fa_bwd_workspace_bytes.argtypes = _SHAPE + [_i, _i]
        L.fa_bwd_workspace_bytes.restype = _sz
        L.fa_bwd_with_workspace.argtypes = ([_vp] * 9 + _SHAPE + [_f, _i, _vp, _vp, _i, _i, _vp,
                                                                  _sz, _vp])
        L.fa_bwd_preprocess.argtypes = [_vp] * 3 + _SHAPE + [_vp, _vp, _i, _i, _vp, _sz, _vp]
        L.fa_bwd_main.argtypes = [_vp] * 6 + _SHAPE + [_f, _i, _vp, _vp, _i, _i, _vp, _sz, _vp]
        L.fa_bwd_postprocess.argtypes = [_vp] + _SHAPE + [_f, _vp, _vp, _i, _i, _vp, _sz, _vp]
        L.fa_bwd_workspace_layout.argtypes = _SHAPE + [_i, _i] + [ctypes.POINTER(_sz)] * 4
        L.fa_fwd.argtypes = [_vp] * 5 + _SHAPE + [_f, _i, _vp, _vp, _i, _vp]
        _ep = ctypes.POINTER(FaExt)
        L.fa_fwd_ext.argtypes = [_vp] * 5 + _SHAPE + [_f, _i, _vp, _vp, _ep, _i, _vp]
        L.fa_bwd_ext.argtypes = ([_vp] * 9 + _SHAPE + [_f, _i, _vp, _vp, _ep, _i, _i, _vp, _sz,
                                                       _vp])
        L.fa_bwd_stages_ext.argtypes = ([_i] + [_vp] * 9 + _SHAPE +
                                        [_f, _i, _vp, _vp, _ep, _i, _i, _vp, _sz, _vp])
        L.fa_device_status.argtypes = [_vp, _vp]
        L.fa_set_wait_timeout_ns.argtypes = [ctypes.c_longlong]
        L.fa_set_wait_timeout_ns.restype = ctypes.c_longlong
        L.fa_status_string.argtypes = [_i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_bwd_noalloc.argtypes = [_vp] * 9 + _SHAPE + [_f, _i, _vp, _vp, _i, _i, _vp]
        L.fa_bwd_noalloc.restype = _i
        L.fa_bwd_noalloc_scratch_bytes.argtypes = []
        L.fa_bwd_noalloc_scratch_bytes.restype = _sz
        L.fa_bwd_noalloc_status.argtypes = [_vp]
        L.fa_bwd_noalloc_status.restype = _i
        L.fa_bwd_workspace_sync_layout.argtypes = _SHAPE + [_i, _i] + [ctypes.POINTER(_sz)] * 3
        L.fa_bwd_workspace_sync_layout.restype = _i
        L.fa_selftest_umma.argtypes = [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]
        L.fa_selftest_semaphore.argtypes = [_vp, _i, ctypes.c_longlong, _vp, _vp]
        L.fa_selftest_tmem_layout.argtypes = [_i, _vp, _vp]
        for name in ("fa_bwd", "fa_bwd_with_workspace", "fa_bwd_preprocess", "fa_bwd_main",
                     "fa_bwd_postprocess", "fa_bwd_workspace_layout", "fa_fwd", "fa_fwd_ext",
                     "fa_bwd_ext",
                     "fa_device_status", "fa_selftest_umma", "fa_selftest_semaphore",
                     "fa_selftest_tmem_layout"):
            getattr(L, name).restype = _i
        _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise ValueError("q/k/v/o/dout must be bf16 or fp16, got %s" % t.dtype)


def _shape(q, k, cu_q, max_seqlen_q, max_seqlen_k):
    """(B, Sq, Sk, Hq, Hkv, D) from dense [B,S,H,D] or packed [total,H,D] tensors."""
    if cu_q is None:
        if q.dim() != 4 or k.dim() != 4:
            raise ValueError("dense q/k are [B, S, H, D]")
        B, Sq, Hq, D = q.shape
        return B, Sq, k.shape[1], Hq, k.shape[2], D
    if q.dim() != 3 or k.dim() != 3 or max_seqlen_q is None or max_seqlen_k is None:
        raise ValueError("varlen q/k are [total, H, D] with max_seqlen_q / max_seqlen_k")
    return cu_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k), q.shape[1], k.shape[1], q.shape[2]


def _value_dim(D, v) -> int:
    """head_dim_v of fa_ext: v's last axis when it differs from the query /
    key head dim, else 0."""
    return 0 if v.shape[-1] == D else int(v.shape[-1])


def default_scale(D: int) -> float:
    return 1.0 / (D ** 0.5)


def fa_fwd(q, k, v, causal=False, softmax_scale=None, cu_seqlens_q=None, cu_seqlens_k=None,
           max_seqlen_q=None, max_seqlen_k=None, stream=None, window=None, alibi_slopes=None,
           seqused_q=None, seqused_k=None, bias=None, dropout=None, totals=None):
    """Forward pass: returns (o, lse); lse fp32 [B,Hq,Sq] or [Hq,total_q].

    ``window=(left, right)`` (-1 = unbounded side), ``alibi_slopes`` (fp32
    [Hq] or [B, Hq]), ``seqused_q`` / ``seqused_k`` (int32 [B]) and ``bias``
    (see ``_ext``) and ``dropout=(p, seed, offset)`` select fa_fwd_ext; rows
    past the used lengths are left as allocated.  ``totals=(total_q, total_k)``
    (varlen: cu_seqlens_q[B], cu_seqlens_k[B]) spares the read-back of the
    packed totals, so the call does not synchronise the stream.
    """
    B, Sq, Sk, Hq, Hkv, D = _shape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k)
    scale = default_scale(D) if softmax_scale is None else float(softmax_scale)
    o = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    if cu_seqlens_q is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    else:
        lse = torch.empty((Hq, q.shape[0]), dtype=torch.float32, device=q.device)
    ext = _ext(Hq, window, alibi_slopes, seqused_q, seqused_k, bias, dropout=dropout,
               totals=totals, head_dim_v=_value_dim(D, v))
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Sq, Sk, Hq, Hkv, D, scale,
            int(bool(causal)), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)]
    if ext is None:
        _check(lib().fa_fwd(*args, _dtype_code(q), _stream(stream)), "fa_fwd")
    else:
        _check(lib().fa_fwd_ext(*args, ext, _dtype_code(q), _stream(stream)), "fa_fwd_ext")
    return o, lse


def fa_bwd(q, k, v, o, dout, lse, causal=False, softmax_scale=None, cu_seqlens_q=None,
           cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, deterministic=False,
           dq=None, dk=None, dv=None, workspace=None, stream=None, window=None,
           alibi_slopes=None, seqused_q=None, seqused_k=None, bias=None, dbias=None,
           dropout=None, totals=None):
    """Backward pass through the C ABI; returns (dq, dk, dv).

    Outputs are allocated when not given.  ``workspace`` (a uint8 CUDA tensor
    of at least ``workspace_bytes(...)``) selects fa_bwd_with_workspace,
    otherwise the library's own workspace is used.  The extension keywords
    (as for fa_fwd, plus ``dbias``, an output tensor filled with dBias = dS)
    select fa_bwd_ext, and so does ``totals=(total_q, total_k)`` (varlen: the
    packed row counts, which spare the stream synchronisation of reading them
    back).
    """
    B, Sq, Sk, Hq, Hkv, D = _shape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k)
    scale = default_scale(D) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), B, Sq, Sk, Hq, Hkv, D, scale, int(bool(causal)), _ptr(cu_seqlens_q),
            _ptr(cu_seqlens_k), int(bool(deterministic)), _dtype_code(q)]
    ext = _ext(Hq, window, alibi_slopes, seqused_q, seqused_k, bias, dbias, dropout, totals,
               _value_dim(D, v))
    if ext is not None:
        st = lib().fa_bwd_ext(*args[:19], ext, *args[19:], _ptr(workspace),
                              0 if workspace is None else workspace.numel(), _stream(stream))
        _check(st, "fa_bwd_ext")
    elif workspace is None:
        st = lib().fa_bwd(*args, _stream(stream))
        _check(st, "fa_bwd")
    else:
        st = lib().fa_bwd_with_workspace(*args, _ptr(workspace), workspace.numel(),
                                          _stream(stream))
        _check(st, "fa_bwd_with_workspace")
    return dq, dk, dv


def noalloc_scratch_bytes() -> int:
    """Size of the fixed scratch array fa_bwd_noalloc works in."""
    return int(lib().fa_bwd_noalloc_scratch_bytes())


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, causal=False, softmax_scale=None,
                   cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
                   deterministic=False, stream=None) -> int:
    """fa_bwd without any device allocation, for callers that cannot allocate
    device memory at call time (its scratch is a fixed array inside the
    library; see include/fa.h).  The outputs must be given.  Returns the
    status (FA_OK, or FA_ERR_SCRATCH_LIMIT for a problem too large)."""
    B, Sq, Sk, Hq, Hkv, D = _shape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k)
    scale = default_scale(D) if softmax_scale is None else float(softmax_scale)
    return int(lib().fa_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, Sq, Sk, Hq, Hkv, D, scale, int(bool(causal)), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k), int(bool(deterministic)), _dtype_code(q), _stream(stream)))


def noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the error status of
    the fixed scratch array fa_bwd_noalloc works in."""
    return int(lib().fa_bwd_noalloc_status(_stream(stream)))


def workspace_sync_layout(B, Sq, Sk, Hq, Hkv, D, varlen=False, deterministic=False) -> dict:
    """Byte offsets of the error word and of the deterministic-order
    semaphores inside a workspace, and the number of semaphores."""
    vals = [_sz() for _ in range(3)]
    st = lib().fa_bwd_workspace_sync_layout(B, Sq, Sk, Hq, Hkv, D, int(bool(varlen)),
                                            int(bool(deterministic)),
                                            *[ctypes.byref(x) for x in vals])
    _check(st, "fa_bwd_workspace_sync_layout")
    return dict(err=vals[0].value, sem=vals[1].value, n_sem=vals[2].value)


def workspace_bytes(B, Sq, Sk, Hq, Hkv, D, varlen=False, deterministic=False) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Sq, Sk, Hq, Hkv, D, int(bool(varlen)),
                                            int(bool(deterministic))))


def workspace_layout(B, Sq, Sk, Hq, Hkv, D, varlen=False, deterministic=False) -> dict:
    """fp32-element offsets of Dv, LSE2 and the dQ accumulator inside a workspace."""
    vals = [_sz() for _ in range(4)]
    st = lib().fa_bwd_workspace_layout(B, Sq, Sk, Hq, Hkv, D, int(bool(varlen)),
                                       int(bool(deterministic)), *[ctypes.byref(x) for x in vals])
    _check(st, "fa_bwd_workspace_layout")
    return dict(dvec=vals[0].value, lse2=vals[1].value, dqacc=vals[2].value, rows=vals[3].value)


def fa_bwd_stages(q, k, v, o, dout, lse, workspace, causal=False, softmax_scale=None,
                  cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
                  deterministic=False, dq=None, dk=None, dv=None, stages=("pre", "main", "post"),
                  stream=None, totals=None):
    """Runs the chosen stages (preprocess / main / postprocess) on ``workspace``.

    ``totals=(total_q, total_k)`` (varlen) goes through fa_bwd_stages_ext with
    the packed row counts, so that no stage synchronises the stream."""
    B, Sq, Sk, Hq, Hkv, D = _shape(q, k, cu_seqlens_q, max_seqlen_q, max_seqlen_k)
    scale = default_scale(D) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    shape = [B, Sq, Sk, Hq, Hkv, D]
    if totals is not None:
        mask = ((1 if "pre" in stages else 0) | (2 if "main" in stages else 0) |
                (4 if "post" in stages else 0))
        ext = _ext(Hq, totals=totals)
        _check(lib().fa_bwd_stages_ext(mask, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                                       _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), *shape, scale,
                                       int(bool(causal)), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                       ext, int(bool(deterministic)), _dtype_code(q),
                                       _ptr(workspace), workspace.numel(), _stream(stream)),
               "fa_bwd_stages_ext")
        return dq, dk, dv
    cu = [_ptr(cu_seqlens_q), _ptr(cu_seqlens_k)]
    det, dt = int(bool(deterministic)), _dtype_code(q)
    ws = [_ptr(workspace), workspace.numel(), _stream(stream)]
    L = lib()
    if "pre" in stages:
        _check(L.fa_bwd_preprocess(_ptr(o), _ptr(dout), _ptr(lse), *shape, *cu, det, dt, *ws),
               "fa_bwd_preprocess")
    if "main" in stages:
        _check(L.fa_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dk), _ptr(dv), *shape,
                             scale,
                             int(bool(causal)), *cu, det, dt, *ws), "fa_bwd_main")
    if "post" in stages:
        _check(L.fa_bwd_postprocess(_ptr(dq), *shape, scale, *cu, det, dt, *ws),
               "fa_bwd_postprocess")
    return dq, dk, dv


def device_status(workspace=None, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(lib().fa_device_status(_ptr(workspace), _stream(stream)))


def set_wait_timeout_ns(ns: int) -> int:
    return int(lib().fa_set_wait_timeout_ns(int(ns)))


def selftest_umma(mode: int, A: torch.Tensor, B: torch.Tensor, N: int, K: int, stream=None):
    """One-CTA tcgen05 GEMM in one of the kernel's operand forms (see fa_selftest.h)."""
    C = torch.empty((128, N), dtype=torch.float32, device=A.device)
    err = torch.zeros(1, dtype=torch.int32, device=A.device)
    st = lib().fa_selftest_umma(mode, N, K, int(A.dtype == torch.bfloat16), _ptr(A), _ptr(B),
                                _ptr(C), _ptr(err), _stream(stream))
    if st != 0:
        raise RuntimeError("fa_selftest_umma returned %d" % st)
    return C, err


def selftest_tmem_layout(which: int, device="cuda", stream=None):
    """The 16-lane tensor-memory access shapes' layout probe (see fa_selftest.h);
    returns the [128, 32] uint32 result as int64."""
    out = torch.zeros((128, 32), dtype=torch.int32, device=device)
    st = lib().fa_selftest_tmem_layout(int(which), _ptr(out), _stream(stream))
    if st != 0:
        raise RuntimeError("fa_selftest_tmem_layout returned %d" % st)
    return out.cpu().to(torch.int64) & 0xFFFFFFFF


def selftest_semaphore(sem: torch.Tensor, target: int, budget_ns: int, stream=None):
    err = torch.zeros(1, dtype=torch.int32, device=sem.device)
    st = lib().fa_selftest_semaphore(_ptr(sem), int(target), int(budget_ns), _ptr(err),
                                     _stream(stream))
    if st != 0:
        raise RuntimeError("fa_selftest_semaphore returned %d" % st)
    return err
