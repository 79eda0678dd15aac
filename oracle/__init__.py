"""fp64 CPU oracle for exact-softmax attention forward and backward.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it; the library under
``attention_backward_preprocess_gb300`` never imports it.

This module is a thin ctypes wrapper around ``fa_oracle.c`` (plain C, fp64,
optionally OpenMP).  The C source documents the mathematics and where each
step is stated on the pages; all arrays here are float64 numpy arrays in the
public layouts:

* dense : q, dq ``[B, Sq, Hq, D]``; k, dk ``[B, Sk, Hkv, D]``; o, dout
  ``[B, Sq, Hq, Dv]``; v, dv ``[B, Sk, Hkv, Dv]``; lse ``[B, Hq, Sq]``
* varlen: ``cu_q`` / ``cu_k`` int32 prefix sums of the ``nseq`` lengths;
  q ``[total_q, Hq, D]``; k ``[total_k, Hkv, D]`` (o, dout, v likewise with
  Dv); lse ``[Hq, total_q]``

The value-side head dim Dv is v's last axis; it may differ from D.

Every function also takes the optional extensions as keywords:
``window=(left, right)`` (a local band around the bottom-right diagonal, -1 =
unbounded on that side), ``alibi`` (slopes ``[Hq]`` or ``[B, Hq]``) and
``seqused_q`` / ``seqused_k`` (used lengths per sequence; rows past them are
neither read nor written, and come back as zeros), ``bias`` (an elementwise
additive bias ``[B or 1, Hq or 1, Sq, Sk]``, dense only; its gradient dBias =
dS comes from ``head_matrices``) and ``dropout=(t, seed, offset)`` (drop
probability t / 256 with a Philox4x32-10 mask, see ``fa_oracle.c``).

Parity status: every function here is pinned by ``tests/test_oracle.py``
(central finite differences, invariants, a hand-derived 2x2 example, closed
forms for degenerate inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "libfa_oracle.so")
_lock = threading.Lock()
_default = None


def compile_library(src: str, out: str, openmp: bool = True) -> str:
    """gcc -O2 (no fast-math) shared build of an oracle C source."""
    tmp = out + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        if not openmp:
            raise subprocess.CalledProcessError(1, base)
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into libfa_oracle.so (gcc, -O2, OpenMP if available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE):
        return _LIB
    return compile_library(SOURCE, _LIB)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class _Ext(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("alibi", ctypes.POINTER(ctypes.c_double)), ("alibi_bstride", ctypes.c_int),
                ("seqused_q", ctypes.POINTER(ctypes.c_int)),
                ("seqused_k", ctypes.POINTER(ctypes.c_int)),
                ("bias", ctypes.POINTER(ctypes.c_double)), ("bias_bs", ctypes.c_long),
                ("bias_hs", ctypes.c_long), ("bias_rs", ctypes.c_long),
                ("dropout_t", ctypes.c_int), ("dropout_seed", ctypes.c_ulonglong),
                ("dropout_offset", ctypes.c_uint), ("head_dim_v", ctypes.c_int)]


def _ext(B, Hq, window=None, alibi=None, seqused_q=None, seqused_k=None, bias=None,
         dropout=None, head_dim_v=0):
    """(ctypes pointer or None, arrays to keep alive) for the extension options.

    ``bias`` is a [B or 1, Hq or 1, Sq, Sk] array (dense problems); a size-1
    batch or head axis is broadcast.  ``dropout`` is (t, seed, offset): drop
    probability t / 256, the Philox key and the counter's fourth word.
    ``head_dim_v``: the value-side head dim when it differs from D (else 0)."""
    if (window is None and alibi is None and seqused_q is None and seqused_k is None
            and bias is None and dropout is None and not head_dim_v):
        return None, ()
    wl, wr = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    keep = []
    e = _Ext(wl, wr, None, 0, None, None)
    e.head_dim_v = int(head_dim_v)
    if dropout is not None:
        e.dropout_t, e.dropout_seed, e.dropout_offset = (int(dropout[0]), int(dropout[1]),
                                                         int(dropout[2]))
    if alibi is not None:
        a = np.ascontiguousarray(alibi, dtype=np.float64)
        if a.shape not in ((Hq,), (B, Hq)):
            raise ValueError("alibi slopes are [Hq] or [B, Hq]")
        e.alibi = _ptr(a)
        e.alibi_bstride = Hq if a.ndim == 2 else 0
        keep.append(a)
    if bias is not None:
        a = np.ascontiguousarray(bias, dtype=np.float64)
        if a.ndim != 4 or a.shape[0] not in (1, B) or a.shape[1] not in (1, Hq):
            raise ValueError("bias is [B or 1, Hq or 1, Sq, Sk]")
        e.bias = _ptr(a)
        e.bias_bs = 0 if a.shape[0] == 1 else a.shape[1] * a.shape[2] * a.shape[3]
        e.bias_hs = 0 if a.shape[1] == 1 else a.shape[2] * a.shape[3]
        e.bias_rs = a.shape[3]
        keep.append(a)
    for name, arr in (("seqused_q", seqused_q), ("seqused_k", seqused_k)):
        if arr is not None:
            a = np.ascontiguousarray(arr, dtype=np.int32)
            if a.shape != (B,):
                raise ValueError(name + " is [B]")
            setattr(e, name, _ptr(a, ctypes.c_int))
            keep.append(a)
    keep.append(e)
    return ctypes.pointer(e), keep


def _shape_args(q, k, scale, causal, cu_q, cu_k):
    if cu_q is None:
        if q.ndim != 4 or k.ndim != 4:
            raise ValueError("dense inputs are [B, S, H, D]")
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
        cq = ck = None
    else:
        cq = np.ascontiguousarray(cu_q, dtype=np.int32)
        ck = np.ascontiguousarray(cu_k, dtype=np.int32)
        B = len(cq) - 1
        Hq, D = q.shape[1], q.shape[2]
        Hkv = k.shape[1]
        Sq = int(np.max(np.diff(cq))) if B > 0 else 0
        Sk = int(np.max(np.diff(ck))) if B > 0 else 0
    args = [B, Sq, Sk, Hq, Hkv, D, float(scale), int(bool(causal)),
            _ptr(cq, ctypes.c_int), _ptr(ck, ctypes.c_int)]
    return args, (cq, ck), (B, Sq, Sk, Hq, Hkv, D)


def _dv(D, Dv):
    """head_dim_v for the C side: 0 when the value head dim equals D."""
    return 0 if int(Dv) == int(D) else int(Dv)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        shape = [ctypes.c_int] * 6 + [ctypes.c_double, ctypes.c_int, ip, ip]
        ep = ctypes.POINTER(_Ext)
        lib.oracle_forward.argtypes = [dp, dp, dp] + shape + [dp, dp, ctypes.c_int, ep]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [dp] * 6 + shape + [dp, dp, dp, ctypes.c_int, ep]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_backward_sampled.argtypes = (
            [dp] * 6 + shape + [ctypes.c_int, ip, dp, ctypes.c_int, ip, dp, dp, ctypes.c_int, ep])
        lib.oracle_backward_sampled.restype = ctypes.c_int
        lib.oracle_head_matrices.argtypes = [dp] * 6 + shape + [ctypes.c_int] * 2 + [dp, dp, ep]
        lib.oracle_head_matrices.restype = ctypes.c_int
        lib.oracle_preprocess.argtypes = [dp] * 6 + shape + [dp, dp, ctypes.c_int, ep]
        lib.oracle_preprocess.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        up = ctypes.POINTER(ctypes.c_uint)
        lib.oracle_philox4x32_10.argtypes = [up, up, up]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_factors.argtypes = [ctypes.c_int] * 6 + [ip, ip, ctypes.c_int,
                                                                     ctypes.c_int, dp, ep]
        lib.oracle_dropout_factors.restype = ctypes.c_int
        self.lib = lib
        self.path = libpath

    def philox(self, ctr, key):
        """Philox4x32-10 output words of one counter (4 words) and key (2 words)."""
        c = (ctypes.c_uint * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
        k = (ctypes.c_uint * 2)(*[int(x) & 0xFFFFFFFF for x in key])
        o = (ctypes.c_uint * 4)()
        self.lib.oracle_philox4x32_10(c, k, o)
        return [int(x) for x in o]

    def dropout_factors(self, B, Sq, Sk, Hq, Hkv, D, b, h, cu_q=None, cu_k=None, lq=None,
                        lk=None, **ext):
        """M * s of every (i, j) of head problem (b, h): [Lq, Lk]."""
        e, keep_e = _ext(B, Hq, **ext)
        cq = None if cu_q is None else np.ascontiguousarray(cu_q, dtype=np.int32)
        ck = None if cu_k is None else np.ascontiguousarray(cu_k, dtype=np.int32)
        lq = (Sq if cq is None else int(cq[b + 1] - cq[b])) if lq is None else lq
        lk = (Sk if ck is None else int(ck[b + 1] - ck[b])) if lk is None else lk
        F = np.zeros((lq, lk))
        rc = self.lib.oracle_dropout_factors(B, Sq, Sk, Hq, Hkv, D, _ptr(cq, ctypes.c_int),
                                             _ptr(ck, ctypes.c_int), int(b), int(h), _ptr(F), e)
        if rc:
            raise ValueError("oracle_dropout_factors rejected its arguments (%d)" % rc)
        return F

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def _threads(self, nthreads):
        return int(nthreads) if nthreads else self.max_threads()

    def forward(self, q, k, v, scale, causal=False, cu_q=None, cu_k=None, nthreads=None,
                **ext):
        """Returns (o, lse) in fp64; lse is natural-log, -inf for a row with no key."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        args, keep, (B, Sq, Sk, Hq, Hkv, D) = _shape_args(q, k, scale, causal, cu_q, cu_k)
        Dv = v.shape[-1]
        e, keep_e = _ext(B, Hq, head_dim_v=_dv(D, Dv), **ext)
        o = np.zeros(q.shape[:-1] + (Dv,))
        lse = np.zeros((B, Hq, Sq) if cu_q is None else (Hq, q.shape[0]), dtype=np.float64)
        rc = self.lib.oracle_forward(_ptr(q), _ptr(k), _ptr(v), *args, _ptr(o), _ptr(lse),
                                     self._threads(nthreads), e)
        if rc:
            raise ValueError("oracle_forward rejected its arguments (%d)" % rc)
        return o, lse

    def backward(self, q, k, v, dout, scale, causal=False, o=None, lse=None, cu_q=None,
                 cu_k=None, nthreads=None, **ext):
        """Returns (dq, dk, dv) in fp64.  o / lse None -> the oracle's own fp64 forward."""
        q, k, v, dout, o, lse = map(_f64, (q, k, v, dout, o, lse))
        args, keep, (B, Sq, Sk, Hq, Hkv, D) = _shape_args(q, k, scale, causal, cu_q, cu_k)
        Dv = v.shape[-1]
        e, keep_e = _ext(B, Hq, head_dim_v=_dv(D, Dv), **ext)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        rc = self.lib.oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(dout), *args, _ptr(dq), _ptr(dk), _ptr(dv),
                                      self._threads(nthreads), e)
        if rc:
            raise ValueError("oracle_backward rejected its arguments (%d)" % rc)
        return dq, dk, dv

    def backward_sampled(self, q, k, v, dout, scale, causal=False, o=None, lse=None, cu_q=None,
                         cu_k=None, qrows=(), krows=(), nthreads=None, **ext):
        """dQ rows for (b, s, h) triples and dK / dV rows for (b, s, hk) triples.

        Returns (dq_rows [nq, D], dk_rows [nk, D], dv_rows [nk, D]).
        """
        q, k, v, dout, o, lse = map(_f64, (q, k, v, dout, o, lse))
        args, keep, (B, Sq, Sk, Hq, Hkv, D) = _shape_args(q, k, scale, causal, cu_q, cu_k)
        Dv = v.shape[-1]
        e, keep_e = _ext(B, Hq, head_dim_v=_dv(D, Dv), **ext)
        qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32).reshape(-1, 3))
        kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32).reshape(-1, 3))
        dq = np.zeros((len(qr), D))
        dk = np.zeros((len(kr), D))
        dv = np.zeros((len(kr), Dv))
        rc = self.lib.oracle_backward_sampled(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), *args,
            len(qr), _ptr(qr, ctypes.c_int), _ptr(dq), len(kr), _ptr(kr, ctypes.c_int),
            _ptr(dk), _ptr(dv), self._threads(nthreads), e)
        if rc:
            raise ValueError("oracle_backward_sampled rejected its arguments (%d)" % rc)
        return dq, dk, dv

    def preprocess(self, q, k, v, dout, scale, causal=False, o=None, lse=None, cu_q=None,
                   cu_k=None, nthreads=None, **ext):
        """(Dv, LSE_guarded) per query row, in lse's layout: Dv_i = <dO_i, O_i>."""
        q, k, v, dout, o, lse = map(_f64, (q, k, v, dout, o, lse))
        args, keep, (B, Sq, Sk, Hq, Hkv, D) = _shape_args(q, k, scale, causal, cu_q, cu_k)
        Dv = v.shape[-1]
        e, keep_e = _ext(B, Hq, head_dim_v=_dv(D, Dv), **ext)
        shape = (B, Hq, Sq) if cu_q is None else (Hq, q.shape[0])
        dvec = np.zeros(shape)
        lse_out = np.zeros(shape)
        rc = self.lib.oracle_preprocess(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                        _ptr(dout), *args, _ptr(dvec), _ptr(lse_out),
                                        self._threads(nthreads), e)
        if rc:
            raise ValueError("oracle_preprocess rejected its arguments (%d)" % rc)
        return dvec, lse_out

    def head_matrices(self, q, k, v, dout, scale, causal=False, o=None, lse=None, cu_q=None,
                      cu_k=None, b=0, h=0, **ext):
        """Dense P and dS [Lq, Lk] of one (sequence, query head) problem (tiny inputs)."""
        q, k, v, dout, o, lse = map(_f64, (q, k, v, dout, o, lse))
        args, keep, (B, Sq, Sk, Hq, Hkv, D) = _shape_args(q, k, scale, causal, cu_q, cu_k)
        Dv = v.shape[-1]
        e, keep_e = _ext(B, Hq, head_dim_v=_dv(D, Dv), **ext)
        if cu_q is None:
            lq, lk = Sq, Sk
        else:
            lq = int(keep[0][b + 1] - keep[0][b])
            lk = int(keep[1][b + 1] - keep[1][b])
        if ext.get("seqused_q") is not None:
            lq = int(ext["seqused_q"][b])
        if ext.get("seqused_k") is not None:
            lk = int(ext["seqused_k"][b])
        P = np.zeros((lq, lk))
        dS = np.zeros((lq, lk))
        rc = self.lib.oracle_head_matrices(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           _ptr(dout), *args, int(b), int(h), _ptr(P), _ptr(dS),
                                           e)
        if rc:
            raise ValueError("oracle_head_matrices rejected its arguments (%d)" % rc)
        return P, dS


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def forward(*a, **kw):
    return default().forward(*a, **kw)


def backward(*a, **kw):
    return default().backward(*a, **kw)


def backward_sampled(*a, **kw):
    return default().backward_sampled(*a, **kw)


def head_matrices(*a, **kw):
    return default().head_matrices(*a, **kw)


def preprocess(*a, **kw):
    return default().preprocess(*a, **kw)


def philox(*a, **kw):
    return default().philox(*a, **kw)


def dropout_factors(*a, **kw):
    return default().dropout_factors(*a, **kw)
