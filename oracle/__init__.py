"""fp64 CPU oracle for the segmented gated delta-rule forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package; the two share no code.

The arithmetic lives in ``oracle.c`` (compiled here with gcc, no fast-math);
this module only marshals numpy arrays through ctypes.  Every function follows
the article "flash-linear-attention 上下文并行CP 从 CP2TP、Ring CP 到 True CP
的设计取舍与源码实现" (cited as [FLA-CP]):

* ``scan``       -- serial per-token recurrence, the definition of the result.
* ``segmented``  -- [FLA-CP] §2.1: per-segment (S_ext, M) from the trailing
                    fragment, the merge loop ``S <- M_j S + S_ext,j``, then the
                    per-fragment forward from S_init.
* ``chunked`` / ``chunked_pre`` -- [FLA-CP] §2.2: the chunk form in WY
                    representation restated in fp64 (pins the chunk equations).
* ``backward``   -- the reverse of the per-token scan: gradients of
                    sum <do, o> + sum <dht, S_final> (the backward that
                    [FLA-CP] §2.2 and §4 split into pre-process, reverse merge
                    and chunk chains has this result).

Inputs q, k, v, beta are the exact values the GPU receives: float32 arrays, or
bfloat16 bit patterns passed as uint16 arrays.  Gates are float32 natural-log
gates, shape [B, T, H] (scalar, GDN) or [B, T, H, dk] (per-dim, KDA).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain -O2, IEEE fp64, pthreads)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("T", ctypes.c_int64),
                ("cu_seqlens", ctypes.POINTER(ctypes.c_int64)), ("num_seqs", ctypes.c_int32),
                ("gate_kind", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("order", ctypes.c_int32), ("scale", ctypes.c_double), ("Hq", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, dp, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            pp = ctypes.POINTER(_Problem)
            lib.oracle_scan.argtypes = [pp, vp, vp, vp, vp, fp, dp, dp, dp, ctypes.c_int]
            lib.oracle_segmented.argtypes = [pp, ctypes.c_int, vp, vp, vp, vp, fp, dp, dp, dp, dp, dp,
                                             ctypes.c_int]
            lib.oracle_chunked.argtypes = [pp, ctypes.c_int, vp, vp, vp, vp, fp, dp, dp]
            lib.oracle_chunked_pre.argtypes = [pp, ctypes.c_int, vp, vp, vp, fp, ctypes.c_int,
                                               ctypes.c_int64, ctypes.c_int64, dp, dp]
            lib.oracle_backward.argtypes = [pp, vp, vp, vp, vp, fp, vp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            for f in (lib.oracle_scan, lib.oracle_segmented, lib.oracle_chunked, lib.oracle_chunked_pre,
                      lib.oracle_backward):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def as_oracle_array(x):
    """Return a C-contiguous numpy view with the oracle's dtype code.

    Accepts numpy arrays or CPU torch tensors; bfloat16 becomes its uint16
    bit pattern (code 1), everything else float32 (code 0).
    """
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16)), 1
        return np.ascontiguousarray(x.to(torch.float32).numpy()), 0
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 1
    return np.ascontiguousarray(x, dtype=np.float32), 0


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class Problem:
    """Shapes and options shared by every oracle call.

    q: [B, T, Hq, dk]; k: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H];
    g: [B, T, H] or [B, T, H, dk] (float32, natural-log gates).  Hq is H, or
    a multiple G H of it (grouped query heads, [FLA-CP] §5.1: query head hq
    reads the state of head hq // G; outputs o are [B, T, Hq, dv]).  With
    ``cu_seqlens`` (N+1 int64 offsets) the batch is packed: B == 1 and T is
    the total.
    """

    def __init__(self, q, k, v, beta, g, cu_seqlens=None, scale=1.0, order=0):
        self.q, dq = as_oracle_array(q)
        self.k, dk_ = as_oracle_array(k)
        self.v, dv_ = as_oracle_array(v)
        self.beta, db = as_oracle_array(beta)
        if not (dq == dk_ == dv_ == db):
            raise ValueError("q, k, v, beta must share one dtype")
        g = g.detach().cpu().numpy() if hasattr(g, "detach") else g
        self.g = np.ascontiguousarray(g, dtype=np.float32)
        B, T, H, dk = self.k.shape
        dv = self.v.shape[3]
        Hq = self.q.shape[2]
        if self.q.shape[:2] != (B, T) or self.q.shape[3] != dk or Hq % H != 0:
            raise ValueError("q must be [B, T, Hq, dk] with Hq a multiple of k's H")
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
            if B != 1 or cu[0] != 0 or cu[-1] != T:
                raise ValueError("packed batches need B == 1 and cu_seqlens spanning T")
            self.cu = cu
            n = len(cu) - 1
        else:
            self.cu = None
            n = B
        gate_kind = 0 if self.g.ndim == 3 else 1
        self.B, self.T, self.H, self.dk, self.dv, self.N = B, T, H, dk, dv, n
        self.Hq = Hq
        self.gate_kind = gate_kind
        self._p = _Problem(B, H, dk, dv, T,
                           self.cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if self.cu is not None else None,
                           n, gate_kind, dq, order, float(scale), Hq)

    def _ptr(self, a):
        return a.ctypes.data_as(ctypes.c_void_p)

    def scan(self, h0=None, nthreads=None):
        """Serial scan: returns (o [B,T,Hq,dv] fp64, final states [N,H,dk,dv] fp64)."""
        lib = _load()
        o = np.zeros((self.B, self.T, self.Hq, self.dv), np.float64)
        ht = np.zeros((self.N, self.H, self.dk, self.dv), np.float64)
        h0p = None
        if h0 is not None:
            h0 = np.ascontiguousarray(h0, dtype=np.float64)
            assert h0.shape == ht.shape
            h0p = self._ptr(h0)
        rc = lib.oracle_scan(ctypes.byref(self._p), self._ptr(self.q), self._ptr(self.k), self._ptr(self.v),
                             self._ptr(self.beta), self._ptr(self.g), h0p, self._ptr(o), self._ptr(ht),
                             nthreads or default_threads())
        assert rc == 0
        return o, ht

    def segmented(self, R, nthreads=None):
        """[FLA-CP] §2.1 on R contiguous segments.

        Returns dict with S_ext [R,B,H,dk,dv], M [R,B,H,dk,dk], S_init
        [R,B,H,dk,dv], o [B,T,Hq,dv], ht [N,H,dk,dv] (all fp64).  Raises
        ValueError when the cut rule of [FLA-CP] §3.3 fails.
        """
        lib = _load()
        R = int(R)
        S_ext = np.zeros((R, self.B, self.H, self.dk, self.dv), np.float64)
        M = np.zeros((R, self.B, self.H, self.dk, self.dk), np.float64)
        S_init = np.zeros_like(S_ext)
        o = np.zeros((self.B, self.T, self.Hq, self.dv), np.float64)
        ht = np.zeros((self.N, self.H, self.dk, self.dv), np.float64)
        rc = lib.oracle_segmented(ctypes.byref(self._p), R, self._ptr(self.q), self._ptr(self.k),
                                  self._ptr(self.v), self._ptr(self.beta), self._ptr(self.g),
                                  self._ptr(S_ext), self._ptr(M), self._ptr(S_init), self._ptr(o),
                                  self._ptr(ht), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"token count per row must be >= R and divisible by R (R={R})")
        return dict(S_ext=S_ext, M=M, S_init=S_init, o=o, ht=ht)

    def chunked(self, C):
        """[FLA-CP] §2.2 chunk form from zero state: (o, final states), fp64 (Hq == H only)."""
        lib = _load()
        if self.Hq != self.H:
            raise ValueError("the chunk restatement covers Hq == H only")
        o = np.zeros((self.B, self.T, self.H, self.dv), np.float64)
        ht = np.zeros((self.N, self.H, self.dk, self.dv), np.float64)
        rc = lib.oracle_chunked(ctypes.byref(self._p), int(C), self._ptr(self.q), self._ptr(self.k),
                                self._ptr(self.v), self._ptr(self.beta), self._ptr(self.g),
                                self._ptr(o), self._ptr(ht))
        assert rc == 0
        return o, ht

    def chunked_pre(self, C, h, t0, t1):
        """Chunk-form (S_ext, M) of global tokens [t0, t1) of head h, fp64."""
        lib = _load()
        S = np.zeros((self.dk, self.dv), np.float64)
        M = np.zeros((self.dk, self.dk), np.float64)
        rc = lib.oracle_chunked_pre(ctypes.byref(self._p), int(C), self._ptr(self.k), self._ptr(self.v),
                                    self._ptr(self.beta), self._ptr(self.g), int(h), int(t0), int(t1),
                                    self._ptr(S), self._ptr(M))
        assert rc == 0
        return S, M


def _backward(self, do, dht=None, nthreads=None):
    """Gradients of sum <do, o> + sum <dht, S_final> (fp64): dict with dq
    [B,T,Hq,dk], dk [B,T,H,dk], dv [B,T,H,dv], dbeta [B,T,H], dg (the gate's
    shape).  ``do`` is [B,T,Hq,dv] in the input dtype of q, k, v (fp32 array
    or bf16 bits)."""
    lib = _load()
    d_o, ddt = as_oracle_array(do)
    if ddt != self._p.in_dtype or d_o.shape != (self.B, self.T, self.Hq, self.dv):
        raise ValueError("do must be [B, T, Hq, dv] in the input dtype")
    out = dict(dq=np.zeros((self.B, self.T, self.Hq, self.dk)), dk=np.zeros((self.B, self.T, self.H, self.dk)),
               dv=np.zeros((self.B, self.T, self.H, self.dv)), dbeta=np.zeros((self.B, self.T, self.H)),
               dg=np.zeros(self.g.shape))
    dhtp = None
    if dht is not None:
        dht = np.ascontiguousarray(dht, dtype=np.float64)
        assert dht.shape == (self.N, self.H, self.dk, self.dv)
        dhtp = self._ptr(dht)
    rc = lib.oracle_backward(ctypes.byref(self._p), self._ptr(self.q), self._ptr(self.k), self._ptr(self.v),
                             self._ptr(self.beta), self._ptr(self.g), self._ptr(d_o), dhtp, self._ptr(out["dq"]),
                             self._ptr(out["dk"]), self._ptr(out["dv"]), self._ptr(out["dbeta"]),
                             self._ptr(out["dg"]), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"backward not covered (code {rc})")
    return out


Problem.backward = _backward
