"""Thin ctypes binding of libcpdr.so (include/cpdr.h).

Argument marshalling only: tensors are passed as raw device pointers and the
current torch CUDA stream as a cudaStream_t; every step of the computation
runs in the library's CUDA kernels.  The library must have been built
(``python -c "import __graft_entry__ as g; g.build()"``); loading raises if it
is missing -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpdr.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = range(6)
FLAG_HOST_ONLY = 1 << 0
FLAG_FORCE_SIMT = 1 << 1
FLAG_LAYOUT_ZIGZAG = 1 << 2
FLAG_STATE_V_FIRST = 1 << 3
FRAG_CONT_PREV, FRAG_CONT_NEXT, FRAG_ENDS_SEQ = 1, 2, 4

EXPORTED = ["cpdr_ctx_create", "cpdr_ctx_destroy", "cpdr_buffer_sizes", "cpdr_plan_num_fragments",
            "cpdr_plan_fragments", "cpdr_plan_counts", "cpdr_wy_bytes", "cpdr_wy_build", "cpdr_preprocess",
            "cpdr_merge", "cpdr_fwd", "cpdr_host_workspace_bytes",
            "cpdr_forward_host", "cpdr_forward_noalloc", "cpdr_check_device_status", "cpdr_selftest_wait_timeout",
            "cpdr_conv1d_fwd", "cpdr_plan_conv_tokens", "cpdr_bwd_workspace_bytes", "cpdr_bwd",
            "cpdr_last_error", "cpdr_version"]


class CpdrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"cpdr status {status}: {msg}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("R", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("T", ctypes.c_int64),
                ("cu_seqlens_host", ctypes.POINTER(ctypes.c_int64)), ("gate_kind", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("flags", ctypes.c_uint32), ("scale", ctypes.c_float),
                ("Hq", ctypes.c_int32), ("conv_width", ctypes.c_int32)]


class Fragment(ctypes.Structure):
    _fields_ = [("tok0", ctypes.c_int64), ("len", ctypes.c_int32), ("seg", ctypes.c_int32),
                ("seq", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load():
    """Load libcpdr.so and declare its signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        st = ctypes.c_int
        lib.cpdr_ctx_create.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(vp)]
        lib.cpdr_ctx_destroy.argtypes = [vp]
        lib.cpdr_ctx_destroy.restype = None
        lib.cpdr_buffer_sizes.argtypes = [vp] + [ctypes.POINTER(sz)] * 4
        lib.cpdr_plan_num_fragments.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.cpdr_plan_fragments.argtypes = [vp, ctypes.POINTER(Fragment), ctypes.c_int32]
        lib.cpdr_plan_counts.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.cpdr_wy_bytes.argtypes = [vp, ctypes.POINTER(sz)]
        lib.cpdr_wy_build.argtypes = [vp] * 7
        lib.cpdr_preprocess.argtypes = [vp] * 9
        lib.cpdr_merge.argtypes = [vp] * 5
        lib.cpdr_fwd.argtypes = [vp] * 11
        lib.cpdr_host_workspace_bytes.argtypes = [vp, ctypes.POINTER(sz)]
        lib.cpdr_conv1d_fwd.argtypes = [vp, vp, vp, vp, ctypes.c_int32, ctypes.c_int32, vp, vp]
        lib.cpdr_plan_conv_tokens.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
        lib.cpdr_bwd_workspace_bytes.argtypes = [vp, ctypes.POINTER(sz)]
        lib.cpdr_bwd.argtypes = [vp] * 16 + [sz, vp]
        lib.cpdr_forward_host.argtypes = [vp] * 9 + [sz, vp]
        lib.cpdr_forward_noalloc.argtypes = [vp] * 9
        lib.cpdr_check_device_status.argtypes = [vp, vp]
        lib.cpdr_selftest_wait_timeout.argtypes = [vp, ctypes.c_longlong, vp]
        for name in EXPORTED:
            f = getattr(lib, name)
            if name not in ("cpdr_ctx_destroy", "cpdr_last_error", "cpdr_version"):
                f.restype = st
        lib.cpdr_last_error.restype = ctypes.c_char_p
        lib.cpdr_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int):
    if status != OK:
        raise CpdrError(status, load().cpdr_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Context:
    """One planned problem: shapes, the R-segment cut, dtype and gate kind.

    ``gate`` is "gdn" (scalar gate g [B,T,H]) or "kda" (per-dim gk [B,T,H,d]);
    ``dtype`` is "fp32" or "bf16" for q, k, v, beta and o; gates are fp32.
    With ``cu_seqlens`` (N+1 offsets) the batch is packed: B must be 1.
    ``layout="zigzag"`` takes the token axis in the zigzag order of R ranks
    (2R parts, rank r holding parts r and 2R-1-r); ``Hq`` (a multiple of H)
    gives q and o grouped query heads; ``state_v_first`` stores the dk x dv
    states S_ext, S_init and final_state as [.., dv, dk].  ``conv_width``
    (1..8) enables ``conv1d_fwd``, the causal conv1d on the same segments.
    """

    def __init__(self, B, T, H, d, R, gate="gdn", dtype="bf16", cu_seqlens=None, scale=1.0,
                 host_only=False, force_simt=False, layout="contiguous", Hq=None, state_v_first=False,
                 conv_width=0):
        lib = load()
        if layout not in ("contiguous", "zigzag"):
            raise ValueError(f"layout must be 'contiguous' or 'zigzag', got {layout!r}")
        self.B, self.T, self.H, self.d, self.R = int(B), int(T), int(H), int(d), int(R)
        self.layout = layout
        # segments of the exchange buffers: the ranks, or 2R zigzag pieces
        self.pieces = 2 * self.R if layout == "zigzag" else self.R
        self.Hq = self.H if Hq is None else int(Hq)
        self.state_v_first = bool(state_v_first)
        self.conv_width = int(conv_width)
        self.gate, self.dtype = gate, dtype
        self.torch_dtype = torch.float32 if dtype == "fp32" else torch.bfloat16
        self._cu = None
        n = self.B
        cu_ptr = None
        if cu_seqlens is not None:
            cu = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
            self._cu = (ctypes.c_int64 * len(cu))(*cu)
            cu_ptr = ctypes.cast(self._cu, ctypes.POINTER(ctypes.c_int64))
            n = len(cu) - 1
        self.N = n
        flags = ((FLAG_HOST_ONLY if host_only else 0) | (FLAG_FORCE_SIMT if force_simt else 0) |
                 (FLAG_LAYOUT_ZIGZAG if layout == "zigzag" else 0) |
                 (FLAG_STATE_V_FIRST if self.state_v_first else 0))
        desc = Desc(self.B, self.H, self.d, self.d, self.R, n, self.T, cu_ptr,
                    0 if gate == "gdn" else 1, 0 if dtype == "fp32" else 1, flags, float(scale), self.Hq,
                    self.conv_width)
        h = ctypes.c_void_p()
        _check(lib.cpdr_ctx_create(ctypes.byref(desc), ctypes.byref(h)))
        self._h = h
        self._lib = lib

    def close(self):
        if getattr(self, "_h", None):
            self._lib.cpdr_ctx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- plan ---------------------------------------------------------
    def fragments(self):
        n = ctypes.c_int32()
        _check(self._lib.cpdr_plan_num_fragments(self._h, ctypes.byref(n)))
        arr = (Fragment * max(1, n.value))()
        _check(self._lib.cpdr_plan_fragments(self._h, arr, n.value))
        return [(f.tok0, f.len, f.seg, f.seq, f.flags) for f in arr[:n.value]]

    def counts(self):
        """Plan counters: fragments, pre items, merge chains, zeroed S_ext/M
        segments, zeroed S_init segments, empty sequences, kernel launches per
        step, tensor-core path selected."""
        out = (ctypes.c_int32 * 8)()
        _check(self._lib.cpdr_plan_counts(self._h, out))
        keys = ["fragments", "pre_items", "chains", "zero_pre", "zero_init", "empty_seqs", "launches", "tc"]
        return dict(zip(keys, list(out)))

    def buffer_sizes(self):
        s = [ctypes.c_size_t() for _ in range(4)]
        _check(self._lib.cpdr_buffer_sizes(self._h, *[ctypes.byref(x) for x in s]))
        return [x.value for x in s]

    def wy_bytes(self):
        """Bytes of the WY tile workspace (0 on the CUDA-core path)."""
        n = ctypes.c_size_t()
        _check(self._lib.cpdr_wy_bytes(self._h, ctypes.byref(n)))
        return n.value

    def alloc_buffers(self, device="cuda"):
        """Caller-owned exchange buffers S_ext, M, S_init and final_state (fp32)
        and the WY tile workspace ``wy`` (bytes; None when not needed).  The
        segment axis has one entry per segment (2R in the zigzag layout); the
        last two axes of the states are (dk, dv), or (dv, dk) with
        ``state_v_first``."""
        d, R, B, H, N = self.d, self.pieces, self.B, self.H, self.N
        f32 = torch.float32
        nwy = self.wy_bytes()
        return dict(S_ext=torch.empty((R, B, H, d, d), dtype=f32, device=device),
                    M=torch.empty((R, B, H, d, d), dtype=f32, device=device),
                    S_init=torch.empty((R, B, H, d, d), dtype=f32, device=device),
                    final_state=torch.empty((N, H, d, d), dtype=f32, device=device),
                    wy=torch.empty(nwy, dtype=torch.uint8, device=device) if nwy else None)

    # ---- the three stages ------------------------------------------------
    def _check_inputs(self, **ts):
        B, T, H, d, Hq = self.B, self.T, self.H, self.d, self.Hq
        shapes = dict(q=(B, T, Hq, d), k=(B, T, H, d), v=(B, T, H, d), beta=(B, T, H), o=(B, T, Hq, d),
                      g=(B, T, H) if self.gate == "gdn" else (B, T, H, d))
        for name, t in ts.items():
            if t is None:
                continue
            if tuple(t.shape) != shapes[name]:
                raise ValueError(f"{name}: expected shape {shapes[name]}, got {tuple(t.shape)}")
            want = torch.float32 if name == "g" else self.torch_dtype
            if t.dtype != want:
                raise ValueError(f"{name}: expected {want}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")

    def wy_build(self, q, k, beta, g, wy, stream=None):
        """WY tiles (and, for the per-dim gate, the pre-gated operand tiles,
        which read q) into ``wy``."""
        self._check_inputs(q=q, k=k, beta=beta, g=g)
        _check(self._lib.cpdr_wy_build(self._h, _ptr(q), _ptr(k), _ptr(beta), _ptr(g), _ptr(wy),
                                       _stream(stream)))

    def preprocess(self, k, v, beta, g, S_ext, M, wy=None, stream=None):
        self._check_inputs(k=k, v=v, beta=beta, g=g)
        _check(self._lib.cpdr_preprocess(self._h, _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(wy), _ptr(S_ext),
                                         _ptr(M), _stream(stream)))

    def merge(self, S_ext, M, S_init, stream=None):
        _check(self._lib.cpdr_merge(self._h, _ptr(S_ext), _ptr(M), _ptr(S_init), _stream(stream)))

    def fwd(self, q, k, v, beta, g, S_init, o, final_state=None, wy=None, stream=None):
        self._check_inputs(q=q, k=k, v=v, beta=beta, g=g, o=o)
        _check(self._lib.cpdr_fwd(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(wy),
                                  _ptr(S_init), _ptr(o), _ptr(final_state), _stream(stream)))

    def run(self, q, k, v, beta, g, bufs=None, o=None, stream=None):
        """WY build -> preprocess -> merge -> fwd on device tensors; returns (o, buffers)."""
        if bufs is None:
            bufs = self.alloc_buffers(q.device)
        if o is None:
            o = torch.empty((self.B, self.T, self.Hq, self.d), dtype=v.dtype, device=v.device)
        wy = bufs.get("wy")
        self.wy_build(q, k, beta, g, wy, stream)
        self.preprocess(k, v, beta, g, bufs["S_ext"], bufs["M"], wy=wy, stream=stream)
        self.merge(bufs["S_ext"], bufs["M"], bufs["S_init"], stream)
        self.fwd(q, k, v, beta, g, bufs["S_init"], o, bufs["final_state"], wy=wy, stream=stream)
        return o, bufs

    # ---- whole path from host memory --------------------------------------
    def host_workspace_bytes(self):
        n = ctypes.c_size_t()
        _check(self._lib.cpdr_host_workspace_bytes(self._h, ctypes.byref(n)))
        return n.value

    def forward_host(self, q, k, v, beta, g, o, final_state, workspace, stream=None):
        """Host tensors in (pinned for async copies), host o / final_state out."""
        self._check_inputs(q=q, k=k, v=v, beta=beta, g=g, o=o)
        _check(self._lib.cpdr_forward_host(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(o),
                                           _ptr(final_state), _ptr(workspace),
                                           ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                                           _stream(stream)))

    def forward_noalloc(self, q, k, v, beta, g, o, final_state=None, stream=None):
        """Whole path through the allocation-free entry point: the library
        keeps its exchange buffers and tables in a fixed device array and
        allocates nothing (works with a host_only context)."""
        self._check_inputs(q=q, k=k, v=v, beta=beta, g=g, o=o)
        _check(self._lib.cpdr_forward_noalloc(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(o),
                                              _ptr(final_state), _stream(stream)))

    # ---- backward ------------------------------------------------------------
    def bwd_workspace_bytes(self):
        n = ctypes.c_size_t()
        _check(self._lib.cpdr_bwd_workspace_bytes(self._h, ctypes.byref(n)))
        return n.value

    def backward(self, q, k, v, beta, g, do, S_init, M, dht=None, workspace=None, stream=None):
        """Gradients of sum <do, o> + sum <dht, final_state> (fp32 tensors
        dq, dk, dv, dbeta, dg).  do is shaped like o ([B, T, Hq, dv]); S_init
        and M are the buffers the forward's merge and pre-process filled for
        the same inputs."""
        self._check_inputs(q=q, k=k, v=v, beta=beta, g=g)
        if tuple(do.shape) != tuple(q.shape[:3]) + (v.shape[3],) or do.dtype != v.dtype or not do.is_contiguous():
            raise ValueError("do must be shaped like o, in the dtype of v")
        dev = q.device
        f32 = torch.float32
        out = dict(dq=torch.empty(q.shape, dtype=f32, device=dev), dk=torch.empty(k.shape, dtype=f32, device=dev),
                   dv=torch.empty(v.shape, dtype=f32, device=dev),
                   dbeta=torch.empty(beta.shape, dtype=f32, device=dev), dg=torch.empty(g.shape, dtype=f32, device=dev))
        if workspace is None:
            workspace = torch.empty(self.bwd_workspace_bytes(), dtype=torch.uint8, device=dev)
        _check(self._lib.cpdr_bwd(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(do), _ptr(dht),
                                  _ptr(S_init), _ptr(M), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                  _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(workspace),
                                  ctypes.c_size_t(workspace.numel()), _stream(stream)))
        return out

    # ---- causal conv1d on the same segments -------------------------------
    def conv_pre_tokens(self):
        """pre_num_conv_tokens per segment (entries: segments x rows)."""
        n = self.pieces * self.B
        out = (ctypes.c_int32 * n)()
        _check(self._lib.cpdr_plan_conv_tokens(self._h, out, n))
        return list(out)

    def conv1d_fwd(self, x, weight, bias, y, activation="silu", stream=None):
        """y = act(bias + causal depthwise conv of x), x and y [B, T, C] in the
        context's token order and input dtype; weight [C, W] and bias [C] fp32."""
        B, T = self.B, self.T
        if x.dim() != 3 or tuple(x.shape[:2]) != (B, T) or x.dtype != self.torch_dtype or not x.is_contiguous():
            raise ValueError(f"x must be a contiguous [{B}, {T}, C] {self.torch_dtype} tensor")
        C = x.shape[2]
        if tuple(y.shape) != tuple(x.shape) or y.dtype != x.dtype or not y.is_contiguous():
            raise ValueError("y must match x")
        if tuple(weight.shape) != (C, self.conv_width) or weight.dtype != torch.float32 or not weight.is_contiguous():
            raise ValueError(f"weight must be a contiguous [{C}, {self.conv_width}] float32 tensor")
        if bias is not None and (tuple(bias.shape) != (C,) or bias.dtype != torch.float32):
            raise ValueError(f"bias must be a [{C}] float32 tensor")
        act = {"silu": 1, None: 0, "none": 0}[activation]
        _check(self._lib.cpdr_conv1d_fwd(self._h, _ptr(x), _ptr(weight), _ptr(bias), C, act, _ptr(y),
                                         _stream(stream)))

    def check_device_status(self, stream=None):
        _check(self._lib.cpdr_check_device_status(self._h, _stream(stream)))

    def selftest_wait_timeout(self, max_cycles=20_000_000, stream=None):
        """Make one bounded device wait give up on purpose (see include/cpdr.h)."""
        _check(self._lib.cpdr_selftest_wait_timeout(self._h, ctypes.c_longlong(int(max_cycles)), _stream(stream)))
