"""Python binding of liblily_q4 (the GB300 MLX-affine Q4 MoE hot path).

Argument marshalling only: every computation runs in the CUDA kernels of
``liblily_q4.so``, reached through its C ABI (``include/lily_q4.h``).  PyTorch
supplies device memory and streams.  There is no CPU fallback: if the library
is missing or cannot load, importing the entry points raises.

The function names are those of the C ABI:

* ``lily_q4_moe_decode(layer, x, y, topk_idx=None, topk_w=None, ws=None, stream=None)``
* ``lily_q4_moe_prefill(layer, x, y, topk_idx=None, topk_w=None, ws=None, stream=None)``
* ``lily_q4_gemv_argmax(W, x, token, logits=None, ws=None, stream=None)``
* ``lily_q4_moe_workspace_bytes``, ``lily_q4_gemv_argmax_workspace_bytes``,
  ``lily_q4_workspace_init``, ``lily_q4_workspace_status``,
  ``lily_q4_status_string``, ``lily_q4_pack``, ``lily_q4_unpack``.

Each compute wrapper returns the C status (0) or raises ``Q4Error``.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE_TOO_SMALL = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5


class Q4Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class lily_q4_mat(C.Structure):
    _fields_ = [("w", C.c_void_p), ("s", C.c_void_p), ("b", C.c_void_p)]


class lily_q4_moe_layer(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_experts", C.c_int32), ("top_k", C.c_int32),
                ("inter", C.c_int32),
                ("gate", lily_q4_mat), ("up", lily_q4_mat), ("down", lily_q4_mat),
                ("has_shared", C.c_int32),
                ("sh_gate", lily_q4_mat), ("sh_up", lily_q4_mat), ("sh_down", lily_q4_mat),
                ("router", C.c_void_p), ("router_bias", C.c_void_p),
                ("shared_gate", C.c_void_p),
                ("shared_bits", C.c_int32), ("router_bits", C.c_int32),
                ("router_q8", lily_q4_mat)]


_lib = None


def load(path: Optional[str] = None):
    """Load liblily_q4.so (raises if it is absent: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"liblily_q4.so not built ({path}); run bit_affine_quantized_mlx_gb300.build")
    L = C.CDLL(path)
    vp, i32, sz = C.c_void_p, C.c_int32, C.c_size_t
    L.lily_q4_moe_decode.argtypes = [C.POINTER(lily_q4_moe_layer), vp, i32, vp, vp, vp, vp, sz, vp]
    L.lily_q4_moe_prefill.argtypes = L.lily_q4_moe_decode.argtypes
    L.lily_q4_gemv_argmax.argtypes = [C.POINTER(lily_q4_mat), i32, i32, vp, vp, vp, vp, sz, vp]
    L.lily_q4_moe_workspace_bytes.argtypes = [C.POINTER(lily_q4_moe_layer), i32, i32]
    L.lily_q4_moe_workspace_bytes.restype = sz
    L.lily_q4_gemv_argmax_workspace_bytes.argtypes = [i32, i32]
    L.lily_q4_gemv_argmax_workspace_bytes.restype = sz
    L.lily_q4_moe_launches.argtypes = [C.POINTER(lily_q4_moe_layer), i32, i32]
    L.lily_q4_gemv_argmax_noalloc.argtypes = [C.POINTER(lily_q4_mat), i32, i32, vp, vp, vp, vp]
    L.lily_q4_gemv_argmax_noalloc_status.argtypes = [vp]
    L.lily_q4_gemv_argmax_logprobs.argtypes = [C.POINTER(lily_q4_mat), i32, i32, vp, vp, vp, vp,
                                               vp, sz, vp]
    L.lily_q8_gemv_argmax.argtypes = L.lily_q4_gemv_argmax.argtypes
    L.lily_q8_gemv_argmax_logprobs.argtypes = L.lily_q4_gemv_argmax_logprobs.argtypes
    L.lily_q8_gemv_argmax_workspace_bytes.argtypes = [i32, i32]
    L.lily_q8_gemv_argmax_workspace_bytes.restype = sz
    L.lily_q4_workspace_init.argtypes = [vp, sz, vp]
    L.lily_q4_selftest_timeout.argtypes = [vp, sz, i32, vp]
    L.lily_q4_workspace_status.argtypes = [vp, vp]
    L.lily_q4_status_string.argtypes = [C.c_int]
    L.lily_q4_status_string.restype = C.c_char_p
    L.lily_q4_pack.argtypes = [vp, i32, i32, vp]
    L.lily_q4_unpack.argtypes = [vp, i32, i32, vp]
    for f in ("lily_q4_moe_decode", "lily_q4_moe_prefill", "lily_q4_gemv_argmax",
              "lily_q4_workspace_init", "lily_q4_workspace_status", "lily_q4_pack",
              "lily_q4_unpack", "lily_q4_version", "lily_q4_moe_launches",
              "lily_q4_gemv_argmax_noalloc", "lily_q4_gemv_argmax_noalloc_status",
              "lily_q4_gemv_argmax_logprobs",
              "lily_q8_gemv_argmax", "lily_q4_selftest_timeout", "lily_q8_gemv_argmax_logprobs"):
        getattr(L, f).restype = C.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().lily_q4_status_string(int(status)).decode()


lily_q4_status_string = status_string


def _check(rc: int, what: str) -> int:
    if rc != OK:
        raise Q4Error(rc, what)
    return rc


# --------------------------------------------------------------------------- torch glue

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else int(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(int(stream.cuda_stream))


def to_device(a: np.ndarray, device="cuda"):
    """Upload a numpy array (uint16/uint32/float32/int32) as a torch tensor of the same bits."""
    torch = _torch()
    a = np.ascontiguousarray(a)
    view = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}.get(a.dtype)
    if view is not None:
        a = a.view(view)
    return torch.from_numpy(a).to(device)


class DeviceQ4:
    """A Q4 matrix (or expert stack) resident on the GPU."""

    def __init__(self, w, s, b):
        self.w, self.s, self.b = w, s, b

    @classmethod
    def upload(cls, m, device="cuda"):
        return cls(to_device(m.w, device), to_device(m.s, device), to_device(m.b, device))

    def c(self) -> lily_q4_mat:
        return lily_q4_mat(_ptr(self.w), _ptr(self.s), _ptr(self.b))

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.w, self.s, self.b))


class DeviceLayer:
    """One MoE layer on the GPU plus its C struct."""

    def __init__(self, H, E, k, I, gate, up, down, router, router_bias=None, sh_gate=None,
                 sh_up=None, sh_down=None, shared_gate=None, shared_bits=4, router_q8=None):
        self.H, self.E, self.k, self.I = H, E, k, I
        self.gate, self.up, self.down = gate, up, down
        self.router, self.router_bias = router, router_bias
        self.sh_gate, self.sh_up, self.sh_down = sh_gate, sh_up, sh_down
        self.shared_gate = shared_gate
        self.shared_bits = shared_bits   # 8: the shared expert's codes are 8-bit
        self.router_q8 = router_q8       # an 8-bit router (DeviceQ4 of [E, H/4] codes) or None
        self._c = None

    @property
    def has_shared(self) -> bool:
        return self.sh_gate is not None

    @classmethod
    def upload(cls, L, device="cuda"):
        up = lambda m: None if m is None else DeviceQ4.upload(m, device)
        arr = lambda a: None if a is None else to_device(a, device)
        return cls(L.H, L.E, L.k, L.I, up(L.gate), up(L.up), up(L.down), arr(L.router),
                   arr(L.router_bias), up(L.sh_gate), up(L.sh_up), up(L.sh_down),
                   arr(L.shared_gate), getattr(L, "shared_bits", 4),
                   up(getattr(L, "router_q8", None)))

    def c(self) -> lily_q4_moe_layer:
        if self._c is None:
            z = lily_q4_mat(None, None, None)
            st = lily_q4_moe_layer()
            st.hidden, st.n_experts, st.top_k, st.inter = self.H, self.E, self.k, self.I
            st.gate, st.up, st.down = self.gate.c(), self.up.c(), self.down.c()
            st.has_shared = 1 if self.has_shared else 0
            st.sh_gate = self.sh_gate.c() if self.has_shared else z
            st.sh_up = self.sh_up.c() if self.has_shared else z
            st.sh_down = self.sh_down.c() if self.has_shared else z
            st.router = _ptr(self.router)
            st.router_bias = _ptr(self.router_bias)
            st.shared_gate = _ptr(self.shared_gate)
            st.shared_bits = 8 if (self.has_shared and self.shared_bits == 8) else 4
            st.router_bits = 8 if self.router_q8 is not None else 16
            st.router_q8 = self.router_q8.c() if self.router_q8 is not None else z
            self._c = st
        return self._c

    def weight_bytes(self) -> int:
        n = self.gate.nbytes + self.up.nbytes + self.down.nbytes
        n += self.router.numel() * 2 if self.router is not None else self.router_q8.nbytes
        if self.has_shared:
            n += self.sh_gate.nbytes + self.sh_up.nbytes + self.sh_down.nbytes
            n += self.shared_gate.numel() * 2
        return n


# --------------------------------------------------------------------------- entry points

def lily_q4_moe_workspace_bytes(layer: DeviceLayer, T: int, prefill: bool = False) -> int:
    return int(load().lily_q4_moe_workspace_bytes(C.byref(layer.c()), int(T), 1 if prefill else 0))


def lily_q4_moe_launches(layer: DeviceLayer, T: int, prefill: bool = False) -> int:
    return int(load().lily_q4_moe_launches(C.byref(layer.c()), int(T), 1 if prefill else 0))


def lily_q4_gemv_argmax_workspace_bytes(N: int, K: int) -> int:
    return int(load().lily_q4_gemv_argmax_workspace_bytes(int(N), int(K)))


def new_workspace(nbytes: int, device="cuda"):
    """A zero-filled, 256-byte aligned workspace (torch allocations are 256-aligned)."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def lily_q4_workspace_init(ws, stream=None) -> int:
    return _check(load().lily_q4_workspace_init(_ptr(ws), ws.numel(), _stream(stream)),
                  "lily_q4_workspace_init")


def lily_q4_workspace_status(ws, stream=None) -> int:
    """0, or ERR_TIMEOUT (returned, not raised) if a bounded device wait gave up."""
    return int(load().lily_q4_workspace_status(_ptr(ws), _stream(stream)))


def _moe(fn, name, layer, x, y, topk_idx, topk_w, ws, stream):
    T = int(x.shape[0])
    return _check(fn(C.byref(layer.c()), _ptr(x), T, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                     _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)), name)


def lily_q4_moe_decode(layer: DeviceLayer, x, y, topk_idx=None, topk_w=None, ws=None, stream=None):
    """y[T,H] (bf16 bits as int16) = decode MoE of x[T,H]; see include/lily_q4.h."""
    return _moe(load().lily_q4_moe_decode, "lily_q4_moe_decode", layer, x, y, topk_idx, topk_w,
                ws, stream)


def lily_q4_moe_prefill(layer: DeviceLayer, x, y, topk_idx=None, topk_w=None, ws=None, stream=None):
    """Prefill-chunk MoE (grouped tcgen05 GEMM); same arguments as lily_q4_moe_decode."""
    return _moe(load().lily_q4_moe_prefill, "lily_q4_moe_prefill", layer, x, y, topk_idx, topk_w,
                ws, stream)


def lily_q4_gemv_argmax(W: DeviceQ4, x, token, logits=None, ws=None, stream=None):
    N, K = int(W.w.shape[-2]), int(W.w.shape[-1]) * 8
    m = W.c()
    return _check(load().lily_q4_gemv_argmax(C.byref(m), N, K, _ptr(x), _ptr(token), _ptr(logits),
                                             _ptr(ws), ws.numel() if ws is not None else 0,
                                             _stream(stream)), "lily_q4_gemv_argmax")


def lily_q8_gemv_argmax(W, x, token, logits=None, ws=None, stream=None):
    """Greedy token of an 8-bit LM head (W: a DeviceQ4 holding uint32 [N, K/4] codes);
    see include/lily_q4.h."""
    N, K = int(W.w.shape[-2]), int(W.w.shape[-1]) * 4
    m = W.c()
    return _check(load().lily_q8_gemv_argmax(C.byref(m), N, K, _ptr(x), _ptr(token), _ptr(logits),
                                             _ptr(ws), ws.numel() if ws is not None else 0,
                                             _stream(stream)), "lily_q8_gemv_argmax")


def lily_q4_selftest_timeout(ws, which: int, stream=None):
    """Enqueue a wait that runs into its bound (which 0: grid barrier, 1: mbarrier); ws=None
    targets the fixed scratch of lily_q4_gemv_argmax_noalloc.  See include/lily_q4.h."""
    return _check(load().lily_q4_selftest_timeout(_ptr(ws), ws.numel() if ws is not None else 0,
                                                  int(which), _stream(stream)),
                  "lily_q4_selftest_timeout")


def lily_q8_gemv_argmax_logprobs(W, x, token, lse, logprobs=None, ws=None, stream=None):
    """lily_q4_gemv_argmax_logprobs for an 8-bit LM head; see include/lily_q4.h."""
    N, K = int(W.w.shape[-2]), int(W.w.shape[-1]) * 4
    m = W.c()
    return _check(load().lily_q8_gemv_argmax_logprobs(C.byref(m), N, K, _ptr(x), _ptr(token),
                                                      _ptr(lse), _ptr(logprobs), _ptr(ws),
                                                      ws.numel() if ws is not None else 0,
                                                      _stream(stream)),
                  "lily_q8_gemv_argmax_logprobs")


def lily_q8_gemv_argmax_workspace_bytes(N: int, K: int) -> int:
    return int(load().lily_q8_gemv_argmax_workspace_bytes(int(N), int(K)))


def lily_q4_gemv_argmax_logprobs(W: DeviceQ4, x, token, lse, logprobs=None, ws=None, stream=None):
    """Greedy token, full-vocabulary log-sum-exp (fp32 [1]) and optionally logprobs (fp32 [N])
    of a Q4 LM head in one pass; see include/lily_q4.h."""
    N, K = int(W.w.shape[-2]), int(W.w.shape[-1]) * 8
    m = W.c()
    return _check(load().lily_q4_gemv_argmax_logprobs(C.byref(m), N, K, _ptr(x), _ptr(token),
                                                      _ptr(lse), _ptr(logprobs), _ptr(ws),
                                                      ws.numel() if ws is not None else 0,
                                                      _stream(stream)),
                  "lily_q4_gemv_argmax_logprobs")


def lily_q4_gemv_argmax_noalloc(W: DeviceQ4, x, token, logits=None, stream=None):
    """lily_q4_gemv_argmax without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed array inside the library (see include/lily_q4.h)."""
    N, K = int(W.w.shape[-2]), int(W.w.shape[-1]) * 8
    m = W.c()
    return _check(load().lily_q4_gemv_argmax_noalloc(C.byref(m), N, K, _ptr(x), _ptr(token),
                                                     _ptr(logits), _stream(stream)),
                  "lily_q4_gemv_argmax_noalloc")


def lily_q4_gemv_argmax_noalloc_status(stream=None) -> int:
    """0, or ERR_TIMEOUT (returned, not raised) if a bounded device wait in a call of
    lily_q4_gemv_argmax_noalloc gave up since the last check; clears the record."""
    return int(load().lily_q4_gemv_argmax_noalloc_status(_stream(stream)))


def lily_q4_pack(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    w = np.empty((N, K // 8), dtype=np.uint32)
    _check(load().lily_q4_pack(q.ctypes.data, N, K, w.ctypes.data), "lily_q4_pack")
    return w


def lily_q4_unpack(w: np.ndarray, N: int, K: int) -> np.ndarray:
    w = np.ascontiguousarray(w, dtype=np.uint32)
    q = np.empty((N, K), dtype=np.uint8)
    _check(load().lily_q4_unpack(w.ctypes.data, N, K, q.ctypes.data), "lily_q4_unpack")
    return q
