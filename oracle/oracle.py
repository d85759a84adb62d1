"""Python front of the CPU oracle (``lily_q4_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the package smoke
check and by the benchmark's CPU-baseline leg, never by the CUDA product path.
It shares no code with the CUDA library; inputs come from the seeded generator
in ``bit_affine_quantized_mlx_gb300.synth``, which holds no arithmetic of the
method.

Every function below is a thin marshalling layer over the C definitions; the
arithmetic and the page passages it follows are documented in the C file.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lily_q4_oracle.c")
LIB = os.path.join(HERE, "liblily_q4_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fast-math, no FP contraction)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", SRC, "-o", LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(LIB + ".tmp", LIB)
    return LIB


class _Mat(C.Structure):
    _fields_ = [("w", C.c_void_p), ("s", C.c_void_p), ("b", C.c_void_p)]


class _Layer(C.Structure):
    _fields_ = [("H", C.c_int32), ("E", C.c_int32), ("k", C.c_int32), ("I", C.c_int32),
                ("gate", _Mat), ("up", _Mat), ("down", _Mat),
                ("has_shared", C.c_int32),
                ("sh_gate", _Mat), ("sh_up", _Mat), ("sh_down", _Mat),
                ("router", C.c_void_p), ("router_bias", C.c_void_p),
                ("shared_gate", C.c_void_p),
                ("shared_bits", C.c_int32), ("router_bits", C.c_int32), ("router8", _Mat)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        vp, i32 = C.c_void_p, C.c_int
        L.orc_q4_dequant.argtypes = [vp, vp, vp, i32, i32, vp]
        L.orc_q4_unpack.argtypes = [vp, i32, i32, vp]
        L.orc_q4_pack.argtypes = [vp, i32, i32, vp]
        L.orc_q4_matvec.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.orc_lm_head.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.orc_lm_head.restype = i32
        L.orc_q8_unpack.argtypes = [vp, i32, i32, vp]
        L.orc_q8_pack.argtypes = [vp, i32, i32, vp]
        L.orc_q8_dequant.argtypes = [vp, vp, vp, i32, i32, vp]
        L.orc_q8_lm_head.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.orc_q8_lm_head.restype = i32
        L.orc_log_sum_exp.argtypes = [vp, i32, vp]
        L.orc_log_sum_exp.restype = C.c_double
        L.orc_router.argtypes = [vp, vp, i32, i32, vp, vp]
        L.orc_topk.argtypes = [vp, i32, i32, vp, vp]
        L.orc_sigmoid_gate.argtypes = [vp, i32, vp]
        L.orc_sigmoid_gate.restype = C.c_double
        L.orc_expert.argtypes = [vp] * 9 + [i32, i32, vp, vp]
        L.orc_moe.argtypes = [C.POINTER(_Layer), vp, i32, vp, vp, vp, vp, vp]
        L.orc_router_tokens.argtypes = [C.POINTER(_Layer), vp, i32, vp]
        L.orc_threads.restype = i32
        L.orc_set_threads.argtypes = [i32]
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def threads() -> int:
    return int(lib().orc_threads())


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


# --------------------------------------------------------------------------- format

def q4_unpack(w: np.ndarray, N: int, K: int) -> np.ndarray:
    w = _c(w, np.uint32)
    q = np.empty((N, K), dtype=np.uint8)
    lib().orc_q4_unpack(_p(w), N, K, _p(q))
    return q


def q4_pack(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8)
    N, K = q.shape
    w = np.empty((N, K // 8), dtype=np.uint32)
    lib().orc_q4_pack(_p(q), N, K, _p(w))
    return w


def q4_dequant(m) -> np.ndarray:
    """Dense fp64 [N, K] of a (single) Q4 matrix."""
    w, s, b = _c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)
    N, K = w.shape[-2], w.shape[-1] * 8
    out = np.empty((N, K), dtype=np.float64)
    lib().orc_q4_dequant(_p(w), _p(s), _p(b), N, K, _p(out))
    return out


def q4_matvec(m, x: np.ndarray) -> np.ndarray:
    w, s, b = _c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)
    N, K = w.shape[-2], w.shape[-1] * 8
    x = _c(x, np.float64)
    out = np.empty(N, dtype=np.float64)
    lib().orc_q4_matvec(_p(w), _p(s), _p(b), N, K, _p(x), _p(out))
    return out


# --------------------------------------------------------------------------- LM head

def lm_head(m, x_bits: np.ndarray) -> Tuple[int, np.ndarray]:
    """fp64 logits of a Q4 LM head for one bf16 token, and the greedy argmax."""
    w, s, b = _c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)
    N, K = w.shape[-2], w.shape[-1] * 8
    x = _c(x_bits, np.uint16)
    logits = np.empty(N, dtype=np.float64)
    tok = lib().orc_lm_head(_p(w), _p(s), _p(b), N, K, _p(x), _p(logits))
    return int(tok), logits


def q8_unpack(w: np.ndarray, N: int, K: int) -> np.ndarray:
    w = _c(w, np.uint32)
    q = np.empty((N, K), dtype=np.uint8)
    lib().orc_q8_unpack(_p(w), N, K, _p(q))
    return q


def q8_pack(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8)
    N, K = q.shape
    w = np.empty((N, K // 4), dtype=np.uint32)
    lib().orc_q8_pack(_p(q), N, K, _p(w))
    return w


def q8_dequant(m) -> np.ndarray:
    """Dense fp64 [N, K] of an affine 8-bit matrix."""
    w, s, b = _c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)
    N, K = w.shape[-2], w.shape[-1] * 4
    out = np.empty((N, K), dtype=np.float64)
    lib().orc_q8_dequant(_p(w), _p(s), _p(b), N, K, _p(out))
    return out


def q8_lm_head(m, x_bits: np.ndarray) -> Tuple[int, np.ndarray]:
    """fp64 logits of an 8-bit LM head for one bf16 token, and the greedy argmax."""
    w, s, b = _c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)
    N, K = w.shape[-2], w.shape[-1] * 4
    x = _c(x_bits, np.uint16)
    logits = np.empty(N, dtype=np.float64)
    tok = lib().orc_q8_lm_head(_p(w), _p(s), _p(b), N, K, _p(x), _p(logits))
    return int(tok), logits


def log_softmax(logits: np.ndarray) -> Tuple[float, np.ndarray]:
    """Full-vocabulary log-sum-exp of fp64 logits and the log-probabilities l - lse."""
    l = _c(logits, np.float64)
    out = np.empty_like(l)
    lse = lib().orc_log_sum_exp(_p(l), int(l.size), _p(out))
    return float(lse), out


def lm_head_rows(m, x_bits: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """fp64 logits of selected rows only (for sampled checks at full size)."""
    rows = np.asarray(rows, dtype=np.int64)
    sub = type(m)(np.ascontiguousarray(m.w[rows]), np.ascontiguousarray(m.s[rows]),
                  np.ascontiguousarray(m.b[rows]))
    _, lg = lm_head(sub, x_bits)
    return lg


# --------------------------------------------------------------------------- routing

def router_logits(Wr_bits: np.ndarray, x_bits: np.ndarray, bias: Optional[np.ndarray] = None):
    Wr = _c(Wr_bits, np.uint16)
    E, H = Wr.shape
    x = _c(x_bits, np.uint16)
    bias = None if bias is None else _c(bias, np.float32)
    out = np.empty(E, dtype=np.float64)
    lib().orc_router(_p(Wr), _p(bias), E, H, _p(x), _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    lg = _c(logits, np.float64)
    idx = np.empty(k, dtype=np.int32)
    p = np.empty(k, dtype=np.float64)
    lib().orc_topk(_p(lg), lg.shape[0], k, _p(idx), _p(p))
    return idx, p


def sigmoid_gate(g_bits: np.ndarray, x_bits: np.ndarray) -> float:
    g, x = _c(g_bits, np.uint16), _c(x_bits, np.uint16)
    return float(lib().orc_sigmoid_gate(_p(g), g.shape[0], _p(x)))


def expert(gate, up, down, x: np.ndarray) -> np.ndarray:
    H, I = gate.K, gate.N
    arrs = []
    for m in (gate, up, down):
        arrs += [_c(m.w, np.uint32), _c(m.s, np.uint16), _c(m.b, np.uint16)]
    x = _c(x, np.float64)
    o = np.empty(H, dtype=np.float64)
    lib().orc_expert(*[_p(a) for a in arrs], H, I, _p(x), _p(o))
    return o


# --------------------------------------------------------------------------- whole layer

class _Keep:
    """Holds the contiguous arrays a _Layer struct points into."""

    def __init__(self):
        self.arrs = []

    def ptr(self, a, dtype):
        if a is None:
            return None
        a = _c(a, dtype)
        self.arrs.append(a)
        return a.ctypes.data


def _layer_struct(L) -> Tuple[_Layer, _Keep]:
    keep = _Keep()

    def mat(m):
        if m is None:
            return _Mat(None, None, None)
        return _Mat(keep.ptr(m.w, np.uint32), keep.ptr(m.s, np.uint16), keep.ptr(m.b, np.uint16))

    st = _Layer()
    st.H, st.E, st.k, st.I = L.H, L.E, L.k, L.I
    st.gate, st.up, st.down = mat(L.gate), mat(L.up), mat(L.down)
    st.has_shared = 1 if L.has_shared else 0
    st.sh_gate, st.sh_up, st.sh_down = mat(L.sh_gate), mat(L.sh_up), mat(L.sh_down)
    st.router = keep.ptr(L.router, np.uint16)
    st.router_bias = keep.ptr(L.router_bias, np.float32)
    st.shared_gate = keep.ptr(L.shared_gate, np.uint16)
    st.shared_bits = getattr(L, "shared_bits", 4)
    st.router_bits = getattr(L, "router_bits", 16)
    st.router8 = mat(getattr(L, "router_q8", None))
    return st, keep


def moe(L, x_bits: np.ndarray):
    """Whole MoE layer for tokens x [T, H] (bf16 bits).

    Returns dict with y [T,H] fp64, idx [T,k] int32, p [T,k] fp64,
    logits [T,E] fp64, sigma [T] fp64.
    """
    x = _c(np.atleast_2d(x_bits), np.uint16)
    T = x.shape[0]
    st, keep = _layer_struct(L)
    y = np.empty((T, L.H), dtype=np.float64)
    idx = np.empty((T, L.k), dtype=np.int32)
    p = np.empty((T, L.k), dtype=np.float64)
    lg = np.empty((T, L.E), dtype=np.float64)
    sig = np.empty(T, dtype=np.float64)
    lib().orc_moe(C.byref(st), _p(x), T, _p(y), _p(idx), _p(p), _p(lg), _p(sig))
    del keep
    return {"y": y, "idx": idx, "p": p, "logits": lg, "sigma": sig}


def router_tokens(L, x_bits: np.ndarray) -> np.ndarray:
    """fp64 router logits [T, E] (offsets included) for tokens x [T, H]."""
    x = _c(np.atleast_2d(x_bits), np.uint16)
    T = x.shape[0]
    st, keep = _layer_struct(L)
    lg = np.empty((T, L.E), dtype=np.float64)
    lib().orc_router_tokens(C.byref(st), _p(x), T, _p(lg))
    del keep
    return lg


# --------------------------------------------------------------------------- near-tie rule

TIE_GAP = 1e-3


def topk_gap(logits_row: np.ndarray, k: int) -> float:
    """Gap between the k-th and (k+1)-th largest logit (inf when k == E)."""
    if k >= logits_row.shape[0]:
        return float("inf")
    srt = np.sort(logits_row)[::-1]
    return float(srt[k - 1] - srt[k])


def tokens_without_near_ties(L, draw, T: int, max_attempts: int = 64):
    """Draw x [T, H] with ``draw(t, attempt)``, redrawing row t until the oracle's
    k-th and (k+1)-th router logits differ by at least 1e-3.

    Returns (x bits [T,H], attempts [T])."""
    x = np.stack([draw(t, 0) for t in range(T)])
    attempts = np.zeros(T, dtype=np.int64)
    lg = router_tokens(L, x)
    for t in range(T):
        while topk_gap(lg[t], L.k) < TIE_GAP:
            attempts[t] += 1
            if attempts[t] > max_attempts:
                raise RuntimeError("no draw without a near-tie")
            x[t] = draw(t, int(attempts[t]))
            lg[t] = router_tokens(L, x[t:t + 1])[0]
    return x, attempts


def lm_x_without_near_tie(m, draw, max_attempts: int = 64, head=None):
    """Redraw x until the oracle's top-2 LM-head logits differ by at least 1e-3 (head: the
    oracle LM head to use, lm_head for 4-bit weights by default, q8_lm_head for 8-bit)."""
    head = head or lm_head
    for a in range(max_attempts):
        x = draw(a)
        tok, lg = head(m, x)
        srt = np.sort(lg)
        if srt[-1] - srt[-2] >= TIE_GAP:
            return x, a, tok, lg
    raise RuntimeError("no draw without a near-tie")
