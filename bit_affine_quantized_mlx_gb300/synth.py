"""Seeded synthetic inputs for the Q4 MoE hot path.

This module only draws numbers.  It holds none of the method's arithmetic: no
dequantisation, no dot products, no routing.  Both the CUDA path (tests, bench)
and the CPU oracle (tests) take their inputs from here, so the two sides see the
same bits.

Storage formats drawn here (MLX affine 4-bit, group size 64, as named in the
Lily README "Requirements" section and in the Lily-vs-MLX performance report's
"Hardware and software" section):

* ``w``: uint32 ``[..., N, K/8]`` -- eight 4-bit codes per word along K, the
  lowest nibble first.  Codes are uniform on 0..15, which is the same as drawing
  every word uniformly on 0..2**32-1.
* ``s``: bf16 bit patterns (uint16) ``[..., N, K/64]`` -- per-group scale,
  drawn U(0.002, 0.02).
* ``b``: bf16 bit patterns ``[..., N, K/64]`` -- per-group bias, drawn as
  ``-8 * s * (1 + N(0, 0.05))`` from the *rounded* scale.

Every array is drawn from ``numpy.random.Generator(PCG64(SeedSequence(key)))``
with a key that names the workload, the layer, the tensor and (for expert
stacks) the expert, so any expert can be re-drawn on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional, Tuple

import numpy as np

GROUP = 64

# Stream ids inside a seed key.
S_ROUTER, S_GSHARED, S_RBIAS = 1, 2, 3
S_GATE, S_UP, S_DOWN = 10, 11, 12
S_SH_GATE, S_SH_UP, S_SH_DOWN = 20, 21, 22
S_X = 100
S_LM = 30
S_LM8 = 31
S_ROUTER8 = 4
S_SH_GATE8, S_SH_UP8, S_SH_DOWN8 = 24, 25, 26


def bf16_from_f32(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bit patterns."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


@dataclass
class Q4Matrix:
    """One MLX-affine Q4 matrix (or a stack of them along a leading expert axis)."""
    w: np.ndarray  # uint32 [..., N, K/8]
    s: np.ndarray  # uint16 bf16 bits [..., N, K/64]
    b: np.ndarray  # uint16 bf16 bits [..., N, K/64]

    @property
    def N(self) -> int:
        return int(self.w.shape[-2])

    @property
    def K(self) -> int:
        return int(self.w.shape[-1]) * 8

    @property
    def nbytes(self) -> int:
        return self.w.nbytes + self.s.nbytes + self.b.nbytes


@dataclass
class Q8Matrix:
    """One MLX-affine 8-bit matrix: codes uint32 [N, K/4] (four codes per word along K, lowest
    byte first), bf16 scales and biases [N, K/64]."""
    w: np.ndarray
    s: np.ndarray
    b: np.ndarray

    @property
    def N(self) -> int:
        return int(self.w.shape[-2])

    @property
    def K(self) -> int:
        return int(self.w.shape[-1]) * 4

    @property
    def nbytes(self) -> int:
        return self.w.nbytes + self.s.nbytes + self.b.nbytes


def draw_q8(N: int, K: int, *key: int) -> Q8Matrix:
    """Draw one 8-bit matrix [N x K]: codes uniform 0..255, s ~ U(0.000125, 0.00125) (the 4-bit
    range over 16x the levels), b = -128 s (1 + N(0, 0.05)), both rounded to bf16."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    g = _rng(*key)
    w = g.integers(0, 2**32, size=(N, K // 4), dtype=np.uint32)
    s64 = g.uniform(0.000125, 0.00125, size=(N, K // GROUP))
    s = bf16_from_f32(s64.astype(np.float32))
    eps = g.normal(0.0, 0.05, size=(N, K // GROUP))
    b64 = -128.0 * bf16_to_f32(s).astype(np.float64) * (1.0 + eps)
    b = bf16_from_f32(b64.astype(np.float32))
    return Q8Matrix(w, s, b)


def draw_q4(N: int, K: int, *key: int) -> Q4Matrix:
    """Draw one Q4 matrix [N x K] with the workload's value distributions."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 64")
    g = _rng(*key)
    w = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s64 = g.uniform(0.002, 0.02, size=(N, K // GROUP))
    s = bf16_from_f32(s64.astype(np.float32))
    eps = g.normal(0.0, 0.05, size=(N, K // GROUP))
    b64 = -8.0 * bf16_to_f32(s).astype(np.float64) * (1.0 + eps)
    b = bf16_from_f32(b64.astype(np.float32))
    return Q4Matrix(w, s, b)


def draw_q4_stack(E: int, N: int, K: int, *key: int) -> Q4Matrix:
    """Draw E independently seeded Q4 matrices stacked as [E, N, ...]."""
    w = np.empty((E, N, K // 8), dtype=np.uint32)
    s = np.empty((E, N, K // GROUP), dtype=np.uint16)
    b = np.empty((E, N, K // GROUP), dtype=np.uint16)
    for e in range(E):
        m = draw_q4(N, K, *key, e)
        w[e], s[e], b[e] = m.w, m.s, m.b
    return Q4Matrix(w, s, b)


def draw_bf16_normal(shape, std: float, *key: int) -> np.ndarray:
    g = _rng(*key)
    return bf16_from_f32(g.normal(0.0, std, size=shape).astype(np.float32))


@dataclass
class MoELayer:
    """Host copy of one synthetic MoE layer (bit patterns, ready to upload)."""
    H: int
    E: int
    k: int
    I: int
    gate: Q4Matrix          # [E, I, H]
    up: Q4Matrix            # [E, I, H]
    down: Q4Matrix          # [E, H, I]
    router: np.ndarray      # uint16 bf16 [E, H]
    router_bias: Optional[np.ndarray] = None   # float32 [E]
    sh_gate: Optional[Q4Matrix] = None       # [I, H]
    sh_up: Optional[Q4Matrix] = None         # [I, H]
    sh_down: Optional[Q4Matrix] = None       # [H, I]
    shared_gate: Optional[np.ndarray] = None  # uint16 bf16 [H]
    router_q8: Optional["Q8Matrix"] = None   # [E, H] affine 8-bit router (replaces router)

    @property
    def has_shared(self) -> bool:
        return self.sh_gate is not None

    @property
    def shared_bits(self) -> int:
        """Code width of the shared expert: 8 for Q8Matrix matrices (q4-xl), else 4."""
        return 8 if isinstance(self.sh_gate, Q8Matrix) else 4

    @property
    def router_bits(self) -> int:
        """16 for the bf16 router, 8 for an affine 8-bit router."""
        return 8 if self.router_q8 is not None else 16

    def expert_bytes(self) -> int:
        """Bytes of one routed expert (gate + up + down, codes and scales)."""
        return (self.gate.nbytes + self.up.nbytes + self.down.nbytes) // self.E


def draw_layer(H: int, E: int, k: int, I: int, *, shared: bool, router_std: float,
               router_bias: bool, key: Tuple[int, ...], router_bits: int = 16,
               shared_bits: int = 4) -> MoELayer:
    """Draw one MoE layer.  ``key`` = (workload id, layer index).  router_bits = 8 draws an
    affine 8-bit router (the checkpoint's router gates); shared_bits = 8 an 8-bit shared expert
    (the q4-xl conversion)."""
    gate = draw_q4_stack(E, I, H, *key, S_GATE)
    up = draw_q4_stack(E, I, H, *key, S_UP)
    down = draw_q4_stack(E, H, I, *key, S_DOWN)
    router = draw_bf16_normal((E, H), router_std, *key, S_ROUTER)
    rb = None
    if router_bias:
        rb = _rng(*key, S_RBIAS).normal(0.0, 1.0, size=E).astype(np.float32)
    L = MoELayer(H, E, k, I, gate, up, down, router, rb)
    if router_bits == 8:
        L.router = None
        L.router_q8 = draw_q8(E, H, *key, S_ROUTER8)
    if shared:
        if shared_bits == 8:
            L.sh_gate = draw_q8(I, H, *key, S_SH_GATE8)
            L.sh_up = draw_q8(I, H, *key, S_SH_UP8)
            L.sh_down = draw_q8(H, I, *key, S_SH_DOWN8)
        else:
            L.sh_gate = draw_q4(I, H, *key, S_SH_GATE)
            L.sh_up = draw_q4(I, H, *key, S_SH_UP)
            L.sh_down = draw_q4(H, I, *key, S_SH_DOWN)
        L.shared_gate = draw_bf16_normal((H,), 0.05, *key, S_GSHARED)
    return L


def draw_x(H: int, key: Tuple[int, ...], t: int, attempt: int = 0) -> np.ndarray:
    """Token t's activation row, bf16 ~ N(0,1).  ``attempt`` > 0 gives a fresh redraw."""
    return draw_bf16_normal((H,), 1.0, *key, S_X, t, attempt)


def draw_tokens(H: int, T: int, key: Tuple[int, ...], attempts=None) -> np.ndarray:
    """x [T, H] bf16 bits; ``attempts[t]`` selects the redraw of row t (default 0)."""
    x = np.empty((T, H), dtype=np.uint16)
    for t in range(T):
        x[t] = draw_x(H, key, t, 0 if attempts is None else int(attempts[t]))
    return x


# ---------------------------------------------------------------------------
# The five workloads (hidden, experts, top-k, expert intermediate, shared, ...)
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    H: int
    E: int = 0
    k: int = 0
    I: int = 0
    shared: bool = False
    router_std: float = 0.0
    router_bias: bool = False
    tokens: Tuple[int, ...] = (1,)
    layers: int = 1
    V: int = 0

    def layer(self, l: int) -> MoELayer:
        return draw_layer(self.H, self.E, self.k, self.I, shared=self.shared,
                          router_std=self.router_std, router_bias=self.router_bias,
                          key=(self.wid, l))

    def tokens_key(self, l: int) -> Tuple[int, ...]:
        return (self.wid, l)


TINY = Workload(0, "tiny moe H256 E16 k2 I128", H=256, E=16, k=2, I=128, shared=False,
                router_std=0.05, tokens=(1,), layers=1)
DECODE = Workload(1, "decode moe H2048 E256 k8 I512 +shared", H=2048, E=256, k=8, I=512,
                  shared=True, router_std=0.02, tokens=(1, 4), layers=40)
LMHEAD = Workload(2, "lm head Q4 V151936 H2048 + argmax", H=2048, V=151936)
PREFILL = Workload(3, "prefill chunk T2048 H2048 E256 k8 I512 +shared, skewed router", H=2048,
                   E=256, k=8, I=512, shared=True, router_std=0.02, router_bias=True,
                   tokens=(2048,), layers=1)
WIDE = Workload(4, "wide moe H2048 E512 k10 I512 +shared", H=2048, E=512, k=10, I=512,
                shared=True, router_std=0.02, tokens=(1, 2, 4), layers=48)

WORKLOADS: Dict[int, Workload] = {w.wid: w for w in (TINY, DECODE, LMHEAD, PREFILL, WIDE)}


def draw_lm_head(V: int = 151936, H: int = 2048, key=(2, 0)) -> Q4Matrix:
    return draw_q4(V, H, *key, S_LM)


def draw_lm_head_q8(V: int = 151936, H: int = 2048, key=(2, 0)) -> Q8Matrix:
    """The LM head kept at 8 bits (the q4-xl conversion)."""
    return draw_q8(V, H, *key, S_LM8)


def draw_lm_x(H: int = 2048, key=(2, 0), attempt: int = 0) -> np.ndarray:
    return draw_x(H, key, 0, attempt)
