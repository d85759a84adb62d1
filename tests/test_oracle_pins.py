"""Pins of the CPU oracle against facts that do not come from the oracle itself.

The pages print no worked numeric example for this path, so the pins are closed
forms, special cases that reduce to a library routine, invariants and brute
force on tiny inputs.  Each test names the plausible mistake it would catch.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special as sp

from bit_affine_quantized_mlx_gb300 import synth
from bit_affine_quantized_mlx_gb300.synth import Q4Matrix, bf16_from_f32, bf16_to_f32
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _bf16(v):
    return bf16_from_f32(np.float32(v)).item()


def _mat_from_codes(q, s_val=1.0, b_val=0.0, s=None, b=None):
    """Q4Matrix from an explicit code array q [N, K] and constant or per-group s/b."""
    q = np.asarray(q, dtype=np.uint8)
    N, K = q.shape
    w = orc.q4_pack(q)
    if s is None:
        s = np.full((N, K // 64), _bf16(s_val), dtype=np.uint16)
    if b is None:
        b = np.full((N, K // 64), _bf16(b_val), dtype=np.uint16)
    return Q4Matrix(w, np.asarray(s, np.uint16), np.asarray(b, np.uint16))


# ----------------------------------------------------------------------------- format

def test_nibble_order_golden():
    """Codes 0..7 pack to 0x76543210 (lowest nibble first); catches a reversed nibble order."""
    for codes, word in _read_golden("q4_nibble_order.txt"):
        q = np.array([[int(c, 16) for c in codes.split(",")]], dtype=np.uint8)
        assert orc.q4_pack(q)[0, 0] == int(word, 16)
        assert list(orc.q4_unpack(np.array([[int(word, 16)]], np.uint32), 1, 8)[0]) == list(q[0])


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(1)
    w = rng.integers(0, 2**32, size=(7, 16), dtype=np.uint32)
    q = orc.q4_unpack(w, 7, 128)
    assert q.max() <= 15
    assert np.array_equal(orc.q4_pack(q), w)


def test_dequant_extreme_codes_exact():
    """q=0 gives exactly b, q=15 gives exactly 15s+b (both exact in fp32 and fp64 here)."""
    rng = np.random.default_rng(2)
    N, K = 8, 128
    for code in (0, 15):
        q = np.full((N, K), code, dtype=np.uint8)
        m = synth.draw_q4(N, K, 99, 1)
        m = Q4Matrix(orc.q4_pack(q), m.s, m.b)
        W = orc.q4_dequant(m)
        s = bf16_to_f32(m.s).astype(np.float64)
        b = bf16_to_f32(m.b).astype(np.float64)
        want = np.repeat(code * s + b, 64, axis=1)   # exact: bf16 operands, <= 12-bit products
        assert np.array_equal(W, want)


def test_dequant_group_and_row_indexing():
    """A distinct scale per (row, group) and a code per column: catches k/8 vs k/64 group
    indexing and row/column transposition (N != K)."""
    N, K = 3, 192
    q = (np.arange(N * K).reshape(N, K) % 16).astype(np.uint8)
    s = np.array([[_bf16(2.0 ** -(n + 1) * (g + 1)) for g in range(K // 64)] for n in range(N)],
                 dtype=np.uint16)
    b = np.array([[_bf16(-(n * 4 + g)) for g in range(K // 64)] for n in range(N)], dtype=np.uint16)
    m = _mat_from_codes(q, s=s, b=b)
    W = orc.q4_dequant(m)
    for n in range(N):
        for k in range(K):
            g = k // 64
            want = 2.0 ** -(n + 1) * (g + 1) * ((n * K + k) % 16) - (n * 4 + g)
            assert W[n, k] == want


# ----------------------------------------------------------------------------- GEMV closed forms

def test_identity_matvec():
    """s=1, b=0, q=identity gives W x = x exactly."""
    K = 128
    q = np.eye(K, dtype=np.uint8)
    m = _mat_from_codes(q, 1.0, 0.0)
    x = bf16_to_f32(synth.draw_bf16_normal((K,), 1.0, 5)).astype(np.float64)
    assert np.array_equal(orc.q4_matvec(m, x), x)


def test_bias_only_matvec():
    """All codes 0: (W x)_n = sum_g b[n,g] * sum_{k in g} x_k."""
    N, K = 5, 256
    m0 = synth.draw_q4(N, K, 7, 7)
    m = Q4Matrix(np.zeros_like(m0.w), m0.s, m0.b)
    x = bf16_to_f32(synth.draw_bf16_normal((K,), 1.0, 8)).astype(np.float64)
    b = bf16_to_f32(m.b).astype(np.float64)
    gs = x.reshape(K // 64, 64).sum(axis=1)   # exact: 64 bf16 values in fp64
    want = b @ gs
    np.testing.assert_allclose(orc.q4_matvec(m, x), want, rtol=1e-13, atol=1e-13)


def test_one_hot_column():
    """x = e_j returns column j of the dequantised matrix (N != K)."""
    N, K = 6, 192
    m = synth.draw_q4(N, K, 9, 9)
    W = orc.q4_dequant(m)
    for j in (0, 63, 64, 100, 191):
        x = np.zeros(K)
        x[j] = 1.0
        assert np.array_equal(orc.q4_matvec(m, x), W[:, j])


def test_matvec_matches_blas_on_dequantised():
    """Library matmul over the dequantised matrix agrees (catches an accumulation bug)."""
    m = synth.draw_q4(33, 320, 11, 1)
    x = bf16_to_f32(synth.draw_bf16_normal((320,), 1.0, 12)).astype(np.float64)
    np.testing.assert_allclose(orc.q4_matvec(m, x), orc.q4_dequant(m) @ x, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- routing

def test_topk_invariants():
    rng = np.random.default_rng(3)
    for E, k in ((16, 2), (256, 8), (512, 10)):
        lg = rng.normal(0, 1, E)
        idx, p = orc.topk(lg, k)
        assert len(set(idx.tolist())) == k
        assert np.all(p > 0)
        assert abs(p.sum() - 1.0) < 1e-12
        assert np.all(np.diff(lg[idx]) <= 0)
        assert lg[idx].min() >= np.sort(lg)[::-1][k - 1]


def test_topk_zero_router_picks_first_k():
    """Wr = 0: all logits equal, experts 0..k-1 with p = 1/k exactly."""
    E, H, k = 16, 256, 4
    Wr = np.zeros((E, H), dtype=np.uint16)
    x = synth.draw_bf16_normal((H,), 1.0, 13)
    lg = orc.router_logits(Wr, x)
    idx, p = orc.topk(lg, k)
    assert idx.tolist() == [0, 1, 2, 3]
    assert np.all(p == 0.25)


def test_topk_brute_force_subsets():
    """Over all C(E,k) subsets, the top-k set maximises the logit sum; exact ties go to the
    lexicographically smallest subset (lower indices)."""
    rng = np.random.default_rng(4)
    for trial in range(40):
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-3, 4, size=E).astype(np.float64)   # many exact ties
        best = None
        for sub in itertools.combinations(range(E), k):
            key = (lg[list(sub)].sum(), [-i for i in sub])
            if best is None or key > best[0]:
                best = (key, sub)
        idx, _ = orc.topk(lg, k)
        assert sorted(idx.tolist()) == list(best[1]), (lg, k)


def test_gates_match_full_softmax_renormalised():
    """p equals a library softmax over all E, renormalised over the selected k."""
    rng = np.random.default_rng(5)
    lg = rng.normal(0, 2, 64)
    idx, p = orc.topk(lg, 6)
    full = sp.softmax(lg)
    want = full[idx] / full[idx].sum()
    np.testing.assert_allclose(p, want, rtol=1e-13)
    idx2, p2 = orc.topk(lg + 123.0, 6)
    assert np.array_equal(idx, idx2)
    np.testing.assert_allclose(p2, p, rtol=1e-12)


def test_top1_gate_is_one():
    idx, p = orc.topk(np.array([0.1, 3.0, -2.0]), 1)
    assert idx.tolist() == [1] and p[0] == 1.0


def test_router_bias_added():
    """A large per-expert offset moves the selection (catches a dropped bias)."""
    E, H = 8, 64
    Wr = synth.draw_bf16_normal((E, H), 0.02, 14)
    x = synth.draw_bf16_normal((H,), 1.0, 15)
    bias = np.zeros(E, np.float32)
    bias[5] = 100.0
    lg = orc.router_logits(Wr, x, bias)
    lg0 = orc.router_logits(Wr, x)
    np.testing.assert_allclose(lg - lg0, bias.astype(np.float64), atol=1e-12)
    assert orc.topk(lg, 1)[0][0] == 5


# ----------------------------------------------------------------------------- gating closed forms

def test_shared_gate_zero_is_half():
    g = np.zeros(128, np.uint16)
    x = synth.draw_bf16_normal((128,), 1.0, 16)
    assert orc.sigmoid_gate(g, x) == 0.5


def test_shared_gate_matches_library_sigmoid():
    g = synth.draw_bf16_normal((256,), 0.05, 17)
    x = synth.draw_bf16_normal((256,), 1.0, 18)
    d = float(bf16_to_f32(g).astype(np.float64) @ bf16_to_f32(x).astype(np.float64))
    assert abs(orc.sigmoid_gate(g, x) - sp.expit(d)) < 1e-15


def test_swiglu_expert_closed_form():
    """Wg = 2*I, Wu = I, Wd = I gives o = silu(2x) * x; swapping gate and up would give
    silu(x) * 2x and fail."""
    H = I = 64
    eye = np.eye(H, dtype=np.uint8)
    Wg = _mat_from_codes(eye, 2.0, 0.0)
    Wu = _mat_from_codes(eye, 1.0, 0.0)
    Wd = _mat_from_codes(eye, 1.0, 0.0)
    x = bf16_to_f32(synth.draw_bf16_normal((H,), 1.0, 19)).astype(np.float64)
    o = orc.expert(Wg, Wu, Wd, x)
    want = 2 * x * sp.expit(2 * x) * x
    np.testing.assert_allclose(o, want, rtol=1e-14, atol=1e-15)


def test_zero_gate_weights_give_zero_output():
    """silu(0) = 0: an expert whose gate projection is identically zero contributes nothing."""
    L = synth.draw_layer(64, 4, 2, 64, shared=False, router_std=0.05, router_bias=False,
                         key=(90, 0))
    L.gate = Q4Matrix(np.zeros_like(L.gate.w), np.zeros_like(L.gate.s), np.zeros_like(L.gate.b))
    x = synth.draw_tokens(64, 3, (90, 0))
    out = orc.moe(L, x)
    assert np.all(out["y"] == 0.0)


# ----------------------------------------------------------------------------- whole layer

def _np_dense(m):
    """Independent dense dequantisation with numpy bit operations."""
    w = np.asarray(m.w, np.uint32)
    shifts = (np.arange(8, dtype=np.uint32) * 4)
    q = ((w[..., None] >> shifts) & 0xF).reshape(*w.shape[:-1], w.shape[-1] * 8)
    s = np.repeat(bf16_to_f32(m.s), 64, axis=-1)
    b = np.repeat(bf16_to_f32(m.b), 64, axis=-1)
    return (s * q.astype(np.float32) + b).astype(np.float64)


def _np_dense8(m):
    """Independent dense dequantisation of 8-bit codes with numpy byte views."""
    w = np.ascontiguousarray(m.w, np.uint32)
    q = w.astype("<u4").view(np.uint8).reshape(*w.shape[:-1], w.shape[-1] * 4)  # little-endian bytes
    s = np.repeat(bf16_to_f32(m.s), 64, axis=-1)
    b = np.repeat(bf16_to_f32(m.b), 64, axis=-1)
    return (s * q.astype(np.float32) + b).astype(np.float64)


def _np_any(m):
    return _np_dense8(m) if isinstance(m, synth.Q8Matrix) else _np_dense(m)


def _np_moe(L, x_bits):
    x = bf16_to_f32(x_bits).astype(np.float64)
    R = _np_dense8(L.router_q8) if L.router_q8 is not None else bf16_to_f32(L.router).astype(np.float64)
    lg = x @ R.T
    if L.router_bias is not None:
        lg = lg + L.router_bias.astype(np.float64)
    G, U, D = _np_dense(L.gate), _np_dense(L.up), _np_dense(L.down)
    y = np.zeros_like(x)
    for t in range(x.shape[0]):
        order = sorted(range(L.E), key=lambda e: (-lg[t, e], e))[:L.k]
        w = np.exp(lg[t, order] - lg[t, order[0]])
        w /= w.sum()
        for wi, e in zip(w, order):
            g = np.einsum("ih,h->i", G[e], x[t])
            u = np.einsum("ih,h->i", U[e], x[t])
            y[t] += wi * np.einsum("hi,i->h", D[e], g * sp.expit(g) * u)
        if L.has_shared:
            sg = sp.expit(bf16_to_f32(L.shared_gate).astype(np.float64) @ x[t])
            g = _np_any(L.sh_gate) @ x[t]
            u = _np_any(L.sh_up) @ x[t]
            y[t] += sg * (_np_any(L.sh_down) @ (g * sp.expit(g) * u))
    return y


@pytest.mark.parametrize("H,E,k,I,shared,bias", [
    (64, 4, 2, 64, False, False), (128, 8, 3, 64, True, False), (128, 6, 6, 128, True, True)])
def test_whole_layer_vs_independent_numpy(H, E, k, I, shared, bias):
    L = synth.draw_layer(H, E, k, I, shared=shared, router_std=0.05, router_bias=bias,
                         key=(91, H + E))
    x = synth.draw_tokens(H, 3, (91, H + E))
    got = orc.moe(L, x)["y"]
    want = _np_moe(L, x)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


@pytest.mark.parametrize("router_bits,shared_bits", [(8, 4), (16, 8), (8, 8)])
def test_whole_layer_8bit_parts_vs_independent_numpy(router_bits, shared_bits):
    """An 8-bit router (the checkpoint's router gates) and/or an 8-bit shared expert (q4-xl):
    the oracle layer against numpy with byte-view dequantisation (catches the 8-bit parts read
    as 4-bit, or the bf16 router used in place of the 8-bit one)."""
    L = synth.draw_layer(128, 8, 3, 64, shared=True, router_std=0.05, router_bias=True,
                         key=(93, router_bits + shared_bits), router_bits=router_bits,
                         shared_bits=shared_bits)
    assert L.router_bits == router_bits and L.shared_bits == shared_bits
    x = synth.draw_tokens(128, 3, (93, 1))
    out = orc.moe(L, x)
    want = _np_moe(L, x)
    np.testing.assert_allclose(out["y"], want, rtol=1e-12, atol=1e-12 * np.abs(want).max())
    R = _np_dense8(L.router_q8) if router_bits == 8 else bf16_to_f32(L.router).astype(np.float64)
    lg = bf16_to_f32(x).astype(np.float64) @ R.T + L.router_bias.astype(np.float64)
    np.testing.assert_allclose(out["logits"], lg, rtol=1e-12, atol=1e-12)


def test_moe_tokens_independent():
    """Prefill = the same per-token computation: a batch equals tokens run one by one."""
    L = synth.draw_layer(128, 8, 2, 64, shared=True, router_std=0.05, router_bias=True, key=(92, 0))
    x = synth.draw_tokens(128, 4, (92, 0))
    full = orc.moe(L, x)
    for t in range(4):
        one = orc.moe(L, x[t:t + 1])
        assert np.array_equal(one["y"][0], full["y"][t])
        assert np.array_equal(one["idx"][0], full["idx"][t])


# ----------------------------------------------------------------------------- argmax

def test_lm_head_planted_max_and_tie():
    """Rows 3 and 9 are identical and dominant: argmax is the lower id 3."""
    N, K = 16, 128
    q = np.zeros((N, K), np.uint8)
    q[3] = 15
    q[9] = 15
    m = _mat_from_codes(q, 1.0, 0.0)
    x = np.full(K, _bf16(1.0), np.uint16)
    tok, lg = orc.lm_head(m, x)
    assert tok == 3
    assert lg[3] == lg[9] == 15.0 * K
    q[9, 0] = 14   # now row 3 alone holds the max
    q[12] = 15
    q[12, 5] = 14
    m = _mat_from_codes(q, 1.0, 0.0)
    tok, _ = orc.lm_head(m, x)
    assert tok == 3


def test_lm_head_matches_matvec():
    m = synth.draw_q4(40, 256, 20, 1)
    x = synth.draw_bf16_normal((256,), 1.0, 21)
    tok, lg = orc.lm_head(m, x)
    want = orc.q4_matvec(m, bf16_to_f32(x).astype(np.float64))
    assert np.array_equal(lg, want)
    assert tok == int(np.argmax(want))


# ----------------------------------------------------------------------------- log-sum-exp

def test_lse_uniform_closed_form():
    """N equal logits c: lse = c + log N, every logprob = -log N (catches returning the max
    alone, or forgetting to add the maximum back)."""
    for N, c in ((1, 0.0), (7, 2.5), (151936, -3.25)):
        lse, lp = orc.log_softmax(np.full(N, c))
        assert lse == pytest.approx(c + math.log(N), rel=0, abs=1e-12)
        assert np.allclose(lp, -math.log(N), rtol=0, atol=1e-12)


def test_lse_two_values_closed_form():
    """lse(a, b) = max + log1p(exp(-|a - b|)) (catches a dropped term of the sum)."""
    for a, b in ((0.0, 0.0), (3.0, -1.0), (-2.0, 5.5), (700.0, 699.0)):
        lse, _ = orc.log_softmax(np.array([a, b]))
        assert lse == pytest.approx(max(a, b) + math.log1p(math.exp(-abs(a - b))), rel=1e-15)


def test_lse_matches_library_and_normalises():
    """Random logits: scipy's logsumexp agrees, exp(logprobs) sums to one and the shift by a
    constant moves lse by that constant (catches a wrong sign or a missing shift)."""
    rng = np.random.default_rng(5)
    l = rng.normal(0.0, 4.0, 5000)
    lse, lp = orc.log_softmax(l)
    assert lse == pytest.approx(float(sp.logsumexp(l)), rel=1e-14)
    assert math.fsum(np.exp(lp)) == pytest.approx(1.0, abs=1e-12)
    lse2, lp2 = orc.log_softmax(l + 123.0)
    assert lse2 == pytest.approx(lse + 123.0, rel=1e-14)
    assert np.allclose(lp2, lp, rtol=0, atol=1e-10)
    assert np.all(lp <= 0.0) and lp.argmax() == l.argmax()


def test_lse_non_finite():
    inf, nan = math.inf, math.nan
    assert orc.log_softmax(np.array([0.0, inf, 1.0]))[0] == inf
    assert orc.log_softmax(np.array([-inf, -inf]))[0] == -inf
    assert math.isnan(orc.log_softmax(np.array([0.0, nan, 1.0]))[0])
    lse, lp = orc.log_softmax(np.array([-inf, 0.0]))   # a -inf logit adds nothing
    assert lse == 0.0 and lp[0] == -inf


# ----------------------------------------------------------------------------- affine 8-bit

def _q8(q, s, b):
    return synth.Q8Matrix(orc.q8_pack(q), np.asarray(s, np.uint16), np.asarray(b, np.uint16))


def test_q8_byte_order_golden():
    """Codes 1,2,3,4 pack to 0x04030201 (lowest byte first); catches a reversed byte order or
    4-bit fields."""
    for codes, word in _read_golden("q8_byte_order.txt"):
        q = np.array([[int(c, 16) for c in codes.split(",")]], dtype=np.uint8)
        assert orc.q8_pack(q)[0, 0] == int(word, 16)
        assert list(orc.q8_unpack(np.array([[int(word, 16)]], np.uint32), 1, 4)[0]) == list(q[0])


def test_q8_pack_unpack_roundtrip():
    rng = np.random.default_rng(11)
    w = rng.integers(0, 2**32, size=(5, 32), dtype=np.uint32)
    q = orc.q8_unpack(w, 5, 128)
    assert q.max() > 15   # all eight bits of a code are kept
    assert np.array_equal(orc.q8_pack(q), w)


def test_q8_dequant_extreme_codes_exact():
    """With s = 2^-8 and b = -1/2: q=0 gives exactly -1/2, q=255 exactly 255/256 - 1/2."""
    N, K = 4, 128
    for code, want in ((0, -0.5), (255, 255.0 / 256.0 - 0.5), (128, 0.0)):
        q = np.full((N, K), code, dtype=np.uint8)
        m = _q8(q, np.full((N, 2), _bf16(2.0 ** -8), np.uint16), np.full((N, 2), _bf16(-0.5), np.uint16))
        assert np.all(orc.q8_dequant(m) == want)


def test_q8_dequant_group_and_row_indexing():
    """A distinct scale per (row, group) and a code per column (N != K): catches k/4 vs k/64
    group indexing and transposition."""
    N, K = 3, 192
    q = (np.arange(N * K).reshape(N, K) % 256).astype(np.uint8)
    s = np.array([[_bf16(2.0 ** -(n + 3) * (g + 1)) for g in range(K // 64)] for n in range(N)],
                 dtype=np.uint16)
    b = np.array([[_bf16(-(n * 4 + g)) for g in range(K // 64)] for n in range(N)], dtype=np.uint16)
    W = orc.q8_dequant(_q8(q, s, b))
    for n in range(N):
        for k in range(K):
            g = k // 64
            assert W[n, k] == 2.0 ** -(n + 3) * (g + 1) * ((n * K + k) % 256) - (n * 4 + g)


def test_q8_lm_head_matches_library_matmul():
    """Logits equal numpy's matrix-vector product of the dequantised matrix (both in fp64, up
    to summation order), argmax included."""
    m = synth.draw_q8(300, 256, 40, 1)
    x = synth.draw_bf16_normal((256,), 1.0, 41)
    tok, lg = orc.q8_lm_head(m, x)
    want = orc.q8_dequant(m) @ bf16_to_f32(x).astype(np.float64)
    assert np.allclose(lg, want, rtol=1e-12, atol=1e-12)
    assert tok == int(np.argmax(want))


def test_q8_lm_head_planted_tie():
    """Rows 5 and 17 identical and dominant: the argmax is the lower id 5."""
    N, K = 24, 128
    q = np.zeros((N, K), np.uint8)
    q[5] = q[17] = 255
    m = _q8(q, np.full((N, 2), _bf16(1.0), np.uint16), np.zeros((N, 2), np.uint16))
    tok, lg = orc.q8_lm_head(m, np.full(K, _bf16(1.0), np.uint16))
    assert tok == 5 and lg[5] == lg[17] == 255.0 * K
