"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
its host-only format helpers agree with the oracle bit for bit, and argument errors
are reported before anything would be launched."""
import ctypes as C
import glob
import os
import re

import numpy as np
import pytest

import bit_affine_quantized_mlx_gb300 as q4
from bit_affine_quantized_mlx_gb300 import build as q4build
from oracle import oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    q4build.build()
    return q4.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        names |= set(re.findall(r"LILY_Q4_API\s+[\w\s\*]*?\b(lily_q4_\w+)\s*\(", txt))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"lily_q4_moe_decode", "lily_q4_moe_prefill", "lily_q4_gemv_argmax"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_pack_unpack_match_oracle(lib):
    rng = np.random.default_rng(0)
    q = rng.integers(0, 16, size=(9, 128), dtype=np.uint8)
    assert np.array_equal(q4.lily_q4_pack(q), orc.q4_pack(q))
    w = rng.integers(0, 2**32, size=(5, 32), dtype=np.uint32)
    assert np.array_equal(q4.lily_q4_unpack(w, 5, 256), orc.q4_unpack(w, 5, 256))
    # high bits of a code byte are ignored
    assert np.array_equal(q4.lily_q4_pack(q | 0xF0), orc.q4_pack(q))


def test_status_strings(lib):
    assert q4.status_string(0) == "ok"
    assert "workspace" in q4.status_string(-3)
    assert "timed out" in q4.status_string(-5)


# --------------------------------------------------------------------------- validation
# Fake, aligned, non-null "device" addresses: every case below must be rejected (or be a
# no-op) before any launch, so nothing dereferences them.
FAKE = 1 << 40


def _fake_layer(H=2048, E=256, k=8, I=512, shared=1):
    m = q4.lily_q4_mat(FAKE, FAKE + 4096, FAKE + 8192)
    L = q4.lily_q4_moe_layer()
    L.hidden, L.n_experts, L.top_k, L.inter = H, E, k, I
    L.gate = L.up = L.down = m
    L.has_shared = shared
    L.sh_gate = L.sh_up = L.sh_down = m
    L.router = FAKE + 65536
    L.router_bias = None
    L.shared_gate = FAKE + 131072 if shared else None
    return L


def _decode(lib, L, x=FAKE, T=1, y=FAKE + (1 << 20), ws=FAKE + (1 << 30), ws_bytes=1 << 30,
            fn="lily_q4_moe_decode"):
    return getattr(lib, fn)(C.byref(L) if L is not None else None, x, T, y, None, None, ws,
                            ws_bytes, None)


@pytest.mark.parametrize("fn", ["lily_q4_moe_decode", "lily_q4_moe_prefill"])
def test_moe_argument_errors(lib, fn):
    INV, UNS, WS = q4.ERR_INVALID_ARG, q4.ERR_UNSUPPORTED, q4.ERR_WORKSPACE_TOO_SMALL
    assert _decode(lib, None, fn=fn) == INV
    assert _decode(lib, _fake_layer(k=300, E=256), fn=fn) == INV          # k > 16 and > E
    assert _decode(lib, _fake_layer(k=9, E=8), fn=fn) == INV
    assert _decode(lib, _fake_layer(E=2000), fn=fn) == INV
    assert _decode(lib, _fake_layer(H=100), fn=fn) == INV                  # not a multiple of 64
    assert _decode(lib, _fake_layer(H=4096), fn=fn) == UNS                 # valid, not built
    assert _decode(lib, _fake_layer(I=192), fn=fn) == UNS
    L = _fake_layer()
    L.gate = q4.lily_q4_mat(FAKE + 4, FAKE, FAKE)                          # misaligned codes
    assert _decode(lib, L, fn=fn) == INV
    L = _fake_layer()
    L.shared_gate = None                                                    # shared without gate
    assert _decode(lib, L, fn=fn) == INV
    assert _decode(lib, _fake_layer(), x=None, fn=fn) == INV
    assert _decode(lib, _fake_layer(), x=FAKE + 2, fn=fn) == INV
    assert _decode(lib, _fake_layer(), ws=FAKE + 16, fn=fn) == INV          # ws not 256-aligned
    assert _decode(lib, _fake_layer(), ws_bytes=1024, fn=fn) == WS
    assert _decode(lib, _fake_layer(), T=-1, fn=fn) == INV
    assert _decode(lib, _fake_layer(), T=0, fn=fn) == q4.OK                # empty: nothing enqueued
    too_many = 17 if fn == "lily_q4_moe_decode" else 8193
    assert _decode(lib, _fake_layer(), T=too_many, fn=fn) == INV


def test_8bit_layer_argument_errors(lib):
    INV = q4.ERR_INVALID_ARG
    L = _fake_layer()
    L.shared_bits = 5                                                      # no such width
    assert _decode(lib, L) == INV
    L = _fake_layer()
    L.router_bits = 12
    assert _decode(lib, L) == INV
    L = _fake_layer()
    L.router_bits = 8                                                      # 8-bit router without its matrix
    assert _decode(lib, L) == INV
    L.router_q8 = q4.lily_q4_mat(FAKE, FAKE + 4096, FAKE + 8192)
    L.router = None                                                        # the bf16 router is then unused
    assert _decode(lib, L, T=0) == q4.OK
    # prefill takes it: 7 launches plus two that prepare the 8-bit router's exact bf16 form
    assert lib.lily_q4_moe_launches(C.byref(L), 4, 1) == 9
    assert lib.lily_q4_moe_prefill(C.byref(L), None, 1, None, None, None, None, 0, None) == q4.ERR_INVALID_ARG


def test_gemv_argument_errors(lib):
    m = q4.lily_q4_mat(FAKE, FAKE + 4096, FAKE + 8192)
    f = lib.lily_q4_gemv_argmax
    ws = FAKE + (1 << 30)
    assert f(None, 10, 2048, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 0, 2048, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 100, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 4096, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_UNSUPPORTED
    assert f(C.byref(m), 10, 2048, FAKE, None, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 2048, FAKE, FAKE + 2, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 2048, FAKE, FAKE, None, ws, 16, None) == q4.ERR_WORKSPACE_TOO_SMALL


def test_gemv_logprobs_argument_errors(lib):
    m = q4.lily_q4_mat(FAKE, FAKE + 4096, FAKE + 8192)
    f = lib.lily_q4_gemv_argmax_logprobs
    ws, big = FAKE + (1 << 30), 1 << 20
    lse, lp = FAKE + 512, FAKE + (1 << 24)
    INV = q4.ERR_INVALID_ARG
    assert f(None, 10, 2048, FAKE, FAKE, lse, lp, ws, big, None) == INV
    assert f(C.byref(m), 10, 2048, FAKE, FAKE, None, lp, ws, big, None) == INV      # lse required
    assert f(C.byref(m), 10, 2048, FAKE, FAKE, lse + 2, lp, ws, big, None) == INV   # misaligned
    assert f(C.byref(m), 10, 2048, FAKE, FAKE, lse, lp + 2, ws, big, None) == INV
    assert f(C.byref(m), 10, 2048, FAKE, None, lse, lp, ws, big, None) == INV
    assert f(C.byref(m), 10, 4096, FAKE, FAKE, lse, lp, ws, big, None) == q4.ERR_UNSUPPORTED
    # the logprobs call needs the per-block log-sum-exp partials on top of the argmax pairs
    n = lib.lily_q4_gemv_argmax_workspace_bytes(151936, 2048)
    assert f(C.byref(m), 151936, 2048, FAKE, FAKE, lse, None, ws, n - 256, None) == \
        q4.ERR_WORKSPACE_TOO_SMALL


def test_q8_gemv_argument_errors(lib):
    m = q4.lily_q4_mat(FAKE, FAKE + 4096, FAKE + 8192)
    f = lib.lily_q8_gemv_argmax
    ws = FAKE + (1 << 30)
    assert f(None, 10, 2048, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 100, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 256, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_UNSUPPORTED
    assert f(C.byref(m), 10, 4096, FAKE, FAKE, None, ws, 1 << 20, None) == q4.ERR_UNSUPPORTED
    assert f(C.byref(m), 10, 2048, FAKE, None, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert f(C.byref(m), 10, 2048, FAKE, FAKE, None, ws, 16, None) == q4.ERR_WORKSPACE_TOO_SMALL
    assert lib.lily_q8_gemv_argmax_workspace_bytes(151936, 2048) > 0
    assert lib.lily_q8_gemv_argmax_workspace_bytes(10, 100) == 0
    g = lib.lily_q8_gemv_argmax_logprobs
    lse = FAKE + 512
    assert g(C.byref(m), 10, 2048, FAKE, FAKE, None, None, ws, 1 << 20, None) == q4.ERR_INVALID_ARG
    assert g(C.byref(m), 10, 256, FAKE, FAKE, lse, None, ws, 1 << 20, None) == q4.ERR_UNSUPPORTED
    n = lib.lily_q8_gemv_argmax_workspace_bytes(151936, 2048)
    assert g(C.byref(m), 151936, 2048, FAKE, FAKE, lse, None, ws, n - 256, None) == \
        q4.ERR_WORKSPACE_TOO_SMALL


def test_selftest_argument_errors(lib):
    f = lib.lily_q4_selftest_timeout
    assert f(None, 1024, 0, None) == q4.ERR_INVALID_ARG
    assert f(FAKE + 16, 1024, 0, None) == q4.ERR_INVALID_ARG     # not 256-aligned
    assert f(FAKE, 64, 0, None) == q4.ERR_INVALID_ARG            # smaller than the header
    assert f(FAKE, 1024, 2, None) == q4.ERR_INVALID_ARG          # no such wait
    assert f(None, 0, 2, None) == q4.ERR_INVALID_ARG             # no such wait (fixed scratch)


def test_workspace_sizes(lib):
    L = _fake_layer()
    d1 = lib.lily_q4_moe_workspace_bytes(C.byref(L), 1, 0)
    d4 = lib.lily_q4_moe_workspace_bytes(C.byref(L), 4, 0)
    assert 0 < d1 < d4
    assert lib.lily_q4_moe_workspace_bytes(C.byref(L), 17, 0) == 0
    assert lib.lily_q4_moe_workspace_bytes(C.byref(L), 2048, 1) > 0
    assert lib.lily_q4_moe_workspace_bytes(None, 1, 0) == 0
    assert lib.lily_q4_gemv_argmax_workspace_bytes(151936, 2048) > 0
    assert lib.lily_q4_gemv_argmax_workspace_bytes(10, 100) == 0
    assert lib.lily_q4_workspace_init(None, 1024, None) == q4.ERR_INVALID_ARG
