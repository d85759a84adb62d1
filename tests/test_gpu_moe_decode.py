"""GPU parity of lily_q4_moe_decode against the oracle.

Top-k expert sets must be identical per token (weights per expert within 1e-5); y within
the output tolerance.  Inputs are redrawn per token until the oracle's k-th and (k+1)-th
router logits differ by at least 1e-3."""
import numpy as np
import pytest

import bit_affine_quantized_mlx_gb300 as q4
from bit_affine_quantized_mlx_gb300 import synth
from helpers import assert_close, assert_topk_equal, bf16_bits_to_f64
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    return torch, torch.device("cuda:0")


def _inputs(L, key, T):
    return orc.tokens_without_near_ties(L, lambda t, a: synth.draw_x(L.H, key, t, a), T)[0]


def run_decode(torch, dev, dl, x_bits, ws=None):
    T = x_bits.shape[0]
    xd = q4.to_device(x_bits, dev)
    y = torch.empty_like(xd)
    idx = torch.full((T, dl.k), -1, dtype=torch.int32, device=dev)
    w = torch.empty((T, dl.k), dtype=torch.float32, device=dev)
    if ws is None:
        ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, T), dev)
    q4.lily_q4_moe_decode(dl, xd, y, topk_idx=idx, topk_w=w, ws=ws)
    torch.cuda.synchronize()
    assert q4.lily_q4_workspace_status(ws) == q4.OK, "a bounded device-side wait timed out"
    return bf16_bits_to_f64(y), idx.cpu().numpy(), w.cpu().numpy()


def check(torch, dev, L, x, what, ws=None, dl=None):
    ref = orc.moe(L, x)
    dl = dl or q4.DeviceLayer.upload(L, dev)
    y, idx, w = run_decode(torch, dev, dl, x, ws)
    assert_topk_equal(idx, w, ref, what)
    assert_close(y, ref["y"], what)
    return y


def test_tiny_workload_seed0(torch_dev):
    """The tiny layer (hidden 256, 16 experts, top-2, intermediate 128, no shared), seed 0."""
    torch, dev = torch_dev
    wl = synth.TINY
    L = wl.layer(0)
    check(torch, dev, L, _inputs(L, wl.tokens_key(0), 1), "tiny")


@pytest.mark.parametrize("H,E,k,I,shared,bias,T", [
    (64, 4, 2, 64, False, False, 1),
    (128, 8, 8, 64, True, True, 3),      # k == E: every expert
    (256, 16, 2, 128, False, False, 16),  # largest batch
    (512, 32, 4, 256, True, False, 5),
    (1024, 64, 16, 128, True, True, 2),   # largest k
    (2048, 40, 3, 2048, True, False, 2),  # widest intermediate
    (256, 1024, 5, 128, True, False, 3),  # most experts
    # hidden 2048 / intermediate 512: the single-launch path (batch <= 4)
    (2048, 64, 16, 512, True, True, 4),   # top-16 of 64, 4 tokens: beyond the staged down tasks
    (2048, 8, 2, 512, False, False, 3),   # one router row per CTA, no shared expert
    (2048, 24, 3, 512, True, False, 2),   # a partial router chunk
    (2048, 256, 8, 512, True, False, 16),  # decode shapes at the largest batch (three launches)
])
def test_shapes(torch_dev, H, E, k, I, shared, bias, T):
    torch, dev = torch_dev
    key = (70, H * 7 + E + T)
    L = synth.draw_layer(H, E, k, I, shared=shared, router_std=0.05, router_bias=bias, key=key)
    check(torch, dev, L, _inputs(L, key, T), f"H{H} E{E} k{k} I{I} T{T}")


@pytest.mark.parametrize("layer,T", [(0, 1), (0, 4), (39, 1), (39, 4)])
def test_decode_workload_full_size(torch_dev, layer, T):
    """Decode layer at hidden 2048, 256 experts, top-8 + shared, intermediate 512."""
    torch, dev = torch_dev
    wl = synth.DECODE
    L = wl.layer(layer)
    check(torch, dev, L, _inputs(L, wl.tokens_key(layer), T), f"decode layer {layer} T{T}")


@pytest.mark.parametrize("T", [1, 2, 4])
def test_wide_workload_full_size(torch_dev, T):
    """Wide layer at hidden 2048, 512 experts, top-10 + shared, intermediate 512."""
    torch, dev = torch_dev
    wl = synth.WIDE
    L = wl.layer(47)
    check(torch, dev, L, _inputs(L, wl.tokens_key(47), T), f"wide T{T}")


def test_repeated_tokens_share_experts(torch_dev):
    """Identical tokens choose identical experts: each expert serves several tokens."""
    torch, dev = torch_dev
    key = (71, 0)
    L = synth.draw_layer(512, 16, 4, 256, shared=True, router_std=0.05, router_bias=False, key=key)
    x1 = _inputs(L, key, 1)
    x = np.repeat(x1, 6, axis=0)
    y = check(torch, dev, L, x, "repeated")
    assert np.all(y == y[0])


def test_deterministic_and_workspace_reuse(torch_dev):
    torch, dev = torch_dev
    wl = synth.DECODE
    L = wl.layer(1)
    dl = q4.DeviceLayer.upload(L, dev)
    x4 = _inputs(L, wl.tokens_key(1), 4)
    ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, 4), dev)
    a = run_decode(torch, dev, dl, x4, ws)
    b = run_decode(torch, dev, dl, x4[:1], ws)   # smaller T in the same workspace
    c = run_decode(torch, dev, dl, x4, ws)
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])
    assert np.array_equal(a[0][0], b[0][0])


@pytest.mark.parametrize("H,I,T", [(256, 128, 1), (256, 128, 3), (256, 128, 6), (2048, 512, 3)])
def test_non_finite_logits_select_lowest_experts(torch_dev, H, I, T):
    """Router offsets of -inf (and NaN, which counts as -inf) make every logit non-finite: the
    selection still names real experts -- the lowest ids, as the (value desc, index asc) order
    gives for equal logits -- and the call completes."""
    torch, dev = torch_dev
    key = (72, T)
    L = synth.draw_layer(H, 16, 4, I, shared=True, router_std=0.05, router_bias=True, key=key)
    L.router_bias = np.full(16, -np.inf, dtype=np.float32)
    L.router_bias[[3, 9]] = np.nan
    x = synth.draw_tokens(H, T, key)
    dl = q4.DeviceLayer.upload(L, dev)
    _, idx, _ = run_decode(torch, dev, dl, x)
    for t in range(T):
        assert sorted(idx[t].tolist()) == [0, 1, 2, 3]


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_reports_timeout_and_context_stays_usable(torch_dev, which):
    """A wait that nothing completes (0: the decode kernel's grid barrier, 1: an mbarrier as in
    the prefill GEMM and LM head) gives up at its bound and is reported as a time-out through
    the workspace; after re-initialising the workspace the same context decodes correctly."""
    torch, dev = torch_dev
    wl = synth.TINY
    L = wl.layer(0)
    dl = q4.DeviceLayer.upload(L, dev)
    x = _inputs(L, wl.tokens_key(0), 1)
    ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, 1), dev)
    q4.lily_q4_selftest_timeout(ws, which)
    assert q4.lily_q4_workspace_status(ws) == q4.ERR_TIMEOUT
    assert q4.lily_q4_workspace_status(ws) == q4.OK   # the status word is cleared on read
    q4.lily_q4_workspace_init(ws)
    check(torch, dev, L, x, f"decode after a time-out ({which})", ws=ws, dl=dl)
    assert q4.lily_q4_workspace_status(ws) == q4.OK


# ----------------------------------------------------------------------------- 8-bit parts

@pytest.mark.parametrize("H,E,k,I,router_bits,shared_bits,T", [
    (256, 16, 2, 128, 8, 4, 1),
    (256, 16, 4, 128, 16, 8, 3),
    (256, 32, 4, 128, 8, 8, 4),
    (2048, 256, 8, 512, 8, 8, 1),   # the decode shapes with the q4-xl shared expert and 8-bit router
    (2048, 256, 8, 512, 8, 8, 4),
    (2048, 256, 8, 512, 16, 8, 2),
    # above four tokens: the three-launch path
    (256, 16, 2, 128, 8, 4, 5),
    (256, 32, 4, 128, 16, 8, 9),
    (2048, 256, 8, 512, 8, 8, 16),
    (1024, 64, 6, 256, 8, 8, 7),
])
def test_8bit_router_and_shared_expert(torch_dev, H, E, k, I, router_bits, shared_bits, T):
    """An affine 8-bit router (the checkpoint's router gates) and/or an 8-bit shared expert
    (q4-xl) in the decode paths (one launch up to four tokens, three or four above), against
    the oracle."""
    torch, dev = torch_dev
    key = (84, H + E + router_bits + shared_bits)
    L = synth.draw_layer(H, E, k, I, shared=True, router_std=0.05, router_bias=True, key=key,
                         router_bits=router_bits, shared_bits=shared_bits)
    check(torch, dev, L, _inputs(L, key, T), f"8-bit parts r{router_bits} s{shared_bits} T{T}")


def test_8bit_parts_launch_counts(torch_dev):
    """Launch counts of a layer with 8-bit parts: decode one launch up to four tokens, four
    above (the 8-bit shared expert's gate/up runs as its own launch); prefill 7 plus two
    preparation launches for an 8-bit router and three for an 8-bit shared expert."""
    torch, dev = torch_dev
    L = synth.draw_layer(256, 16, 2, 128, shared=True, router_std=0.05, router_bias=False,
                         key=(85, 0), router_bits=8, shared_bits=8)
    dl = q4.DeviceLayer.upload(L, dev)
    assert q4.lily_q4_moe_launches(dl, 4) == 1 and q4.lily_q4_moe_launches(dl, 5) == 4
    assert q4.lily_q4_moe_launches(dl, 64, prefill=True) == 12
    Lr = synth.draw_layer(256, 16, 2, 128, shared=True, router_std=0.05, router_bias=False,
                          key=(85, 1), router_bits=8, shared_bits=4)
    assert q4.lily_q4_moe_launches(q4.DeviceLayer.upload(Lr, dev), 64, prefill=True) == 9
