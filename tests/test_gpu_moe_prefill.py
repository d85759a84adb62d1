"""GPU parity of lily_q4_moe_prefill (tcgen05 grouped GEMM) against the oracle.

Top-k sets identical per token; y within the output tolerance.  At the full prompt-chunk
size (2048 tokens) every token's routing and every token's y are checked (the oracle runs the
tokens in parallel); at 4096 tokens y is checked on a sample."""
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


def run_prefill(torch, dev, dl, x_bits, ws=None):
    T = x_bits.shape[0]
    xd = q4.to_device(x_bits, dev)
    y = torch.empty_like(xd)
    idx = torch.full((T, dl.k), -1, dtype=torch.int32, device=dev)
    w = torch.empty((T, dl.k), dtype=torch.float32, device=dev)
    if ws is None:
        ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, T, prefill=True), dev)
    q4.lily_q4_moe_prefill(dl, xd, y, topk_idx=idx, topk_w=w, ws=ws)
    torch.cuda.synchronize()
    assert q4.lily_q4_workspace_status(ws) == 0, "a bounded device-side wait timed out"
    return bf16_bits_to_f64(y), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("H,E,k,I,shared,bias,T", [
    (128, 8, 2, 128, True, True, 37),
    (256, 16, 4, 256, True, False, 300),    # > 128 tokens per expert: several token tiles
    (512, 32, 8, 128, False, True, 129),
    (2048, 4, 2, 512, True, False, 1),      # a single token
    (256, 64, 6, 1024, True, True, 200),
    (256, 32, 8, 128, True, False, 8192),   # the largest chunk: selections not staged in bucketing
    (256, 1024, 16, 128, True, True, 100),  # most experts, largest k: one count-table group
    (256, 512, 4, 128, False, True, 2100),  # two groups of 72 top-k blocks (segments read in chunks)
])
def test_shapes(torch_dev, H, E, k, I, shared, bias, T):
    torch, dev = torch_dev
    key = (80, H + E + T)
    L = synth.draw_layer(H, E, k, I, shared=shared, router_std=0.05, router_bias=bias, key=key)
    x = _inputs(L, key, T)
    ref = orc.moe(L, x)
    dl = q4.DeviceLayer.upload(L, dev)
    y, idx, w = run_prefill(torch, dev, dl, x)
    what = f"H{H} E{E} k{k} I{I} T{T}"
    assert_topk_equal(idx, w, ref, what)
    assert_close(y, ref["y"], what)


def test_prefill_matches_decode_path(torch_dev):
    """The tensor-core path and the decode path agree on the same tokens."""
    torch, dev = torch_dev
    key = (81, 0)
    L = synth.draw_layer(512, 16, 4, 256, shared=True, router_std=0.05, router_bias=False, key=key)
    x = _inputs(L, key, 16)
    dl = q4.DeviceLayer.upload(L, dev)
    yp, ip, _ = run_prefill(torch, dev, dl, x)
    xd = q4.to_device(x, dev)
    yd = torch.empty_like(xd)
    ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, 16), dev)
    q4.lily_q4_moe_decode(dl, xd, yd, ws=ws)
    torch.cuda.synchronize()
    assert_close(yp, bf16_bits_to_f64(yd), "prefill vs decode")


def test_prefill_workload_full_size(torch_dev):
    """2048-token chunk through a 256-expert top-8 + shared layer with skewed router offsets:
    every token's routing and every token's output against the oracle."""
    torch, dev = torch_dev
    wl = synth.PREFILL
    L = wl.layer(0)
    T = wl.tokens[0]
    x = _inputs(L, wl.tokens_key(0), T)
    dl = q4.DeviceLayer.upload(L, dev)
    y, idx, w = run_prefill(torch, dev, dl, x)
    # load is skewed as intended (uneven tokens per expert)
    counts = np.bincount(idx.ravel(), minlength=L.E)
    assert counts.max() > 2 * counts.mean()
    ref = orc.moe(L, x)
    assert_topk_equal(idx, w, ref, "prefill 2048 tokens")
    assert_close(y, ref["y"], "prefill 2048 tokens, every token")


def test_prefill_4096_token_chunk_sampled(torch_dev):
    """The same layer with a 4096-token chunk (the larger chunk size the pages use): every
    token's routing, and y on a sample of tokens."""
    torch, dev = torch_dev
    wl = synth.PREFILL
    L = wl.layer(0)
    T = 4096
    x = _inputs(L, (wl.wid, 4096), T)
    dl = q4.DeviceLayer.upload(L, dev)
    y, idx, w = run_prefill(torch, dev, dl, x)
    lg = orc.router_tokens(L, x)
    for t in range(T):
        ref_idx, _ = orc.topk(lg[t], L.k)
        assert sorted(idx[t].tolist()) == sorted(ref_idx.tolist()), t
    rng = np.random.default_rng(1)
    sample = np.sort(rng.choice(T, 64, replace=False))
    ref = orc.moe(L, x[sample])
    assert_topk_equal(idx[sample], w[sample], ref, "prefill 4096 sample")
    assert_close(y[sample], ref["y"], "prefill 4096-token sample")


def test_deterministic(torch_dev):
    torch, dev = torch_dev
    key = (82, 0)
    L = synth.draw_layer(1024, 32, 4, 512, shared=True, router_std=0.05, router_bias=True, key=key)
    x = _inputs(L, key, 400)
    dl = q4.DeviceLayer.upload(L, dev)
    ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(dl, 400, prefill=True), dev)
    a = run_prefill(torch, dev, dl, x, ws)
    b = run_prefill(torch, dev, dl, x[:100], ws)
    c = run_prefill(torch, dev, dl, x, ws)
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])
    assert b[0].shape == (100, 1024)


def test_non_finite_logits_select_lowest_experts(torch_dev):
    """All logits -inf or NaN (NaN counts as -inf): every token still routes to real experts,
    the lowest ids, nothing is written out of bounds, and the call completes."""
    torch, dev = torch_dev
    key = (83, 0)
    L = synth.draw_layer(256, 16, 4, 128, shared=True, router_std=0.05, router_bias=True, key=key)
    L.router_bias = np.full(16, -np.inf, dtype=np.float32)
    L.router_bias[[3, 9]] = np.nan
    x = synth.draw_tokens(256, 40, key)
    dl = q4.DeviceLayer.upload(L, dev)
    _, idx, _ = run_prefill(torch, dev, dl, x)
    for t in range(40):
        assert sorted(idx[t].tolist()) == [0, 1, 2, 3]


# ----------------------------------------------------------------------------- 8-bit parts

@pytest.mark.parametrize("H,E,k,I,router_bits,shared_bits,T", [
    (256, 16, 4, 128, 8, 4, 300),     # 8-bit router: several token tiles per expert
    (256, 16, 2, 128, 16, 8, 129),    # 8-bit shared expert
    (512, 32, 8, 256, 8, 8, 77),
    (2048, 64, 4, 512, 8, 8, 200),    # the decode widths
    (128, 8, 2, 128, 8, 8, 1),        # a single token
])
def test_8bit_router_and_shared_expert(torch_dev, H, E, k, I, router_bits, shared_bits, T):
    """An affine 8-bit router (the checkpoint's router gates) and/or an 8-bit shared expert
    (q4-xl) through the tensor-core prefill path, against the oracle."""
    torch, dev = torch_dev
    key = (86, H + E + router_bits + shared_bits)
    L = synth.draw_layer(H, E, k, I, shared=True, router_std=0.05, router_bias=True, key=key,
                         router_bits=router_bits, shared_bits=shared_bits)
    x = _inputs(L, key, T)
    ref = orc.moe(L, x)
    dl = q4.DeviceLayer.upload(L, dev)
    y, idx, w = run_prefill(torch, dev, dl, x)
    what = f"8-bit parts r{router_bits} s{shared_bits} H{H} T{T}"
    assert_topk_equal(idx, w, ref, what)
    assert_close(y, ref["y"], what)


def test_prefill_q4xl_layout_full_size(torch_dev):
    """The prefill workload's layer in the q4-xl layout (8-bit router and shared expert, routed
    experts at 4 bits), 2048 tokens: every token's routing and output against the oracle."""
    torch, dev = torch_dev
    wl = synth.PREFILL
    key = (wl.wid, 500)
    L = synth.draw_layer(wl.H, wl.E, wl.k, wl.I, shared=True, router_std=wl.router_std,
                         router_bias=True, key=key, router_bits=8, shared_bits=8)
    T = wl.tokens[0]
    x = _inputs(L, key, T)
    dl = q4.DeviceLayer.upload(L, dev)
    assert q4.lily_q4_moe_launches(dl, T, prefill=True) == 12
    y, idx, w = run_prefill(torch, dev, dl, x)
    ref = orc.moe(L, x)
    assert_topk_equal(idx, w, ref, "q4-xl prefill 2048 tokens")
    assert_close(y, ref["y"], "q4-xl prefill 2048 tokens, every token")


def test_prefill_weights_16_byte_aligned(torch_dev):
    """The API promises 16-byte aligned code arrays.  When a gate/up code array is not 32-byte
    aligned, the gate/up GEMM takes each row's k-block with two threads (128-bit loads)
    instead of one (a 256-bit load): same values, so y is bit-identical to the aligned run,
    and within the tolerance of the oracle."""
    torch, dev = torch_dev
    H, E, k, I, T = 512, 8, 2, 256, 150
    key = (83, 0)
    L = synth.draw_layer(H, E, k, I, shared=True, router_std=0.05, router_bias=False, key=key)
    x = _inputs(L, key, T)
    dl = q4.DeviceLayer.upload(L, dev)
    ya, ia, _ = run_prefill(torch, dev, dl, x)

    def shifted(t):
        # the same words 16 bytes into a fresh buffer: 16-byte but not 32-byte aligned
        buf = torch.zeros(t.numel() + 4, dtype=t.dtype, device=dev)
        buf[4:].copy_(t.reshape(-1))
        view = buf[4:].view(t.shape)
        assert view.data_ptr() % 32 == 16
        return view, buf

    keep = []
    for m in (dl.gate, dl.up, dl.sh_gate, dl.sh_up):
        m.w, b = shifted(m.w)
        keep.append(b)
    dl._c = None
    yb, ib, _ = run_prefill(torch, dev, dl, x)
    assert (ia == ib).all()
    assert np.array_equal(ya, yb), "two-threads-per-row gate/up differs from the one-thread form"
    ref = orc.moe(L, x)
    assert_close(yb, ref["y"], "16-byte aligned weights")
