"""GPU parity of lily_q4_gemv_argmax (Q4 LM-head GEMV + greedy argmax) against the oracle.

Token ids must be identical; logits within the output tolerance (see helpers.py)."""
import numpy as np
import pytest

import bit_affine_quantized_mlx_gb300 as q4
from bit_affine_quantized_mlx_gb300 import synth
from bit_affine_quantized_mlx_gb300.synth import Q4Matrix
from helpers import assert_close
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    return torch, torch.device("cuda:0")


def _run(torch, dev, W, x_bits, with_logits=True):
    N, K = W.N, W.K
    dW = q4.DeviceQ4.upload(W, dev)
    xd = q4.to_device(x_bits, dev)
    tok = torch.full((1,), -7, dtype=torch.int32, device=dev)
    lg = torch.empty(N, dtype=torch.float32, device=dev) if with_logits else None
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(N, K), dev)
    q4.lily_q4_gemv_argmax(dW, xd, tok, logits=lg, ws=ws)
    torch.cuda.synchronize()
    assert q4.lily_q4_workspace_status(ws) == q4.OK, "a bounded device-side wait timed out"
    return int(tok.item()), (lg.cpu().numpy().astype(np.float64) if with_logits else None)


@pytest.mark.parametrize("N,K", [(1, 64), (37, 128), (1000, 256), (4097, 512), (333, 1024),
                                 (50001, 2048),
                                 (7297, 2048)])  # the last blocks' row ranges are empty
def test_shapes(torch_dev, N, K):
    torch, dev = torch_dev
    W = synth.draw_q4(N, K, 60, N, K)
    if N == 1:
        x = synth.draw_x(K, (60, N), 0, 0)
        tok, lg = orc.lm_head(W, x)
    else:
        x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_x(K, (60, N), 0, a))
    got_tok, got_lg = _run(torch, dev, W, x)
    assert got_tok == tok
    assert_close(got_lg, lg, f"logits N={N} K={K}")


def test_full_size_lm_head(torch_dev):
    """The LM-head workload at its full size (vocab 151,936 x hidden 2048), every logit checked."""
    torch, dev = torch_dev
    wl = synth.LMHEAD
    W = synth.draw_lm_head(wl.V, wl.H)
    x, attempt, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_lm_x(wl.H, attempt=a))
    got_tok, got_lg = _run(torch, dev, W, x)
    assert got_tok == tok
    assert_close(got_lg, lg, "full LM head")
    # without the logits output, same token
    got_tok2, _ = _run(torch, dev, W, x, with_logits=False)
    assert got_tok2 == tok


def test_planted_tie_goes_to_lower_index(torch_dev):
    torch, dev = torch_dev
    N, K = 3000, 512
    W = synth.draw_q4(N, K, 61, 0)
    w, s, b = W.w.copy(), W.s.copy(), W.b.copy()
    # rows 1234 and 2345 identical and dominant: all codes 15, scale +, bias 0
    for r in (2345, 1234):
        w[r] = 0xFFFFFFFF
        s[r] = synth.bf16_from_f32(np.float32(0.05))
        b[r] = 0
    x = np.full(K, synth.bf16_from_f32(np.float32(0.5)).item(), np.uint16)
    W2 = Q4Matrix(w, s, b)
    tok, lg = orc.lm_head(W2, x)
    assert tok == 1234 and lg[1234] == lg[2345]
    got_tok, got_lg = _run(torch, dev, W2, x)
    assert got_tok == 1234
    assert got_lg[1234] == got_lg[2345]


def test_deterministic(torch_dev):
    torch, dev = torch_dev
    W = synth.draw_q4(20000, 2048, 62, 0)
    x = synth.draw_x(2048, (62, 0), 0, 0)
    a = _run(torch, dev, W, x)
    b = _run(torch, dev, W, x)
    assert a[0] == b[0] and np.array_equal(a[1], b[1])


def test_all_nan_logits_give_a_real_token(torch_dev):
    """NaN scales make every logit NaN: the token is still a real id (0, as ties and NaN
    candidates resolve to the lowest id) and nothing faults."""
    torch, dev = torch_dev
    N, K = 3000, 256
    W = synth.draw_q4(N, K, 63, 0)
    W = Q4Matrix(W.w, np.full_like(W.s, 0x7FC0), W.b)   # bf16 NaN scales
    x = synth.draw_x(K, (63, 0), 0, 0)
    got_tok, _ = _run(torch, dev, W, x)
    assert got_tok == 0


# ----------------------------------------------------------------------------- logprobs

def _run_lp(torch, dev, W, x_bits, with_lp=True):
    N, K = W.N, W.K
    dW = q4.DeviceQ4.upload(W, dev)
    xd = q4.to_device(x_bits, dev)
    tok = torch.full((1,), -7, dtype=torch.int32, device=dev)
    lse = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    lp = torch.empty(N, dtype=torch.float32, device=dev) if with_lp else None
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(N, K), dev)
    q4.lily_q4_gemv_argmax_logprobs(dW, xd, tok, lse, logprobs=lp, ws=ws)
    torch.cuda.synchronize()
    return (int(tok.item()), float(lse.item()),
            lp.cpu().numpy().astype(np.float64) if with_lp else None)


def _check_lp(got, tok, lg, what):
    """Token identical; logprobs within the output tolerance; lse within the largest logit
    error (log-sum-exp moves by at most the largest change of any logit) plus 1e-4 for the
    fp32 sum of exponentials; the returned logprobs normalise."""
    got_tok, got_lse, got_lp = got
    lse, lp = orc.log_softmax(lg)
    assert got_tok == tok, what
    assert_close(got_lp, lp, f"logprobs {what}")
    logit_err = np.abs((got_lp + got_lse) - lg).max()
    assert abs(got_lse - lse) <= logit_err + 1e-4 + 1e-6 * abs(lse), (what, got_lse, lse)
    import scipy.special as sp
    assert abs(float(sp.logsumexp(got_lp))) <= 1e-4, what


@pytest.mark.parametrize("N,K", [(1, 64), (37, 128), (1000, 256), (4097, 512), (7297, 2048)])
def test_logprobs_shapes(torch_dev, N, K):
    torch, dev = torch_dev
    W = synth.draw_q4(N, K, 64, N, K)
    if N == 1:
        x = synth.draw_x(K, (64, N), 0, 0)
        tok, lg = orc.lm_head(W, x)
    else:
        x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_x(K, (64, N), 0, a))
    got = _run_lp(torch, dev, W, x)
    _check_lp(got, tok, lg, f"N={N} K={K}")
    if N == 1:
        assert got[2][0] == 0.0  # one row: lse is the logit itself
    # lse alone (no vector): same token and the same lse bits
    t2, lse2, _ = _run_lp(torch, dev, W, x, with_lp=False)
    assert t2 == got[0] and lse2 == got[1]


def test_logprobs_full_size(torch_dev):
    """Vocabulary 151,936 x hidden 2048: every log-probability checked against the oracle,
    and two calls give identical bits."""
    torch, dev = torch_dev
    wl = synth.LMHEAD
    W = synth.draw_lm_head(wl.V, wl.H)
    x, attempt, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_lm_x(wl.H, attempt=a))
    a = _run_lp(torch, dev, W, x)
    _check_lp(a, tok, lg, "full LM head")
    b = _run_lp(torch, dev, W, x)
    assert a[0] == b[0] and a[1] == b[1] and np.array_equal(a[2], b[2])
    # the argmax-only call on the same inputs picks the same token
    assert _run(torch, dev, W, x, with_logits=False)[0] == tok


# ----------------------------------------------------------------------------- 8-bit LM head

def _run_q8(torch, dev, W, x_bits, with_logits=True):
    N, K = W.N, W.K
    dW = q4.DeviceQ4.upload(W, dev)
    xd = q4.to_device(x_bits, dev)
    tok = torch.full((1,), -7, dtype=torch.int32, device=dev)
    lg = torch.empty(N, dtype=torch.float32, device=dev) if with_logits else None
    ws = q4.new_workspace(q4.lily_q8_gemv_argmax_workspace_bytes(N, K), dev)
    q4.lily_q8_gemv_argmax(dW, xd, tok, logits=lg, ws=ws)
    torch.cuda.synchronize()
    return int(tok.item()), (lg.cpu().numpy().astype(np.float64) if with_logits else None)


@pytest.mark.parametrize("N,K", [(1, 512), (37, 1024), (4097, 512), (333, 2048), (7297, 2048),
                                 (50001, 2048)])
def test_q8_shapes(torch_dev, N, K):
    torch, dev = torch_dev
    W = synth.draw_q8(N, K, 65, N, K)
    if N == 1:
        x = synth.draw_x(K, (65, N), 0, 0)
        tok, lg = orc.q8_lm_head(W, x)
    else:
        x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_x(K, (65, N), 0, a),
                                                  head=orc.q8_lm_head)
    got_tok, got_lg = _run_q8(torch, dev, W, x)
    assert got_tok == tok
    assert_close(got_lg, lg, f"8-bit logits N={N} K={K}")


def test_q8_full_size_lm_head(torch_dev):
    """An 8-bit LM head of vocabulary 151,936 x hidden 2048 (the q4-xl conversion's), every
    logit checked; the token also without the logits output; two calls identical."""
    torch, dev = torch_dev
    wl = synth.LMHEAD
    W = synth.draw_lm_head_q8(wl.V, wl.H)
    x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_lm_x(wl.H, attempt=a),
                                              head=orc.q8_lm_head)
    a = _run_q8(torch, dev, W, x)
    assert a[0] == tok
    assert_close(a[1], lg, "full 8-bit LM head")
    assert _run_q8(torch, dev, W, x, with_logits=False)[0] == tok
    b = _run_q8(torch, dev, W, x)
    assert np.array_equal(a[1], b[1])


def test_q8_planted_tie_goes_to_lower_index(torch_dev):
    torch, dev = torch_dev
    N, K = 3000, 512
    W = synth.draw_q8(N, K, 66, 0)
    w, s, b = W.w.copy(), W.s.copy(), W.b.copy()
    for r in (2345, 1234):
        w[r] = 0xFFFFFFFF
        s[r] = synth.bf16_from_f32(np.float32(0.003))
        b[r] = 0
    x = np.full(K, synth.bf16_from_f32(np.float32(0.5)).item(), np.uint16)
    W2 = synth.Q8Matrix(w, s, b)
    tok, lg = orc.q8_lm_head(W2, x)
    assert tok == 1234 and lg[1234] == lg[2345]
    got_tok, got_lg = _run_q8(torch, dev, W2, x)
    assert got_tok == 1234 and got_lg[1234] == got_lg[2345]


def _run_q8_lp(torch, dev, W, x_bits, with_lp=True):
    N, K = W.N, W.K
    dW = q4.DeviceQ4.upload(W, dev)
    xd = q4.to_device(x_bits, dev)
    tok = torch.full((1,), -7, dtype=torch.int32, device=dev)
    lse = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    lp = torch.empty(N, dtype=torch.float32, device=dev) if with_lp else None
    ws = q4.new_workspace(q4.lily_q8_gemv_argmax_workspace_bytes(N, K), dev)
    q4.lily_q8_gemv_argmax_logprobs(dW, xd, tok, lse, logprobs=lp, ws=ws)
    torch.cuda.synchronize()
    return (int(tok.item()), float(lse.item()),
            lp.cpu().numpy().astype(np.float64) if with_lp else None)


@pytest.mark.parametrize("N,K", [(37, 1024), (4097, 512), (7297, 2048)])
def test_q8_logprobs_shapes(torch_dev, N, K):
    torch, dev = torch_dev
    W = synth.draw_q8(N, K, 67, N, K)
    x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_x(K, (67, N), 0, a),
                                              head=orc.q8_lm_head)
    got = _run_q8_lp(torch, dev, W, x)
    _check_lp(got, tok, lg, f"8-bit N={N} K={K}")
    t2, lse2, _ = _run_q8_lp(torch, dev, W, x, with_lp=False)
    assert t2 == got[0] and lse2 == got[1]


def test_q8_logprobs_full_size(torch_dev):
    """The 8-bit LM head (151,936 x 2048) with the log-sum-exp and every log-probability."""
    torch, dev = torch_dev
    wl = synth.LMHEAD
    W = synth.draw_lm_head_q8(wl.V, wl.H)
    x, _, tok, lg = orc.lm_x_without_near_tie(W, lambda a: synth.draw_lm_x(wl.H, attempt=a),
                                              head=orc.q8_lm_head)
    a = _run_q8_lp(torch, dev, W, x)
    _check_lp(a, tok, lg, "full 8-bit LM head")
    b = _run_q8_lp(torch, dev, W, x)
    assert a[0] == b[0] and a[1] == b[1] and np.array_equal(a[2], b[2])


def test_back_to_back_calls_share_a_workspace(torch_dev):
    """Calls enqueued back to back on one stream with one workspace (each a programmatic
    dependent of the previous one, its weight copies starting while that one drains) alternate
    two heads; every token matches the oracle, so the packed grid maximum and the block counter
    are re-armed by each call before the next one folds into them."""
    torch, dev = torch_dev
    N, K = 50001, 2048
    heads = [synth.draw_q4(N, K, 61, h, 0) for h in range(2)]
    xs, wants = [], []
    for c in range(4):
        for attempt in range(20):  # a token row whose top-2 logits are not a near tie
            x = synth.draw_x(K, (61, c), 0, attempt)
            tok, lg = orc.lm_head(heads[c % 2], x)
            top2 = np.sort(lg)[-2:]
            if top2[1] - top2[0] >= 1e-3:
                break
        xs.append(x)
        wants.append(tok)
    dWs = [q4.DeviceQ4.upload(W, dev) for W in heads]
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(N, K), dev)
    toks = [torch.full((1,), -7, dtype=torch.int32, device=dev) for _ in xs]
    xds = [q4.to_device(x, dev) for x in xs]
    st = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(st):
        for c in range(len(xs)):
            q4.lily_q4_gemv_argmax(dWs[c % 2], xds[c], toks[c], ws=ws, stream=st)
    st.synchronize()
    assert q4.lily_q4_workspace_status(ws, st) == q4.OK
    for c in range(len(xs)):
        assert int(toks[c].item()) == wants[c], f"call {c}"
