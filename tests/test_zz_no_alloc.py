"""The allocation-free LM-head entry point (lily_q4_gemv_argmax_noalloc).

Callers that cannot call cudaMalloc -- code on a memory budget fixed at start-up, or a
host framework that owns every device allocation and hands this library only input and
output pointers -- use this entry point; its scratch is a fixed array inside the library.
Checked through the C ABI against lily_q4_gemv_argmax (which takes a workspace) on two
calls in a row, so that contents left in the shared scratch by one call cannot leak into
the next.  Kept in a file collected last."""
import numpy as np
import pytest

import bit_affine_quantized_mlx_gb300 as q4
from bit_affine_quantized_mlx_gb300 import synth
from helpers import assert_close

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    N, K = 30000, 2048
    W = q4.DeviceQ4.upload(synth.draw_q4(N, K, 95, 0), dev)
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(N, K), dev)
    for call in range(2):
        x = q4.to_device(synth.draw_x(K, (95, 0), call, 0), dev)
        tok_ref = torch.full((1,), -1, dtype=torch.int32, device=dev)
        lg_ref = torch.empty(N, dtype=torch.float32, device=dev)
        q4.lily_q4_gemv_argmax(W, x, tok_ref, logits=lg_ref, ws=ws)
        tok = torch.full((1,), -1, dtype=torch.int32, device=dev)
        lg = torch.empty(N, dtype=torch.float32, device=dev)
        q4.lily_q4_gemv_argmax_noalloc(W, x, tok, logits=lg)
        torch.cuda.synchronize()
        assert int(tok.item()) == int(tok_ref.item()), f"call {call}"
        assert_close(lg.cpu().numpy().astype(np.float64),
                     lg_ref.cpu().numpy().astype(np.float64), f"logits, call {call}")


@pytest.mark.parametrize("which", [0, 1])
def test_noalloc_status_reports_a_timed_out_wait(which):
    """A bounded wait that gives up inside the fixed scratch (the diagnostic kernel of
    lily_q4_selftest_timeout, pointed at that scratch: 0 a grid barrier, 1 an mbarrier) is
    reported by lily_q4_gemv_argmax_noalloc_status, even after a later call of the entry point
    (which resets only the counters); the read clears it, and that later call is still right."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    N, K = 4096, 2048
    W = q4.DeviceQ4.upload(synth.draw_q4(N, K, 96, which), dev)
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(N, K), dev)
    x = q4.to_device(synth.draw_x(K, (96, which), 0, 0), dev)
    tok = torch.full((1,), -1, dtype=torch.int32, device=dev)
    q4.lily_q4_gemv_argmax_noalloc(W, x, tok)
    assert q4.lily_q4_gemv_argmax_noalloc_status() == q4.OK
    q4.lily_q4_selftest_timeout(None, which)
    tok_ref = torch.full((1,), -1, dtype=torch.int32, device=dev)
    q4.lily_q4_gemv_argmax(W, x, tok_ref, ws=ws)
    tok.fill_(-1)
    q4.lily_q4_gemv_argmax_noalloc(W, x, tok)
    assert q4.lily_q4_gemv_argmax_noalloc_status() == q4.ERR_TIMEOUT
    assert q4.lily_q4_gemv_argmax_noalloc_status() == q4.OK    # cleared on read
    assert int(tok.item()) == int(tok_ref.item())
    assert q4.lily_q4_workspace_status(ws) == q4.OK            # the workspace call is untouched
