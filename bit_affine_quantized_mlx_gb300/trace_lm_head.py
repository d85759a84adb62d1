"""Timeline of the streaming LM-head kernel (greedy token of a 151,936 x 2048 Q4 head).

Builds the profiling variant of the library (``build(trace=True)``), runs
``lily_q4_gemv_argmax`` back to back on one stream (a ~1 ms spin kernel first, so the host is
ahead of the GPU; events around each call, as the bench times it; each repetition makes two
calls), and prints for the second call when the blocks reached each point, in us after its
first block was set up:

  setup    mbarriers initialised (block start)
  x        x prepared by the compute warps
  stage0   the first stage of weights landed in shared memory
  copies   the copy thread issued its last stage
  stages   the last stage computed
  fold     the block's argmax about to be folded into the grid maximum
  done     the block finished (the last one also wrote the token)

with the median, earliest and latest block, and the event-timed durations of both calls.
The timestamps are %globaltimer reads, so the figures profile the kernel as it runs.

    python -m bit_affine_quantized_mlx_gb300.trace_lm_head [--reps 20]
"""
from __future__ import annotations

import argparse
import ctypes as C
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

POINTS = [(0, "setup"), (1, "x"), (2, "stage0"), (6, "copies"), (3, "stages"), (4, "fold"),
          (5, "done")]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--reps", type=int, default=20)
    args = ap.parse_args(argv)

    from bit_affine_quantized_mlx_gb300 import build as _build
    lib_path = _build.build(trace=True)
    import torch
    import bit_affine_quantized_mlx_gb300 as q4
    from bit_affine_quantized_mlx_gb300 import synth
    L = q4.load(lib_path)
    L.lily_q4_lm_trace_read.argtypes = [C.c_void_p, C.c_size_t]
    L.lily_q4_lm_trace_read.restype = C.c_int

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    st = torch.cuda.Stream(device=dev)
    lmw = synth.LMHEAD
    W = q4.DeviceQ4.upload(synth.draw_lm_head(lmw.V, lmw.H), dev)
    x = q4.to_device(synth.draw_lm_x(lmw.H), dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    ws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(lmw.V, lmw.H), dev)
    G = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = np.zeros(1024 * 8, dtype=np.uint64)
    rel = {name: [] for _, name in POINTS}
    ev_us = []
    with torch.cuda.stream(st):
        for _ in range(3):
            q4.lily_q4_gemv_argmax(W, x, tok, ws=ws, stream=st)
    st.synchronize()
    ev2_us = []
    for _ in range(args.reps):
        a0, a1, a2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(st):
            torch.cuda._sleep(2_000_000)
            a0.record(st)
            q4.lily_q4_gemv_argmax(W, x, tok, ws=ws, stream=st)
            a1.record(st)
            q4.lily_q4_gemv_argmax(W, x, tok, ws=ws, stream=st)
            a2.record(st)
        st.synchronize()
        ev_us.append(a0.elapsed_time(a1) * 1e3)
        ev2_us.append(a1.elapsed_time(a2) * 1e3)
        assert L.lily_q4_lm_trace_read(buf.ctypes.data, buf.nbytes) == 0
        t = buf.reshape(1024, 8)[:G].astype(np.int64)
        ref = t[:, 0].min()
        for i, name in POINTS:
            rel[name].append(t[:, i] - ref)
    assert q4.lily_q4_workspace_status(ws, st) == 0
    print(f"{lmw.name}: event-timed call {np.median(ev_us):.2f} us after a spin kernel, "
          f"{np.median(ev2_us):.2f} us right after another LM-head call (medians of {args.reps}); "
          f"{G} blocks; the timeline is the second call's")
    print(f"  {'point':8s} {'median':>8s} {'min':>8s} {'max':>8s}   (us after the first block's "
          f"set-up; median over runs)")
    for _, name in POINTS:
        a = np.stack(rel[name])
        print(f"  {name:8s} {np.median(np.median(a, 1)) / 1e3:8.2f} "
              f"{np.median(a.min(1)) / 1e3:8.2f} {np.median(a.max(1)) / 1e3:8.2f}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
