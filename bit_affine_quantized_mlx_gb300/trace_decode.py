"""Phase timeline of the single-launch decode kernel on a chain of seeded MoE layers.

Builds the profiling variant of the library (``build(trace=True)``: the same sources with
``-DLILY_Q4_TRACE``), runs ``lily_q4_moe_decode`` over N independently seeded layers back
to back on one stream (each launch a programmatic dependent of the previous one, as in a
decode step), and prints, for the last launch, when each block reached each point of the
kernel, relative to the moment the previous launch had completed (the earliest return of
``griddepcontrol.wait`` over the blocks):

  wait     griddepcontrol.wait returned (previous kernel complete)
  x        x prepared in shared memory
  A        phase A done: router rows and shared-expert gate/up rows
  bar1     first grid barrier passed (every block's logits written)
  routed   top-k, softmax and the pair table built
  B        routed gate/up rows done, down rows being copied in
  bar2     second grid barrier passed (every pair's h written)
  h        h of every pair prepared, the down rows landed
  down     down rows done
  y        y written (the block's end)

and the gap between launches: from the previous launch's last block writing y to this
launch's first return from the wait.  The timestamps are %globaltimer reads by thread 0 of
each block, so the figures are a profile of the kernel as it runs, not a bench number.

    python -m bit_affine_quantized_mlx_gb300.trace_decode [--layers 40] [--reps 20]
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

POINTS = [(7, "wait"), (0, "x"), (1, "A"), (2, "bar1"), (3, "routed"), (4, "B"), (5, "bar2"),
          (6, "h"), (8, "down"), (9, "y")]
NPOINT = 16  # slots per block in the trace array
NBLOCK = 1024


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--tokens", type=int, nargs="*", default=[1, 4])
    ap.add_argument("--wide", action="store_true", help="the 512-expert top-10 layer shapes")
    args = ap.parse_args(argv)

    from bit_affine_quantized_mlx_gb300 import build as _build
    lib_path = _build.build(trace=True)
    import torch
    import bit_affine_quantized_mlx_gb300 as q4
    from bit_affine_quantized_mlx_gb300 import synth
    L = q4.load(lib_path)
    L.lily_q4_trace_read.argtypes = [C.c_void_p, C.c_size_t]
    L.lily_q4_trace_read.restype = C.c_int

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    st = torch.cuda.Stream(device=dev)
    wl = synth.WIDE if args.wide else synth.DECODE
    layers = [q4.DeviceLayer.upload(wl.layer(l), dev) for l in range(args.layers)]
    G = torch.cuda.get_device_properties(dev).multi_processor_count
    buf = np.zeros(2 * NBLOCK * NPOINT, dtype=np.uint64)
    for T in args.tokens:
        xs = [q4.to_device(synth.draw_tokens(wl.H, T, wl.tokens_key(l)), dev)
              for l in range(args.layers)]
        ys = [torch.empty_like(x) for x in xs]
        ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(layers[0], T), dev)
        assert q4.lily_q4_moe_launches(layers[0], T) == 1, "shapes outside the single launch"

        def run():
            for l in range(args.layers):
                q4.lily_q4_moe_decode(layers[l], xs[l], ys[l], ws=ws, stream=st)

        with torch.cuda.stream(st):
            for _ in range(3):
                run()
        st.synchronize()
        rel = {name: [] for _, name in POINTS}
        gaps, periods = [], []
        for _ in range(args.reps):
            with torch.cuda.stream(st):
                run()
            st.synchronize()
            assert L.lily_q4_trace_read(buf.ctypes.data, buf.nbytes) == 0
            t = buf.reshape(2, NBLOCK, NPOINT)[:, :G, :].astype(np.int64)
            # the later of the two launches held (parities) is the last one
            last = 0 if t[0, :, 7].min() > t[1, :, 7].min() else 1
            cur, prev = t[last], t[1 - last]
            ref = cur[:, 7].min()
            for i, name in POINTS:
                rel[name].append(cur[:, i] - ref)
            gaps.append(ref - prev[:, 9].max())
            periods.append(ref - prev[:, 7].min())
        q4.lily_q4_workspace_status(ws, st)
        print(f"{wl.name}, T={T}, {args.layers} layers, {G} blocks: per-layer period "
              f"{np.median(periods) / 1e3:.2f} us; previous launch's last y -> this launch's "
              f"first wait return {np.median(gaps) / 1e3:.2f} us")
        print(f"  {'point':8s} {'median':>8s} {'min':>8s} {'max':>8s}   (us after the wait, "
              f"over blocks; median over {args.reps} runs)")
        for _, name in POINTS:
            a = np.stack(rel[name])  # [reps][blocks]
            print(f"  {name:8s} {np.median(np.median(a, 1)) / 1e3:8.2f} "
                  f"{np.median(a.min(1)) / 1e3:8.2f} {np.median(a.max(1)) / 1e3:8.2f}")
        del xs, ys, ws
    return 0


if __name__ == "__main__":
    sys.exit(main())
