"""Benchmark of the Q4 MoE hot path on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over synthetic inputs resident in HBM:
  * decode: 40 independently seeded MoE layers (hidden 2048, 256 experts, top-8 + shared,
    intermediate 512), batch 1, one lily_q4_moe_decode call per layer, back to back;
  * LM head: lily_q4_gemv_argmax over a 151,936 x 2048 Q4 head;
  * prefill: one 2048-token chunk through one such layer with skewed router offsets
    (lily_q4_moe_prefill).
`value` is decode tokens/s per MoE layer (layers x tokens / decode time).  Weights of the
40 layers (18.2 GB), the LM head (175 MB) and the prefill layer (455 MB) are each larger
than L2 (129 MB), so every timed read comes from HBM without an explicit flush.

Outside the step, on the same GPU and timed the same way: the 40 layers at batch 4, the
wide-MoE sweep (48 layers of hidden 2048, 512 experts, top-10 + shared, batch 1, 2 and 4),
the LM head with its log-sum-exp and logprobs, the LM head at 8 bits, the decode layer in the
q4-xl layout, and the end-to-end figures through the public API with host copies.  Every
workspace's device-side status is checked after its timed region.

`--impl reference` times the CPU oracle instead (the same metric on the same workload,
a bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4 MoE decode tok/s per layer & HBM GB/s vs peak; prefill chunk TFLOP/s"
UNIT = "tok/s per layer"
EXPERT_BYTES = 1769472  # gate + up + down of one expert at H=2048, I=512 (codes + s + b)
# DRAM bytes (read + write) of one single-launch decode-layer kernel at batch 1, from one ncu
# capture of that kernel (bench.py --layers 2, the third launch).  Set to None whenever that
# kernel changes until it is captured again.
DECODE_TRAFFIC_BYTES = 17064960  # dram__bytes_read.sum 17,064,960 + dram__bytes_write.sum 0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-copy end-to-end section (e.g. under a profiler)")
    ap.add_argument("--no-wide", action="store_true",
                    help="skip the wide-MoE sweep (48 layers, 43.7 GB of weights)")
    return ap.parse_args()


def max_over_ranks(values, device=None):
    """Max of each timing over all ranks (a no-op without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_throughput(units_per_rank, seconds_max, world):
    """Weak-scaling throughput: units all ranks processed / the slowest rank's time."""
    return units_per_rank * world / seconds_max


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi samples during the timed region."""

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"lily_q4_clocks_{os.getpid()}.csv")

    def start(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def check_status(q4, ws, stream, what):
    """Raise if a bounded device-side wait of the workspace's last calls gave up."""
    rc = q4.lily_q4_workspace_status(ws, stream)
    if rc != 0:
        raise RuntimeError(f"{what}: device-side status {rc} ({q4.status_string(rc)})")


def layer_bytes(uniq, E, H, T, expert_bytes=EXPERT_BYTES):
    """Bytes a decode layer must read: the unique routed experts and the shared one, the router
    (bf16 [E][H]), g_shared, x and y."""
    return (uniq + 1) * expert_bytes + E * H * 2 + H * 2 + 2 * T * H * 2


def time_isolated(torch, stream, fn, warmup, reps):
    """Per-call device time of fn (direct launches on `stream`), each call bracketed by its own
    pair of events.  A ~1 ms spin kernel first lets the host enqueue every call before the GPU
    reaches them, so no interval includes host (ctypes) time; the events between calls also
    keep each call from overlapping its neighbours."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
        for a0, a1 in evs:
            a0.record(stream)
            fn()
            a1.record(stream)
    stream.synchronize()
    return [a0.elapsed_time(a1) for a0, a1 in evs]


def time_decode_layers(torch, q4, synth, stream, layers, wl, T, reps, warmup):
    """Layers launched back to back on `stream` (each a programmatic dependent of the previous
    kernel), `reps` passes timed with CUDA events; returns per-layer time and the bytes the
    layers' routing touched."""
    nl = len(layers)
    xs = [q4.to_device(synth.draw_tokens(wl.H, T, wl.tokens_key(l)), torch.device(stream.device))
          for l in range(nl)]
    ys = [torch.empty_like(x) for x in xs]
    idx = torch.empty((nl, T, wl.k), dtype=torch.int32, device=stream.device)
    iv = [idx[l] for l in range(nl)]
    ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(layers[0], T), stream.device)

    def run():
        for l in range(nl):
            q4.lily_q4_moe_decode(layers[l], xs[l], ys[l], topk_idx=iv[l], ws=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            run()
    stream.synchronize()
    ms = []
    for _ in range(reps):
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # the host enqueues the layers before the GPU reaches them
            a0.record(stream)
            run()
            a1.record(stream)
        a1.synchronize()
        ms.append(a0.elapsed_time(a1))
    check_status(q4, ws, stream, f"decode {wl.name} T{T}")
    ih = idx.cpu().numpy()
    uniq = [len(np.unique(ih[l])) for l in range(nl)]
    byts = statistics.mean(layer_bytes(u, wl.E, wl.H, T) for u in uniq)
    us = statistics.mean(ms) * 1e3 / nl
    return us, byts, statistics.mean(uniq), q4.lily_q4_moe_launches(layers[0], T)


def decode_entry(us, byts, uniq, T, launches, hbm_peak, what):
    gbs = byts / (us * 1e-6) / 1e9
    return {"us_per_layer": round(us, 3), "tok_s_per_layer": round(T / (us * 1e-6), 1),
            "bytes_per_layer": int(byts), "unique_experts": round(uniq, 2),
            "hbm_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
            "launches_per_layer": launches, "workload": what}


# ----------------------------------------------------------------------------- GB300 arm

def run_gb300(args):
    import torch
    import torch.distributed as dist

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from bit_affine_quantized_mlx_gb300 import build as q4build
    q4build.build()
    import bit_affine_quantized_mlx_gb300 as q4
    from bit_affine_quantized_mlx_gb300 import synth

    pk = peaks()
    wl, lmw, pfw = synth.DECODE, synth.LMHEAD, synth.PREFILL
    T = args.tokens
    nl = args.layers

    # ---- inputs, resident in HBM before timing
    t0 = time.time()
    layers = [q4.DeviceLayer.upload(wl.layer(l), dev) for l in range(nl)]
    xs = [q4.to_device(synth.draw_tokens(wl.H, T, wl.tokens_key(l)), dev) for l in range(nl)]
    ys = [torch.empty_like(x) for x in xs]
    dws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(layers[0], T), dev)
    idx_all = torch.empty((nl, T, wl.k), dtype=torch.int32, device=dev)
    W = q4.DeviceQ4.upload(synth.draw_lm_head(lmw.V, lmw.H), dev)
    xl = q4.to_device(synth.draw_lm_x(lmw.H), dev)
    tok = torch.empty(1, dtype=torch.int32, device=dev)
    lmws = q4.new_workspace(q4.lily_q4_gemv_argmax_workspace_bytes(lmw.V, lmw.H), dev)
    pl = q4.DeviceLayer.upload(pfw.layer(0), dev)
    Tp = pfw.tokens[0]
    xp = q4.to_device(synth.draw_tokens(pfw.H, Tp, pfw.tokens_key(0)), dev)
    yp = torch.empty_like(xp)
    idxp = torch.empty((Tp, pfw.k), dtype=torch.int32, device=dev)
    pws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(pl, Tp, prefill=True), dev)
    torch.cuda.synchronize()
    gen_s = time.time() - t0

    # The prefill part runs as a CUDA graph (captured after a warm-up call, so one-time library
    # set-up happens outside capture); replaying it keeps the host (ctypes per call) off the
    # critical path, as a serving loop would.  The decode layers and the LM head are launched
    # directly on the stream: each of their kernels is enqueued as a programmatic dependent of
    # the previous kernel, which lets its blocks take SMs while that kernel drains (a graph
    # replay adds its own launch latency, several us for a single-kernel graph).  The host
    # enqueues a launch in a few microseconds, well ahead of the ~16 us kernels, so the GPU
    # never waits for it.
    stream = torch.cuda.Stream(device=dev)

    idx_v = [idx_all[l] for l in range(nl)]  # views made once: slicing costs host time per call

    def dec_part():
        for l in range(nl):
            q4.lily_q4_moe_decode(layers[l], xs[l], ys[l], topk_idx=idx_v[l], ws=dws,
                                  stream=stream)

    def lm_part():
        q4.lily_q4_gemv_argmax(W, xl, tok, ws=lmws, stream=stream)

    def pf_part():
        q4.lily_q4_moe_prefill(pl, xp, yp, topk_idx=idxp, ws=pws, stream=stream)

    parts = [dec_part, lm_part, pf_part]
    with torch.cuda.stream(stream):
        for f in parts:
            f()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pf_part()
    stream.synchronize()
    runs = [dec_part, lm_part, g.replay]

    def step(ev=None):
        with torch.cuda.stream(stream):
            for i, run in enumerate(runs):
                if ev:
                    ev[i].record(stream)
                run()
            if ev:
                ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    check_status(q4, dws, stream, "decode (warm-up)")
    check_status(q4, pws, stream, "prefill (warm-up)")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = Clocks(local)
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    # A ~1 ms spin kernel ahead of the timed region: the host then enqueues the first steps
    # before the GPU reaches them, so no interval includes host (ctypes) launch time (in steady
    # state the host stays ahead: a decode layer's launch costs the host less than the layer
    # takes on the GPU).  It runs before g0, outside the timed region.
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)
    g0.record(stream)
    for s_ in range(args.steps):
        step(evs[s_])
    g1.record(stream)
    torch.cuda.synchronize()
    if ws_n > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = g0.elapsed_time(g1)
    dec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    lm_ms = [e[1].elapsed_time(e[2]) for e in evs]
    pf_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms, dec_mean, lm_mean, pf_mean = max_over_ranks(
        [total_ms, statistics.mean(dec_ms), statistics.mean(lm_ms), statistics.mean(pf_ms)], dev)
    check_status(q4, dws, stream, "decode")
    check_status(q4, lmws, stream, "LM head")
    check_status(q4, pws, stream, "prefill")

    # ---- algorithmic work
    idx_h = idx_all.cpu().numpy()
    uniq = [len(np.unique(idx_h[l])) for l in range(nl)]
    layer_bytes = [(u + 1) * EXPERT_BYTES + wl.E * wl.H * 2 + wl.H * 2 + 2 * T * wl.H * 2
                   for u in uniq]
    bytes_per_layer = statistics.mean(layer_bytes)
    t_layer_s = dec_mean / 1e3 / nl
    dec_gbs = bytes_per_layer / t_layer_s / 1e9
    tok_per_s_layer = replica_throughput(T, t_layer_s, ws_n)
    lm_bytes = lmw.V * lmw.H // 2 + lmw.V * (lmw.H // 64) * 4 + lmw.H * 2 + 4
    lm_gbs = lm_bytes / (lm_mean / 1e3) / 1e9
    P = Tp * (pfw.k + 1)
    pf_flops = 6.0 * P * pfw.H * pfw.I + 2.0 * Tp * pfw.H * pfw.E
    pf_tflops = pf_flops / (pf_mean / 1e3) / 1e12
    # bytes the chunk must read: the experts its routing touched (and the shared one), the
    # router, x and y
    pf_touched = len(np.unique(idxp.cpu().numpy()))
    pf_bytes = (pf_touched + 1) * EXPERT_BYTES + pfw.E * pfw.H * 2 + 2 * Tp * pfw.H * 2

    # ---- end to end through the public API: every step copies all layers' x from pinned host
    # memory in one transfer, makes one lily_q4_moe_decode call per layer, and reads every
    # layer's y back to pinned host memory in one transfer.
    #  * dependent (the e2e value): the host waits for each step's y before it copies the next
    #    step's x in, as a greedy decode loop must (its next input depends on this output);
    #  * overlapped (reported beside it): two buffer sets, step s+1's copy in (on a copy stream)
    #    overlapping step s's layers -- what independent inputs would allow.
    x_host = torch.empty((nl, T, wl.H), dtype=torch.int16, pin_memory=True)
    for l in range(nl):
        x_host[l].copy_(xs[l].cpu())
    y_host = [torch.empty((nl, T, wl.H), dtype=torch.int16, pin_memory=True) for _ in range(2)]
    xdev = [torch.empty((nl, T, wl.H), dtype=torch.int16, device=dev) for _ in range(2)]
    ydev = [torch.empty((nl, T, wl.H), dtype=torch.int16, device=dev) for _ in range(2)]
    xdev_v, ydev_v = [list(b) for b in xdev], [list(b) for b in ydev]
    copy_st = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    buf_free = [torch.cuda.Event(), torch.cuda.Event()]
    for ev in buf_free:
        ev.record(stream)

    def e2e_dep_step():
        with torch.cuda.stream(stream):
            xdev[0].copy_(x_host, non_blocking=True)
            for l in range(nl):
                q4.lily_q4_moe_decode(layers[l], xdev_v[0][l], ydev_v[0][l], ws=dws, stream=stream)
            y_host[0].copy_(ydev[0], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
        ev.synchronize()  # y is on the host

    def e2e_step(s_):
        b = s_ % 2
        with torch.cuda.stream(copy_st):
            copy_st.wait_event(buf_free[b])  # the step two back is done with this buffer set
            xdev[b].copy_(x_host, non_blocking=True)
            h2d_done[b].record(copy_st)
        with torch.cuda.stream(stream):
            stream.wait_event(h2d_done[b])
            for l in range(nl):
                q4.lily_q4_moe_decode(layers[l], xdev_v[b][l], ydev_v[b][l], ws=dws, stream=stream)
            y_host[b].copy_(ydev[b], non_blocking=True)
            buf_free[b].record(stream)

    # ---- LM head with the full-vocabulary log-sum-exp and log-probabilities (the same weights
    # and x as the argmax-only LM head above), timed as the isolated LM heads below
    lse_d = torch.empty(1, dtype=torch.float32, device=dev)
    lp_d = torch.empty(lmw.V, dtype=torch.float32, device=dev)

    def lp_part():
        q4.lily_q4_gemv_argmax_logprobs(W, xl, tok, lse_d, logprobs=lp_d, ws=lmws, stream=stream)

    lp_ms = time_isolated(torch, stream, lp_part, args.warmup, max(args.steps, 3))
    lp_mean = max_over_ranks([statistics.mean(lp_ms)], dev)[0]

    # ---- the argmax LM head in a chain of programmatic-dependent launches, timed as the decode
    # layers are (one event pair around the chain): two independently drawn heads (350 MB,
    # beyond L2) alternate, so no launch finds the previous one's weights in L2.  A launch's
    # weight copies start while the previous launch drains, as they would behind the last
    # decode layer of a step.
    W2 = q4.DeviceQ4.upload(synth.draw_lm_head(lmw.V, lmw.H, key=(lmw.wid, 1)), dev)
    n_chain = 8

    def lm_chain():
        for i in range(n_chain):
            q4.lily_q4_gemv_argmax(W if i % 2 == 0 else W2, xl, tok, ws=lmws, stream=stream)

    ch_ms = time_isolated(torch, stream, lm_chain, args.warmup, max(args.steps, 3))
    ch_mean = max_over_ranks([statistics.mean(ch_ms) / n_chain], dev)[0]
    del W2

    # ---- the same LM head kept at 8 bits (q4-xl), argmax only, timed the same way
    W8 = q4.DeviceQ4.upload(synth.draw_lm_head_q8(lmw.V, lmw.H), dev)
    ws8 = q4.new_workspace(q4.lily_q8_gemv_argmax_workspace_bytes(lmw.V, lmw.H), dev)

    def q8_part():
        q4.lily_q8_gemv_argmax(W8, xl, tok, ws=ws8, stream=stream)

    q8_ms = time_isolated(torch, stream, q8_part, args.warmup, max(args.steps, 3))
    q8_mean = max_over_ranks([statistics.mean(q8_ms)], dev)[0]
    q8_bytes = lmw.V * lmw.H + lmw.V * (lmw.H // 64) * 4 + lmw.H * 2 + 4
    q8_gbs = q8_bytes / (q8_mean / 1e3) / 1e9
    del W8, ws8

    # ---- decode layers in the q4-xl layout (8-bit router and shared expert), batch 1: eight
    # independently seeded layers (3.6 GB, beyond L2) cycled, stream launches as above
    xl_layers = [q4.DeviceLayer.upload(synth.draw_layer(wl.H, wl.E, wl.k, wl.I, shared=True,
                                                        router_std=0.02, router_bias=False,
                                                        key=(wl.wid, 1000 + l), router_bits=8,
                                                        shared_bits=8), dev) for l in range(8)]
    xl_x = [q4.to_device(synth.draw_tokens(wl.H, T, (wl.wid, 1000 + l)), dev) for l in range(8)]
    xl_y = torch.empty_like(xl_x[0])
    xl_ws = q4.new_workspace(q4.lily_q4_moe_workspace_bytes(xl_layers[0], T), dev)

    def xl_part(n):
        for i in range(n):
            q4.lily_q4_moe_decode(xl_layers[i % 8], xl_x[i % 8], xl_y, ws=xl_ws, stream=stream)

    with torch.cuda.stream(stream):
        xl_part(16)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        xl_part(200)
        a1.record(stream)
        a1.synchronize()
    xl_us = max_over_ranks([a0.elapsed_time(a1) * 1e3 / 200], dev)[0]
    check_status(q4, xl_ws, stream, "q4-xl decode")
    del xl_layers

    # ---- the 40 decode layers at batch 4, and the wide-MoE sweep: 48 independently seeded
    # layers of hidden 2048, 512 experts, top-10 + shared, intermediate 512, at batch 1, 2, 4
    # (43.7 GB of weights), each timed over `steps` passes of all its layers
    t4 = time_decode_layers(torch, q4, synth, stream, layers, wl, 4, args.steps, args.warmup)
    decode_t4 = decode_entry(*t4[:3], 4, t4[3], pk["hbm_gbs"],
                             f"decode MoE H2048 E256 top-8 + shared I512, batch 4, {nl} layers")
    wide = {}
    if not args.no_wide:
        ww = synth.WIDE
        wlayers = [q4.DeviceLayer.upload(ww.layer(l), dev) for l in range(ww.layers)]
        for Tw in ww.tokens:
            r_ = time_decode_layers(torch, q4, synth, stream, wlayers, ww, Tw, args.steps, args.warmup)
            wide[f"wide_t{Tw}"] = decode_entry(*r_[:3], Tw, r_[3], pk["hbm_gbs"],
                                               f"wide MoE H2048 E512 top-10 + shared I512, batch {Tw}, "
                                               f"{ww.layers} layers")
        del wlayers
        torch.cuda.empty_cache()

    e2e_val = e2e_ovl = None
    if not args.no_e2e:
        ref_y = torch.stack(ys).cpu().numpy()
        for _ in range(2):
            e2e_dep_step()
        e0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_dep_step()
        e2e_s = max_over_ranks([(time.perf_counter() - e0) / args.steps], dev)[0]
        e2e_val = round(replica_throughput(nl * T, e2e_s, ws_n), 1)
        if not np.array_equal(y_host[0].numpy(), ref_y):
            raise RuntimeError("end-to-end decode outputs differ from the device-timed ones")
        for s_ in range(2):
            e2e_step(s_)
        torch.cuda.synchronize()
        e0 = time.perf_counter()
        for s_ in range(args.steps):
            e2e_step(s_)
        torch.cuda.synchronize()
        e2e_o = max_over_ranks([(time.perf_counter() - e0) / args.steps], dev)[0]
        e2e_ovl = round(replica_throughput(nl * T, e2e_o, ws_n), 1)
        if not np.array_equal(y_host[(args.steps - 1) % 2].numpy(), ref_y):
            raise RuntimeError("end-to-end decode outputs differ from the device-timed ones")
        check_status(q4, dws, stream, "decode (end to end)")

    launches_per_step = (sum(q4.lily_q4_moe_launches(L_, T) for L_ in layers) + 1 +
                         q4.lily_q4_moe_launches(pl, Tp, prefill=True))
    res = {
        "metric": METRIC,
        "value": round(tok_per_s_layer, 1),
        "unit": UNIT,
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4 weights, bf16 activations, fp32 accumulation",
        "data": "synthetic (seeded generator; value distributions of the workloads)",
        "config": {
            "workload": f"decode MoE H2048 E256 top-8 + shared I512, batch {T}, {nl} "
                        "independently seeded layers; + LM head 151936x2048 argmax; + prefill "
                        "chunk 2048 tokens through one skewed-router layer",
            "layers": nl, "tokens": T, "parallelism": f"replicas x{ws_n}",
            "l2": "no flush: every timed read set (18.2 GB layers, 175 MB head, 455 MB prefill "
                  "layer) exceeds the 129 MB L2",
        },
        "decode": {"tok_s_per_layer": round(tok_per_s_layer, 1), "us_per_layer": round(t_layer_s * 1e6, 3),
                   "bytes_per_layer": int(bytes_per_layer), "hbm_gbs": round(dec_gbs, 1),
                   "frac_of_measured_hbm": round(dec_gbs / pk["hbm_gbs"], 4)},
        "lm_head": {"us": round(lm_mean * 1e3, 2), "bytes": lm_bytes,
                    "hbm_gbs": round(lm_gbs, 1), "frac_of_measured_hbm": round(lm_gbs / pk["hbm_gbs"], 4),
                    "with_logprobs_us": round(lp_mean * 1e3, 2),
                    "chained_us": round(ch_mean * 1e3, 2),
                    "chained_hbm_gbs": round(lm_bytes / (ch_mean / 1e3) / 1e9, 1),
                    "chained_frac_of_measured_hbm": round(lm_bytes / (ch_mean / 1e3) / 1e9 / pk["hbm_gbs"], 4),
                    "scope": "us: one launch between events after the step's decode layers; "
                             "chained_us: per launch in a chain of 8 programmatic-dependent "
                             "launches alternating two heads"},
        "lm_head_q8": {"us": round(q8_mean * 1e3, 2), "bytes": q8_bytes, "hbm_gbs": round(q8_gbs, 1),
                       "frac_of_measured_hbm": round(q8_gbs / pk["hbm_gbs"], 4)},
        "decode_q4xl": {"us_per_layer": round(xl_us, 3), "tok_s_per_layer": round(T / (xl_us * 1e-6), 1),
                        "layout": "8-bit router and shared expert, 4-bit routed experts; 8 layers cycled"},
        "decode_t4": decode_t4,
        **wide,
        "prefill": {"us": round(pf_mean * 1e3, 1), "gflop": round(pf_flops / 1e9, 2),
                    "tflops": round(pf_tflops, 1),
                    "frac_of_measured_bf16": round(pf_tflops / pk["bf16_tflops_sustained"], 4),
                    "tok_s": round(Tp / (pf_mean / 1e3), 1),
                    "experts_touched": pf_touched, "bytes": pf_bytes,
                    "hbm_gbs": round(pf_bytes / (pf_mean / 1e3) / 1e9, 1),
                    "frac_of_burst_bf16": round(pf_tflops / pk["bf16_tflops"], 4)},
        "roofline": {"bound": "hbm", "kernel": "lily_q4_moe_decode (router+top-k, gate/up, down)",
                     "achieved": round(dec_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(dec_gbs / pk["hbm_gbs"], 4), "peak_source": pk["source"],
                     "traffic": DECODE_TRAFFIC_BYTES if T == 1 else None},
        "e2e": {"value": e2e_val, "unit": UNIT,
                "h2d_bytes_per_step": nl * T * wl.H * 2, "d2h_bytes_per_step": nl * T * wl.H * 2,
                "scope": "decode layers through lily_q4_moe_decode; per step one copy of all "
                         "layers' x from pinned host memory, the layers, and one copy of all y "
                         "back, which the host waits for before the next step's copy in",
                "overlapped_value": e2e_ovl,
                "overlapped_scope": "the same with two buffer sets, the next step's copy in "
                                    "overlapping the current step's layers (independent inputs)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "setup_s": round(gen_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws_n > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- oracle timing

def _oracle_layer_time(wl, l, T):
    from bit_affine_quantized_mlx_gb300 import synth
    from oracle import oracle as orc
    L = wl.layer(l)
    x = synth.draw_tokens(wl.H, T, wl.tokens_key(l))
    t0 = time.perf_counter()
    orc.moe(L, x)
    return time.perf_counter() - t0


def cpu_model():
    """The host CPU's model name (/proc/cpuinfo or lscpu) and logical core count."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip().lower() in ("model name", "vendor id") and ":" in line:
                v = line.split(":", 1)[1].strip()
                name = v if name is None else f"{name} {v}"
    except Exception:
        pass
    if not name:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    name = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return name or "unknown", os.cpu_count()


def cpu_baseline(wl):
    """The oracle (as it stands: OpenMP over tokens, over rows for the LM head) on this host's
    cores, on bounded samples of the workloads:
      * decode layer, batch 1 (the metric): one token runs on one thread;
      * decode layer, a batch of one token per thread, all threads (tokens in parallel);
      * LM head 151,936 x 2048 + argmax: all threads (rows in parallel) and one thread;
      * prefill chunk of 2048 tokens: a 64-token sample on all threads, scaled to the chunk."""
    from bit_affine_quantized_mlx_gb300 import synth
    from oracle import oracle as orc
    orc.build()
    n_all = orc.threads()
    model, ncpu = cpu_model()
    # decode, batch 1, one thread: two layers, three timings each
    dec = []
    for l in range(2):
        L = wl.layer(l)
        x = synth.draw_tokens(wl.H, 1, wl.tokens_key(l))
        for _ in range(3):
            t0 = time.perf_counter()
            orc.moe(L, x)
            dec.append(time.perf_counter() - t0)
    per_layer = statistics.median(dec)
    # decode, one token per thread, all threads (the last layer drawn above)
    xb = synth.draw_tokens(wl.H, n_all, wl.tokens_key(1))
    t0 = time.perf_counter()
    orc.moe(L, xb)
    batch_s = time.perf_counter() - t0
    # LM head: all threads, then one thread
    lmw = synth.LMHEAD
    W = synth.draw_lm_head(lmw.V, lmw.H)
    xl = synth.draw_lm_x(lmw.H)
    t0 = time.perf_counter()
    orc.lm_head(W, xl)
    lm_all = time.perf_counter() - t0
    orc.set_threads(1)
    try:
        t0 = time.perf_counter()
        orc.lm_head(W, xl)
        lm_one = time.perf_counter() - t0
    finally:
        orc.set_threads(n_all)
    del W
    # prefill: 64 tokens of the 2048-token chunk on all threads
    pw = synth.PREFILL
    Lp = pw.layer(0)
    xp = synth.draw_tokens(pw.H, 64, pw.tokens_key(0))
    t0 = time.perf_counter()
    orc.moe(Lp, xp)
    pf64 = time.perf_counter() - t0
    Tp = pw.tokens[0]
    return {"value": round(1 / per_layer, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "decode MoE layer (H2048 E256 top-8 + shared I512) at batch 1: 2 of the 40 "
                      "layers, 3 timings each, median; input generation excluded",
            "cpu_model": model, "host_logical_cpus": ncpu, "oracle_threads": n_all,
            "decode_ms_per_layer_1_thread": round(per_layer * 1e3, 2),
            "decode_batch_all_threads": {"tokens": n_all, "threads": n_all,
                                         "ms_per_layer": round(batch_s * 1e3, 1),
                                         "tok_s_per_layer": round(n_all / batch_s, 2)},
            "lm_head_ms": {"all_threads": round(lm_all * 1e3, 1), "threads": n_all,
                           "one_thread": round(lm_one * 1e3, 1)},
            "prefill_chunk_s": {"all_threads": round(pf64 * Tp / 64, 2), "threads": n_all,
                                "sample": "64 of the 2048 tokens, scaled to the chunk",
                                "tok_s": round(64 / pf64, 1)}}


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    from bit_affine_quantized_mlx_gb300 import synth
    from oracle import oracle as orc
    orc.build()
    wl = synth.DECODE
    T = args.tokens
    for s in range(args.warmup):
        _oracle_layer_time(wl, s % wl.layers, T)
    times = [_oracle_layer_time(wl, s % wl.layers, T) for s in range(args.steps)]
    per_layer = statistics.mean(times)
    val = T / per_layer
    cores = 1 if T == 1 else orc.threads()
    res = {
        "impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": UNIT,
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_layer * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 dequant, fp64 accumulation", "data": "synthetic",
        "config": {"workload": f"decode MoE H2048 E256 top-8 + shared I512, batch {T}; one "
                               "layer per step (the CPU oracle)", "tokens": T},
        "cpu_baseline": {"value": round(val, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"one decode layer per step, {args.steps} steps"},
        "e2e": {"value": round(val, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
