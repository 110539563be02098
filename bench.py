"""Benchmark of the GB300 sparse-MoE expert path (one JSON line on rank 0).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path (route -> grouped FFN -> combine) over one batch of
synthetic input of the workload.  Default workload: the 512-token prefill chunk (T=512, d=2048,
256 experts, top-8, I=512 + shared expert), whose 455 MB of 4-bit weights exceed L2, so every
step streams its inputs from HBM (a workload whose layer fits in L2 rotates through enough
independent layer copies to exceed it).  Timing: W untimed steps, then K steps between CUDA events on
the launching stream (prefill steps are replayed 8 at a time from one CUDA graph of the library
calls; every 8th such chunk runs its steps from one graph per phase instead, with events between
the phases that give the gate/up and down kernel times; K is rounded up to a multiple of 8),
barrier + synchronize on both sides, max over ranks.  Multi-GPU (torchrun): every rank runs its own
chunks (weak scaling, no collective on the data path).

--impl reference times the CPU oracle on bounded samples of the same workload on the host
cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer routed tokens/s (prefill) & decode µs/token; % of TC/HBM roofline"
DEFAULT_WORKLOAD = "prefill_t512_d2048"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ablations", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode: layer copies (default: the workload's); fewer for small profiling captures")
    ap.add_argument("--cpu-sample-tokens", type=int, default=32)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_rotation(items, rank):
    """Weak scaling: rank r takes the chunks starting at its own offset r (mod the chunk count)."""
    k = rank % len(items)
    return items[k:] + items[:k]


def max_over_ranks(x, dist=None):
    """The slowest rank's value (a host-tensor all-reduce over the process group; the data path
    itself has no collective)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=open(self.out, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.out):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), active=f[4], hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        try:
            os.remove(self.out)
        except OSError:
            pass
        if not rows:
            return {"samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in rows])), "sm_max_mhz": rows[0]["smax"],
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------------------------- work
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the roofline kernel,
# from an ncu full capture of the current kernels on each workload (None: not captured)
TRAFFIC_BYTES = {
    "prefill_t512_d2048": 322.273536e6 + 9.660928e6,     # ffn_tm_kernel<0, 0> (gate/up)
    "prefill_t4096_d2048": 454.402304e6 + 61.936384e6,   # ffn_tm_kernel<0, 0> (gate/up)
    "decode_t1_d2048": 17.082624e6,                       # decode_fused, one layer
}


def algorithmic_counts(shp, counts):
    """Per-launch algorithmic bytes and FLOPs of the gate/up and down kernels (real rows only)."""
    T, d, I = shp.T, shp.d, shp.I
    touched = int((counts > 0).sum()) + 1                       # + the shared expert
    q4 = lambda rows, cols: rows * cols // 2 + rows * (cols // 64) * 4   # codes + bf16 scale/bias
    gu_w = touched * 2 * q4(I, d)
    dn_w = touched * q4(d, I)
    rows = 9 * T                                                # routed assignments + shared rows
    gu_bytes = gu_w + rows * d * 2 + rows * 2 * I * 2           # weights + activation rows + h (hi|lo)
    dn_bytes = dn_w + rows * 2 * I * 2 + T * d * 4 * 2          # weights + h + fp32 sum (read+write)
    gu_flops = 2.0 * rows * d * 2 * I
    dn_flops = 2.0 * rows * I * d
    return dict(gu_bytes=gu_bytes, dn_bytes=dn_bytes, gu_flops=gu_flops, dn_flops=dn_flops,
                weights_bytes=gu_w + dn_w, touched=touched)


def run_ours(args, rank, world, local):
    import torch
    import quantized_grouped_gemm_gb300 as moe
    from moe_workload import configs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = configs.WORKLOADS[args.workload]
    sh = wl.shape
    decode = sh.T == 1
    T = wl.chunk or sh.T
    shp = moe.shape(T, sh.d, sh.E, sh.k, sh.I, sh.I_shared)
    L2_BYTES = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 10**6)
    # 4-bit codes plus a bf16 scale and bias per 64 weights, gate/up/down of every expert
    layer_bytes = sum(n * (3 * sh.d * i // 2 + 3 * sh.d * i // 16) for n, i in ((sh.E, sh.I), (1, sh.I_shared)))
    # a step's weights must not sit in L2 between steps: a workload whose layer fits rotates
    # through enough independent layer copies to exceed twice the L2 size
    layers = (args.layers or wl.layers) if decode else max(1, -(-2 * L2_BYTES // layer_bytes))

    def to_dev(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a)).to(dev)

    # weights: `layers` independent copies (decode; small prefill layers), else one layer
    L = []
    for li in range(layers):
        lay = configs.make_layer(wl, layer=li)
        q = lambda m: (to_dev(m.codes), to_dev(m.scales), to_dev(m.biases))
        pr = moe.moe_pack_weights(shp, q(lay.routed.gate), q(lay.routed.up), q(lay.routed.down), sh.I)
        ps = moe.moe_pack_weights(shp, q(lay.shared.gate), q(lay.shared.up), q(lay.shared.down), sh.I_shared)
        torch.cuda.synchronize()
        L.append(dict(wr=to_dev(lay.w_router), bias=None if lay.logit_bias is None else to_dev(lay.logit_bias),
                      pr=pr, ps=ps))
        del lay
    # activations: prefill chunks of this rank, or decode steps
    if decode:
        nsteps_x = 1000
        x_all = to_dev(configs.make_decode_x(wl, nsteps_x))
    else:
        x_full = configs.make_x(wl)
        nchunk = sh.T // T
        xs = [to_dev(np.ascontiguousarray(x_full[c * T:(c + 1) * T])) for c in range(nchunk)]
        del x_full
        if world > 1:      # weak scaling: each rank its own rotation of the chunks
            xs = rank_rotation(xs, rank)
    rt = moe.Routing(T)
    ws = moe.workspace(shp)
    y = torch.empty(T, sh.d, dtype=torch.int16, device=dev)
    x_in = torch.zeros(T, sh.d, dtype=torch.int16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    opts = moe.options()

    # ---- capture one step as graphs (per phase for prefill, all layers for decode)
    n0 = moe.moe_launch_count()
    graphs = {}
    with torch.cuda.stream(stream):
        if decode:
            g = torch.cuda.CUDAGraph()
            for li in range(layers):   # warm the kernels once outside capture
                moe.moe_forward(shp, x_in, L[li]["wr"], L[li]["bias"], L[li]["pr"], L[li]["ps"], rt, ws, y, opts,
                                stream)
            stream.synchronize()
            n0 = moe.moe_launch_count()
            with torch.cuda.graph(g, stream=stream):
                for li in range(layers):
                    moe.moe_forward(shp, x_in, L[li]["wr"], L[li]["bias"], L[li]["pr"], L[li]["ps"], rt, ws, y, opts,
                                    stream)
            graphs["step"] = g
        else:
            # one set of phase graphs per (layer copy, resident chunk buffer): a step reads its
            # chunk in place; step s runs layer s % layers on chunk s % chunks
            def calls_for(lw, xc):
                return {
                    "route": lambda: moe.moe_route(shp, xc, lw["wr"], lw["bias"], rt, ws, opts, stream),
                    "gate_up": lambda: moe.moe_ffn_gate_up(shp, xc, rt, lw["pr"], lw["ps"], ws, opts, stream),
                    "down": lambda: moe.moe_ffn_down(shp, rt, lw["pr"], lw["ps"], ws, opts, stream),
                    "combine": lambda: moe.moe_combine(shp, rt, ws, y, opts, stream),
                }
            nsets = int(np.lcm(layers, len(xs)))
            for gi in range(nsets):
                for f in calls_for(L[gi % layers], xs[gi % len(xs)]).values():
                    f()
            stream.synchronize()
            # per set: the four phases as separate graphs (probe chunks, below, run these with
            # events between them for the kernel times); and MULTI consecutive steps (a multiple
            # of the set count) as one graph, in which consecutive kernels, also across steps,
            # overlap their prologues through programmatic dependent launch
            graphs = []
            for gi in range(nsets):
                if gi == 0:
                    n0 = moe.moe_launch_count()
                gc = {}
                calls = calls_for(L[gi % layers], xs[gi % len(xs)])
                for name, f in calls.items():
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        f()
                    gc[name] = g
                if gi == 0:
                    launches_one_chunk = moe.moe_launch_count() - n0
                graphs.append(gc)
            MULTI = nsets * -(-8 // nsets)
            multi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(multi, stream=stream):
                for s in range(MULTI):
                    for f in calls_for(L[s % layers], xs[s % len(xs)]).values():
                        f()
    launches_per_step = moe.moe_launch_count() - n0 if decode else launches_one_chunk
    torch.cuda.synchronize()

    # prefill: steps run in chunks of MULTI (one graph replay; each step reads its chunk where it
    # resides); every PROBE-th chunk runs its steps phase by phase with events in between.
    # decode: a step copies its token's activations (4 KB) into the graph's input buffer first
    PROBE = 8
    if decode:
        MULTI = 1

    def step(s, ev=None):
        if decode:
            x_in.copy_(x_all[s % nsteps_x:s % nsteps_x + 1], non_blocking=True)
            graphs["step"].replay()
        else:
            gc = graphs[s % len(graphs)]
            gc["route"].replay()
            if ev is not None:
                ev[0].record(stream)
            gc["gate_up"].replay()
            if ev is not None:
                ev[1].record(stream)
            gc["down"].replay()
            if ev is not None:
                ev[2].record(stream)
            gc["combine"].replay()

    def chunk(c, evs=None):
        """Steps c*MULTI .. c*MULTI + MULTI - 1."""
        if decode:
            step(c)
        elif evs is None:
            multi.replay()
        else:
            for j in range(MULTI):
                step(c * MULTI + j, evs[j])

    dist = None
    if world > 1:
        import torch.distributed as dist
    with torch.cuda.stream(stream):
        nwarm = -(-args.warmup // MULTI)
        for c in range(nwarm):
            chunk(c)
        if not decode:   # the phase graphs too
            chunk(0, [None] * MULTI)
        stream.synchronize()
        warmup_steps = nwarm * MULTI + (0 if decode else MULTI)
        # auto step count: about 1.5 s of timed work
        if args.steps is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = max(1, 24 // MULTI)
            e0.record(stream)
            for c in range(n):
                chunk(c)
            e1.record(stream)
            e1.synchronize()
            per = e0.elapsed_time(e1) / (n * MULTI)
            K = int(min(20000, max(20, 1500.0 / max(per, 1e-3))))
        else:
            K = args.steps
        nchunks = -(-K // MULTI)
        K = nchunks * MULTI
        evs = {c: [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(MULTI)]
               for c in range(0, nchunks, PROBE)} if not decode else {}
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.15)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for c in range(nchunks):
            chunk(c, evs.get(c))
        t1.record(stream)
        t1.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist)
    ms_step = ms_total / K
    rc, bits = moe.moe_read_status(ws, stream)
    assert rc == moe.MOE_OK, f"device status {rc} bits {bits}"

    P = peaks()
    res = dict(metric=METRIC, n_gpus=world, steps=K, warmup=warmup_steps, ms_per_step=ms_step, data="synthetic",
               scaling="weak", vs_baseline=None, dtype="bf16", clocks=clk,
               gpu_launches=int(launches_per_step * K))
    if decode:
        us_tok_layer = ms_step * 1000.0 / layers
        res.update(value=us_tok_layer, unit="us/token/layer", higher_is_better=False)
        # router weight (bf16) + gate, up, down of 8 routed + 1 shared expert (4-bit + bf16 scale/bias per 64)
        bytes_layer = sh.E * sh.d * 2 + 9 * (3 * sh.d * sh.I // 2 + 3 * sh.d * sh.I // 64 * 4)
        gbs = bytes_layer / (us_tok_layer * 1e-6) / 1e9
        res["roofline"] = dict(bound="hbm", achieved=gbs, peak=P["hbm_gbs"], unit="GB/s", frac=gbs / P["hbm_gbs"],
                               traffic=TRAFFIC_BYTES.get(wl.name), kernel="decode_fused (one launch per layer: route + gate/up + down + combine)",
                               bytes_per_token_layer=bytes_layer, peak_source=P["source"])
        res["config"] = dict(workload=wl.name, T=1, d=sh.d, E=sh.E, k=sh.k, I=sh.I, I_shared=sh.I_shared,
                             layers=layers, l2=f"inputs larger than L2: {layers} layer copies of the weights, "
                                                 f"{layers * layer_bytes / 1e9:.0f} GB",
                             parallelism=f"replicas x{world}")
    else:
        value = world * T * K / (ms_total / 1000.0)
        res.update(value=value, unit="routed tokens/s", higher_is_better=True)
        ph = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])] for ce in evs.values() for e in ce])
        gu_ms, dn_ms = float(ph[:, 0].mean()), float(ph[:, 1].mean())
        counts = rt.counts.cpu().numpy()
        A = algorithmic_counts(shp, counts)
        # dominant kernel: gate/up. Bound: HBM when its arithmetic intensity is below the ridge
        ai = A["gu_flops"] / A["gu_bytes"]
        ridge = P["bf16_tflops"] * 1e12 / (P["hbm_gbs"] * 1e9)
        if ai < ridge:
            ach = A["gu_bytes"] / (gu_ms * 1e-3) / 1e9
            roof = dict(bound="hbm", achieved=ach, peak=P["hbm_gbs"], unit="GB/s", frac=ach / P["hbm_gbs"])
        else:
            ach = A["gu_flops"] / (gu_ms * 1e-3) / 1e12
            roof = dict(bound="tensor", achieved=ach, peak=P["bf16_tflops"], unit="TFLOP/s", frac=ach / P["bf16_tflops"])
        roof.update(traffic=TRAFFIC_BYTES.get(wl.name), kernel="ffn_tm_kernel<0> (gate/up + SwiGLU; tcgen05, dequantised weights in TMEM)", algorithmic_bytes=A["gu_bytes"],
                    algorithmic_flops=A["gu_flops"], kernel_ms=gu_ms, peak_source=P["source"])
        res["roofline"] = roof
        ffn_ms = gu_ms + dn_ms
        res["ffn"] = dict(gate_up_ms=gu_ms, down_ms=dn_ms, ffn_tflops=(A["gu_flops"] + A["dn_flops"]) / (ffn_ms * 1e-3) / 1e12,
                          ffn_frac_bf16_peak=(A["gu_flops"] + A["dn_flops"]) / (ffn_ms * 1e-3) / 1e12 / P["bf16_tflops"],
                          ffn_weight_gbs=A["weights_bytes"] / (ffn_ms * 1e-3) / 1e9,
                          experts_touched=A["touched"], other_ms=ms_step - ffn_ms)
        res["config"] = dict(workload=wl.name, T=T, d=sh.d, E=sh.E, k=sh.k, I=sh.I, I_shared=sh.I_shared,
                             chunks=sh.T // T, layers=layers,
                             l2=f"inputs larger than L2: {layers} layer cop{'y' if layers == 1 else 'ies'} of "
                                f"{layer_bytes / 1e6:.0f} MB of 4-bit weights, a step reads one",
                             parallelism=f"replicas x{world}")

    # ---- end to end through the public API with host buffers (pinned), copies timed
    if not decode:
        # Every step copies its chunk in from pinned host memory, runs moe_forward and copies its
        # output back, all inside the timed region.  The copies run on a copy stream into two
        # device buffers, so the input of step s+1 and the output of step s-1 move while step s
        # computes (consecutive steps share the workspace and run in order on `stream`).
        xh = [t.cpu().pin_memory() for t in xs[:4]]
        cs = torch.cuda.Stream(device=dev)
        xb = [torch.empty(T, sh.d, dtype=torch.int16, device=dev) for _ in range(2)]
        yb = [torch.empty(T, sh.d, dtype=torch.int16, device=dev) for _ in range(2)]
        yh = [torch.empty(T, sh.d, dtype=torch.int16).pin_memory() for _ in range(2)]
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]

        def h2d(s):   # waits until step s-2 (same buffers) has finished
            i = s & 1
            cs.wait_event(ev_done[i])
            with torch.cuda.stream(cs):
                xb[i].copy_(xh[s % len(xh)], non_blocking=True)
            ev_in[i].record(cs)

        def compute(s):
            i = s & 1
            lw = L[s % layers]
            stream.wait_event(ev_in[i])
            moe.moe_forward(shp, xb[i], lw["wr"], lw["bias"], lw["pr"], lw["ps"], rt, ws, yb[i], opts, stream)
            ev_done[i].record(stream)

        def d2h(s):
            i = s & 1
            cs.wait_event(ev_done[i])
            with torch.cuda.stream(cs):
                yh[i].copy_(yb[i], non_blocking=True)

        def run(n, start):
            cs.wait_event(start)
            h2d(0)
            for s in range(n):
                if s + 1 < n:
                    h2d(s + 1)
                compute(s)
                d2h(s)

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run(3, a)
        torch.cuda.synchronize()
        Ke = min(K, 2000)
        a.record(stream)
        run(Ke, a)
        b.record(cs)   # after the last output copy, which follows the last step
        b.synchronize()
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b)
        res["e2e"] = dict(value=world * T * Ke / (e_ms / 1000.0), unit="routed tokens/s",
                          h2d_bytes_per_step=T * sh.d * 2, d2h_bytes_per_step=T * sh.d * 2,
                          copies="pinned host buffers; copy stream overlapped with compute, two buffers")
        if not args.no_ablations:
            res["ablations"] = ablations(moe, shp, L, layers, xs, rt, ws, y, stream, T, world)
    else:
        xh = configs.make_decode_x(wl, 16)
        xh_t = torch.from_numpy(xh.view(np.int16)).pin_memory()
        yh = torch.empty(1, sh.d, dtype=torch.int16).pin_memory()
        with torch.cuda.stream(stream):
            def e2e_step(s):
                x_in.copy_(xh_t[s % 16:s % 16 + 1], non_blocking=True)
                graphs["step"].replay()
                yh.copy_(y, non_blocking=True)
            for s in range(3):
                e2e_step(s)
            stream.synchronize()
            Ke = min(K, 200)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for s in range(Ke):
                e2e_step(s)
            b.record(stream)
            b.synchronize()
        e_ms = a.elapsed_time(b)
        res["e2e"] = dict(value=e_ms * 1000.0 / Ke / layers, unit="us/token/layer",
                          h2d_bytes_per_step=sh.d * 2, d2h_bytes_per_step=sh.d * 2)
    return res, wl


def ablations(moe, shp, L, layers, xs, rt, ws, y, stream, T, world, n=100):
    """Outside the timed region: the step launched eagerly through moe_forward with the default
    design and with each ablation of it: the host round trip of the routing counts
    (moe_options.host_routing, one stream synchronisation per step) and dequantisation as a
    separate pass that writes bf16 weights before the GEMMs (moe_options.unfused_dequant)."""
    import torch

    def eager(opts, w):
        def one(s):
            lw = L[s % layers]
            moe.moe_forward(shp, xs[s % len(xs)], lw["wr"], lw["bias"], lw["pr"], lw["ps"], rt, w, y, opts, stream)
        with torch.cuda.stream(stream):
            for s in range(3):
                one(s)
            stream.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for s in range(n):
                one(s)
            b.record(stream)
            b.synchronize()
        rc, bits = moe.moe_read_status(w, stream)
        assert rc == moe.MOE_OK, f"device status {rc} bits {bits}"
        return a.elapsed_time(b) / n

    dev_ms = eager(moe.options(), ws)
    host_ms = eager(moe.options(host_routing=1), ws)
    uf = moe.options(unfused_dequant=1)
    ws_u = moe.workspace(shp, uf)
    uf_ms = eager(uf, ws_u)
    del ws_u
    tok_s = lambda ms: world * T / (ms / 1000.0)
    return dict(
        launch=f"eager moe_forward, {n} steps each (no CUDA graph)",
        default=dict(ms_per_step=dev_ms, value=tok_s(dev_ms)),
        host_routing=dict(what="counts to the host, scan and block map there, results back, then scatter "
                               "(one stream sync per step)",
                          ms_per_step=host_ms, value=tok_s(host_ms), slowdown=host_ms / dev_ms),
        unfused_dequant=dict(what="every expert's weights of a projection dequantised to bf16 in HBM by a separate "
                                  "kernel, then streamed by the same grouped GEMM",
                             ms_per_step=uf_ms, value=tok_s(uf_ms), slowdown=uf_ms / dev_ms))


# ------------------------------------------------------------------------------------- oracle
class OracleSampler:
    """Times the oracle (route + FFN + combine) on bounded token samples of a workload."""

    def __init__(self, wl):
        from moe_workload import configs
        self.wl = wl
        self.lay = configs.make_layer(wl)
        sh = wl.shape
        self.x_pool = configs.make_decode_x(wl, 64) if sh.T == 1 else configs.make_x(wl)[: (wl.chunk or sh.T)]

    def run(self, n_tokens: int, seed: int = 0):
        import oracle
        rng = np.random.default_rng(seed)
        pool = self.x_pool
        x = np.ascontiguousarray(pool[np.sort(rng.choice(pool.shape[0], min(n_tokens, pool.shape[0]), replace=False))])
        t0 = time.perf_counter()
        r = oracle.route(x, self.lay.w_router, self.lay.logit_bias)
        oracle.moe_tokens(x, r["topk_idx"], r["topk_w"], self.lay.routed, self.lay.shared)
        dt = time.perf_counter() - t0
        return x.shape[0], dt, oracle.num_threads()


def cpu_baseline(wl, n_tokens):
    n, dt, cores = OracleSampler(wl).run(n_tokens)
    if wl.shape.T == 1:
        return dict(value=dt * 1e6 / n, unit="us/token/layer", cores=cores, kind="oracle",
                    sample=f"{n} decode tokens through one layer")
    return dict(value=n / dt, unit="routed tokens/s", cores=cores, kind="oracle",
                sample=f"{n} of {wl.chunk or wl.shape.T} tokens of one chunk (routing of the sample + FFN + combine)")


def run_reference(args, rank, world):
    from moe_workload import configs
    wl = configs.WORKLOADS[args.workload]
    K = args.steps if args.steps is not None else 10
    # the same 32-token sample as the in-line CPU baseline, smaller when many steps are asked
    # for, so that the whole run stays within a few minutes
    n = 8 if wl.shape.T == 1 else int(min(32, max(4, 4 * (240 // (K + args.warmup)))))
    smp = OracleSampler(wl)
    for s in range(args.warmup):
        smp.run(n, seed=100 + s)
    tot, toks, cores = 0.0, 0, 1
    for s in range(K):
        m, dt, cores = smp.run(n, seed=s)
        tot += dt
        toks += m
    decode = wl.shape.T == 1
    if decode:
        value, unit, hib = tot * 1e6 / toks, "us/token/layer", False
    else:
        value, unit, hib = toks / tot, "routed tokens/s", True
    sample = f"{n} tokens per step through one layer (routing + FFN + combine)"
    return dict(impl="reference", metric=METRIC, value=value, unit=unit, n_gpus=world, steps=K, warmup=args.warmup,
                ms_per_step=tot * 1000.0 / K, higher_is_better=hib, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic",
                config=dict(workload=wl.name, T=wl.chunk or wl.shape.T, d=wl.shape.d, E=wl.shape.E, k=wl.shape.k,
                            I=wl.shape.I, I_shared=wl.shape.I_shared, parallelism="host cores"),
                cpu_baseline=dict(value=value, unit=unit, cores=cores, kind="oracle", sample=sample),
                e2e=dict(value=value, unit=unit, h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)))
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("gloo")
    res, wl = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_tokens if wl.shape.T != 1 else 16)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
