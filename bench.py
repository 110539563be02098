"""Benchmark of the GB300 sparse-MoE expert path (one JSON line on rank 0).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--extras LIST|none]
                [--impl ours|reference]

A step is one pass of the whole hot path (route -> grouped FFN -> combine) over one batch of
synthetic input of the workload.  Default (headline) workload: the skewed long prefill, 16,384
tokens in four chunks of 4096 (d=2048, 256 experts, top-8, I=512 + shared expert, Zipf(1.2)
router bias): a step is one chunk, the chunks taking turns; its 455 MB of 4-bit weights exceed
L2, so every step streams them from HBM (a workload whose layer fits in L2 rotates through
enough independent layer copies to exceed it).  The other workloads (the 4096- and 512-token
chunks, the tiny layer and batch-1 decode) follow as keys of the same line under "extra", each
with its own roofline, end-to-end number and oracle baseline (N=1 only).

Timing: W warm-up steps (the first runs eagerly, the rest as the timed steps run), then exactly
K steps between CUDA events on the launching stream, barrier + synchronize on both sides, max
over ranks.  Prefill steps replay from CUDA graphs of the library calls, 8 steps per graph; the
first step of every 4th block of 8 runs phase by phase (one graph per phase, events in between),
which gives the per-kernel times of the roofline, and the rest of that block, like a last
partial block, runs one graph per step.  Without
--steps, K is chosen for about 1.5 s of timed work (the calibration steps count as warm-up).
Multi-GPU (torchrun): every rank runs its own rotation of the chunks (weak scaling, no
collective on the data path).

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
DEFAULT_WORKLOAD = "skew_t16384_d2048"
EXTRA_WORKLOADS = ("prefill_t4096_d2048", "prefill_t512_d2048", "tiny_t128_d512", "decode_t1_d2048")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--extras", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads reported under 'extra' (N=1 only), or 'none'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ablations", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode: layer copies (default: the workload's); fewer for small profiling captures")
    ap.add_argument("--cpu-sample-tokens", type=int, default=32)
    args = ap.parse_args()
    args.ablations = not args.no_ablations
    args.extra_list = [] if args.extras in ("", "none") else [w for w in args.extras.split(",") if w != args.workload]
    return args


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
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of each of a
# workload's kernels, from an ncu full capture of the current kernels (profiles/ncu_*.md):
# {workload: {kernel: bytes}}.  A kernel that is not listed reports null.
TRAFFIC_BYTES = {
    "skew_t16384_d2048": {"gate_up": 177.104384e6 + 47.760896e6, "down": 122.410752e6 + 3.363584e6},
    "prefill_t4096_d2048": {"gate_up": 454.290432e6 + 62.292992e6, "down": 276.466176e6 + 27.593728e6},
    "prefill_t512_d2048": {"gate_up": 322.247936e6 + 10.189056e6, "down": 165.381632e6 + 3.507968e6},
    "decode_t1_d2048": {"decode": 17.078528e6},
}


def algorithmic_counts(shp, counts):
    """Per-launch algorithmic bytes and FLOPs of the gate/up and down kernels (real rows only):
    the 4-bit weights of the experts that have rows (plus the shared expert), the activation
    rows read once, h (bf16) written once and read once, the fp32 output written once."""
    T, d, I = shp.T, shp.d, shp.I
    touched = int((counts > 0).sum()) + 1                       # + the shared expert
    q4 = lambda rows, cols: rows * cols // 2 + rows * (cols // 64) * 4   # codes + bf16 scale/bias
    gu_w = touched * 2 * q4(I, d)
    dn_w = touched * q4(d, I)
    rows = 9 * T                                                # routed assignments + shared rows
    gu_bytes = gu_w + rows * d * 2 + rows * I * 2               # weights + activation rows + h
    dn_bytes = dn_w + rows * I * 2 + T * d * 4                  # weights + h + fp32 weighted sum
    gu_flops = 2.0 * rows * d * 2 * I
    dn_flops = 2.0 * rows * I * d
    return dict(gu_bytes=gu_bytes, dn_bytes=dn_bytes, gu_flops=gu_flops, dn_flops=dn_flops,
                weights_bytes=gu_w + dn_w, touched=touched)


def step_plan(n, multi, probe_every=None):
    """How n consecutive steps run: blocks of `multi` steps replay one graph ("multi"); the first
    step of every probe_every-th block runs phase by phase with events in between ("probe") and
    the rest of that block step by step ("single", one graph per step), as does a last partial
    block.  Entries: (kind, first step)."""
    ops, s, b = [], 0, 0
    while s < n:
        m = min(multi, n - s)
        if probe_every and b % probe_every == 0:
            ops += [("probe", s)] + [("single", s + j) for j in range(1, m)]
        elif m == multi:
            ops.append(("multi", s))
        else:
            ops += [("single", s + j) for j in range(m)]
        s += m
        b += 1
    return ops


def roofline_entry(kernel, P, work, ms, unit_kind, long_region, traffic):
    """achieved = algorithmic work per launch / measured launch time; frac against the measured
    peak (bf16: the sustained figure when the timed region is long, else the burst one)."""
    if unit_kind == "hbm":
        ach = work / (ms * 1e-3) / 1e9
        return dict(bound="hbm", achieved=ach, peak=P["hbm_gbs"], unit="GB/s", frac=ach / P["hbm_gbs"],
                    traffic=traffic, kernel=kernel, algorithmic_bytes=work, kernel_ms=ms, peak_source=P["source"])
    ach = work / (ms * 1e-3) / 1e12
    peak = P["bf16_tflops_sustained"] if long_region else P["bf16_tflops"]
    return dict(bound="tensor", achieved=ach, peak=peak, unit="TFLOP/s", frac=ach / peak,
                frac_burst=ach / P["bf16_tflops"], frac_sustained=ach / P["bf16_tflops_sustained"],
                peak_kind="sustained" if long_region else "burst", traffic=traffic, kernel=kernel,
                algorithmic_flops=work, kernel_ms=ms, peak_source=P["source"])


def run_ours(wname, args, rank, world, local, headline=True):
    import torch
    import quantized_grouped_gemm_gb300 as moe
    from moe_workload import configs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = configs.WORKLOADS[wname]
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
    if decode:
        nsteps_x = 1000
        x_all = to_dev(configs.make_decode_x(wl, nsteps_x))
        xs = None
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
    W = max(1, args.warmup)
    PROBE = 4      # the first step of every 4th block of MULTI steps is timed phase by phase

    # ---- warm-up step 1 runs eagerly (the library's one-time set-up: kernel attributes, the
    # one-launch decode kernel's occupancy check); then the graphs are captured
    with torch.cuda.stream(stream):
        if decode:
            for li in range(layers):
                moe.moe_forward(shp, x_in, L[li]["wr"], L[li]["bias"], L[li]["pr"], L[li]["ps"], rt, ws, y, opts,
                                stream)
            stream.synchronize()
            n0 = moe.moe_launch_count()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for li in range(layers):
                    moe.moe_forward(shp, x_in, L[li]["wr"], L[li]["bias"], L[li]["pr"], L[li]["ps"], rt, ws, y, opts,
                                    stream)
            launches_per_step = moe.moe_launch_count() - n0
            MULTI = 1
        else:
            # step s runs layer copy s % layers on resident chunk s % chunks, reading it in place
            def calls_for(lw, xc):
                return [lambda: moe.moe_route(shp, xc, lw["wr"], lw["bias"], rt, ws, opts, stream),
                        lambda: moe.moe_ffn_gate_up(shp, xc, rt, lw["pr"], lw["ps"], ws, opts, stream),
                        lambda: moe.moe_ffn_down(shp, rt, lw["pr"], lw["ps"], ws, opts, stream),
                        lambda: moe.moe_combine(shp, rt, ws, y, opts, stream)]
            nsets = int(np.lcm(layers, len(xs)))
            for f in calls_for(L[0], xs[0]):
                f()
            stream.synchronize()
            # per set: the four phases as separate graphs (probe steps run these with events in
            # between, for the kernel times), the whole step as one graph, and MULTI consecutive
            # steps (a multiple of the set count) as one graph; inside a graph consecutive
            # kernels, also across steps, overlap their prologues through programmatic dependent
            # launch
            graphs, step_graphs = [], []
            for gi in range(nsets):
                n0 = moe.moe_launch_count()
                gc = []
                calls = calls_for(L[gi % layers], xs[gi % len(xs)])
                for f in calls:
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        f()
                    gc.append(g)
                if gi == 0:
                    launches_per_step = moe.moe_launch_count() - n0
                graphs.append(gc)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for f in calls:
                        f()
                step_graphs.append(g)
            MULTI = nsets * -(-8 // nsets)
            multi = torch.cuda.CUDAGraph()
            with torch.cuda.graph(multi, stream=stream):
                for s in range(MULTI):
                    for f in calls_for(L[s % layers], xs[s % len(xs)]):
                        f()
    torch.cuda.synchronize()

    probes = []   # per probe step: [route, gate/up, down, combine] ms

    def run(n, with_probes, keep=True):
        for kind, s in step_plan(n, MULTI, PROBE if with_probes else None):
            if decode:
                x_in.copy_(x_all[s % nsteps_x:s % nsteps_x + 1], non_blocking=True)
                g.replay()
            elif kind == "multi":
                multi.replay()
            elif kind == "single":
                step_graphs[s % len(step_graphs)].replay()
            else:
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
                ev[0].record(stream)
                for i, gph in enumerate(graphs[s % len(graphs)]):
                    gph.replay()
                    ev[i + 1].record(stream)
                if keep:
                    probes.append(ev)

    dist = None
    if world > 1:
        import torch.distributed as dist
    with torch.cuda.stream(stream):
        run(W - 1, True, keep=False)   # the same mix of graphs as the timed steps
        stream.synchronize()
        warmup_steps = W
        if args.steps is None:       # auto: about 1.5 s of timed work (these steps count as warm-up)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = max(MULTI, 24 // MULTI * MULTI)
            e0.record(stream)
            run(n, False)
            e1.record(stream)
            e1.synchronize()
            per = e0.elapsed_time(e1) / n
            warmup_steps += n
            K = int(min(20000, max(20, 1500.0 / max(per, 1e-3))))
        else:
            K = max(1, args.steps)
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.15)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        run(K, True)
        t1.record(stream)
        t1.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        clk = clocks.stop()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist)
    ms_step = ms_total / K
    long_region = ms_total > 1000.0
    rc, bits = moe.moe_read_status(ws, stream)
    assert rc == moe.MOE_OK, f"device status {rc} bits {bits}"

    P = peaks()
    res = dict(metric=METRIC, n_gpus=world, steps=K, warmup=warmup_steps, ms_per_step=ms_step, data="synthetic",
               scaling="weak", vs_baseline=None, dtype="bf16", clocks=clk, gpu_launches=int(launches_per_step * K))
    traffic = TRAFFIC_BYTES.get(wl.name, {})
    if decode:
        us_tok_layer = ms_step * 1000.0 / layers
        res.update(value=us_tok_layer, unit="us/token/layer", higher_is_better=False)
        # router weight (bf16) + gate, up, down of 8 routed + 1 shared expert (4-bit + bf16 scale/bias per 64)
        bytes_layer = sh.E * sh.d * 2 + 9 * (3 * sh.d * sh.I // 2 + 3 * sh.d * sh.I // 64 * 4)
        res["roofline"] = roofline_entry("decode_fused (one launch per layer: route + gate/up + down + combine)", P,
                                         bytes_layer, us_tok_layer * 1e-3, "hbm", long_region,
                                         traffic.get("decode"))
        res["roofline"]["bytes_per_token_layer"] = bytes_layer
        res["config"] = dict(workload=wl.name, T=1, d=sh.d, E=sh.E, k=sh.k, I=sh.I, I_shared=sh.I_shared,
                             layers=layers, l2=f"inputs larger than L2: {layers} layer copies of the weights, "
                                                 f"{layers * layer_bytes / 1e9:.0f} GB",
                             parallelism=f"replicas x{world}")
    else:
        value = world * T * K / (ms_total / 1000.0)
        res.update(value=value, unit="routed tokens/s", higher_is_better=True)
        ph = np.array([[ev[i].elapsed_time(ev[i + 1]) for i in range(4)] for ev in probes])
        route_ms, gu_ms, dn_ms, comb_ms = (float(v) for v in ph.mean(axis=0))
        counts = rt.counts.cpu().numpy()
        A = algorithmic_counts(shp, counts)
        ridge = P["bf16_tflops"] * 1e12 / (P["hbm_gbs"] * 1e9)
        # dominant kernel: the slower of the two FFN kernels; HBM-bound below the ridge point
        down_dom = dn_ms > gu_ms
        name = ("ffn_tm_kernel<1,0> (down projection + weighted sum; tcgen05, dequantised weights in TMEM)"
                if down_dom else "ffn_tm_kernel<0,0> (gate/up + SwiGLU; tcgen05, dequantised weights in TMEM)")
        flops, byts, kms = (A["dn_flops"], A["dn_bytes"], dn_ms) if down_dom else (A["gu_flops"], A["gu_bytes"], gu_ms)
        hbm = flops / byts < ridge
        tr = traffic.get("down" if down_dom else "gate_up")
        res["roofline"] = roofline_entry(name, P, byts if hbm else flops, kms, "hbm" if hbm else "tensor",
                                         long_region, tr)
        ffn_ms = gu_ms + dn_ms
        ffn_tf = (A["gu_flops"] + A["dn_flops"]) / (ffn_ms * 1e-3) / 1e12
        res["ffn"] = dict(
            route_ms=route_ms, gate_up_ms=gu_ms, down_ms=dn_ms, combine_ms=comb_ms, probe_steps=len(probes),
            gate_up=roofline_entry("gate/up", P, A["gu_flops"], gu_ms, "tensor", long_region, None),
            down=roofline_entry("down", P, A["dn_flops"], dn_ms, "tensor", long_region, None),
            gate_up_hbm=roofline_entry("gate/up", P, A["gu_bytes"], gu_ms, "hbm", long_region, None),
            down_hbm=roofline_entry("down", P, A["dn_bytes"], dn_ms, "hbm", long_region, None),
            ffn_tflops=ffn_tf, ffn_frac_bf16_burst=ffn_tf / P["bf16_tflops"],
            ffn_frac_bf16_sustained=ffn_tf / P["bf16_tflops_sustained"],
            ffn_weight_gbs=A["weights_bytes"] / (ffn_ms * 1e-3) / 1e9, experts_touched=A["touched"],
            other_ms=ms_step - ffn_ms)
        for key in ("gate_up", "down", "gate_up_hbm", "down_hbm"):
            for drop in ("kernel", "traffic", "peak_source"):
                res["ffn"][key].pop(drop, None)
        res["config"] = dict(workload=wl.name, T=T, d=sh.d, E=sh.E, k=sh.k, I=sh.I, I_shared=sh.I_shared,
                             chunks=sh.T // T, layers=layers,
                             l2=f"inputs larger than L2: {layers} layer cop{'y' if layers == 1 else 'ies'} of "
                                f"{layer_bytes / 1e6:.0f} MB of 4-bit weights, a step reads one",
                             parallelism=f"replicas x{world}")

    res["e2e"] = e2e(moe, torch, shp, sh, T, K, L, layers, xs, rt, ws, y, x_in, stream, dev, decode,
                     g if decode else None, world, wl)
    if not decode and args.ablations and world == 1:
        res["ablations"] = ablations(moe, shp, L, layers, xs, rt, ws, y, stream, T, world, wl.name)
    del L, xs, rt, ws, y, x_in
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, wl


def e2e(moe, torch, shp, sh, T, K, L, layers, xs, rt, ws, y, x_in, stream, dev, decode, graph, world, wl):
    """The same metric through the public API with host buffers: every step copies its input from
    pinned host memory and its output back, inside the timed region."""
    if decode:
        from moe_workload import configs
        xh = configs.make_decode_x(wl, 16)
        xh_t = torch.from_numpy(xh.view(np.int16)).pin_memory()
        yh = torch.empty(1, sh.d, dtype=torch.int16).pin_memory()
        layers_n = layers
        with torch.cuda.stream(stream):
            def e2e_step(s):
                x_in.copy_(xh_t[s % 16:s % 16 + 1], non_blocking=True)
                graph.replay()
                yh.copy_(y, non_blocking=True)
            for s in range(3):
                e2e_step(s)
            stream.synchronize()
            Ke = min(K, 1000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for s in range(Ke):
                e2e_step(s)
            b.record(stream)
            b.synchronize()
        e_ms = a.elapsed_time(b)
        return dict(value=e_ms * 1000.0 / Ke / layers_n, unit="us/token/layer", h2d_bytes_per_step=sh.d * 2,
                    d2h_bytes_per_step=sh.d * 2, steps=Ke,
                    copies="4 KB in and out per token, in order on the compute stream (pinned host buffers)")
    # Prefill: every step copies its chunk in from pinned host memory, runs moe_forward and copies
    # its output back.  The copies run on a copy stream into two device buffers, so the input of
    # step s+1 and the output of step s-1 move while step s computes (consecutive steps share the
    # workspace and run in order on `stream`).
    opts = moe.options()
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
    return dict(value=world * T * Ke / (e_ms / 1000.0), unit="routed tokens/s", h2d_bytes_per_step=T * sh.d * 2,
                d2h_bytes_per_step=T * sh.d * 2, steps=Ke,
                copies="pinned host buffers; copy stream overlapped with compute, two buffers")


def ablations(moe, shp, L, layers, xs, rt, ws, y, stream, T, world, wname, n=50):
    """Outside the timed region: the step launched eagerly through moe_forward with the default
    design and with variants of it -- the largest token block of the grouped GEMMs
    (moe_options.gemm_rows, the pages' tile-size choice), and for the 512-token chunk the two
    mechanisms the pages measure: the host round trip of the routing counts
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

    tok_s = lambda ms: world * T / (ms / 1000.0)
    dev_ms = eager(moe.options(), ws)
    out = dict(launch=f"eager moe_forward, {n} steps each (no CUDA graph)",
               default=dict(ms_per_step=dev_ms, value=tok_s(dev_ms)))
    rows = {}
    for r in (16, 32, 64, 128):
        ms = eager(moe.options(gemm_rows=r), ws)
        rows[str(r)] = dict(ms_per_step=ms, value=tok_s(ms), vs_default=ms / dev_ms)
    out["gemm_rows"] = dict(what="largest token block of the grouped GEMMs (moe_options.gemm_rows; default 128)",
                            **rows)
    if wname == "prefill_t512_d2048":
        host_ms = eager(moe.options(host_routing=1), ws)
        uf = moe.options(unfused_dequant=1)
        ws_u = moe.workspace(shp, uf)
        uf_ms = eager(uf, ws_u)
        del ws_u
        out["host_routing"] = dict(what="counts to the host, scan and block map there, results back, then scatter "
                                        "(one stream sync per step)",
                                   ms_per_step=host_ms, value=tok_s(host_ms), slowdown=host_ms / dev_ms)
        out["unfused_dequant"] = dict(what="every expert's weights of a projection dequantised to bf16 in HBM by a "
                                           "separate kernel, then streamed by the same grouped GEMM",
                                      ms_per_step=uf_ms, value=tok_s(uf_ms), slowdown=uf_ms / dev_ms)
    return out


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
    res, wl = run_ours(args.workload, args, rank, world, local)
    if rank == 0 and world == 1:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_tokens if wl.shape.T != 1 else 16)
        extra = {}
        for name in args.extra_list:
            r, w2 = run_ours(name, args, rank, world, local, headline=False)
            if not args.no_cpu_baseline:
                r["cpu_baseline"] = cpu_baseline(w2, args.cpu_sample_tokens if w2.shape.T != 1 else 16)
            for key in ("metric", "n_gpus", "data", "scaling", "vs_baseline", "dtype"):
                r.pop(key, None)
            extra[name] = r
        if extra:
            res["extra"] = extra
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
