"""Benchmark: routed MoE layer stack on GB300 (libmoe) or the CPU oracle.

Default workload: the Gemma-4-26B-A4B-shaped stack (30 MoE layers, d=2816, E=128, top-8,
f=704, SwiGLU, Q8_0 experts, bf16 activations), decode, one token per step.  A step is one
pass of the whole hot path over every layer of the stack: router, top-k, permutation,
gate.up + SwiGLU, sparse down, combine, and the RMS-norm glue that feeds the next layer.
The 30 layers are captured once into CUDA graphs; weights, inputs and workspaces are
resident in HBM before timing starts.

One JSON line on rank 0:  metric / value / unit (tokens per second through the stack), the
roofline of the dominant kernel (gate.up, live CUDA-event timing inside the graphs against
the measured HBM copy bandwidth), the oracle timed on the host cores (cpu_baseline), an
end-to-end figure with host<->device copies inside the timed region, clocks sampled during
the timed region and the number of libmoe kernels launched.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gemma|nemotron|minimax|zipf|zipf_nvfp4] [--tokens T] [--no-secondary]
The default run adds a "secondary" list to the line: Gemma-shaped prefill (T = 512) on the
headline stack's weights, the 40-layer Nemotron-shaped NVFP4 stack at one token, and
MiniMax-shaped prefill (T = 4096, 8 layers), each with its own config, roofline and oracle
baseline (a shorter sample).
The zipf workloads are the skewed-routing sweep on the Gemma layer shape (Q8_0 or NVFP4
experts): the routing is supplied (each token draws k distinct experts with probability
proportional to rank^-1.1), so the router is skipped, and a stack of 4 layers with their
own weights keeps the routed experts of one step out of L2 at the next.
Under torchrun (N > 1) every rank runs its own replica (the layer needs no exchange on
one GPU); value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode active-expert GB/s vs GB300 HBM roofline"
N_ROTATE = 8          # distinct token inputs, replayed round robin (no step reuses the last one's experts)
ZIPF_LAYERS = 4       # layers of the supplied-routing sweep's stack (4 x 50 MB of routed experts at T=1 > L2)


def routed(w) -> bool:
    """The workload supplies its routing (the Zipf sweep) instead of running the router."""
    return w.name.startswith("zipf")


def default_layers(w) -> int:
    return ZIPF_LAYERS if routed(w) else w.layers


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemma")
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0, help="override the stack depth (0 = the workload's)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (0 = the workload's): small cases of a shape for profiling")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-weights", choices=["none", "down", "all"], default="none",
                    help="expert stacks in page-locked host memory, read in place (NVLink-C2C on GB300): "
                         "the down stack, or both")
    ap.add_argument("--act-quant", choices=["none", "q8_0"], default="none",
                    help="q8_0: the activation-quantised expert path (Q8_0 weights only)")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false",
                    help="time only the headline workload (the default run also times the SECONDARY list)")
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device="cuda") -> float:
    """The largest of every rank's value, returned on all ranks (the job's time is its
    slowest replica's); the value itself when there is one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms / 1e3)


def host_link_peak():
    """GB/s of a 2 GiB page-locked host -> device copy (best of 3, CUDA events): the host link's
    read rate (NVLink-C2C on GB300), the bound of weights read in place from host memory."""
    import torch
    n = 2 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, n / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return round(best, 1), "measured in this run: page-locked host -> device copy of 2 GiB (best of 3)"


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def hbm_peak():
    p = peaks()
    if p and p.get("hbm_gbs"):
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def workload_config(w, T, layers, act_quant="none"):
    return {
        "workload": f"{w.name}-shaped MoE stack: {layers} layers, d={w.d}, E={w.E}, top-{w.k}, f={w.f}, "
                    f"{'SwiGLU' if w.act == 'swiglu' else 'ReLU^2'}, {w.wfmt.upper()} experts, "
                    f"{w.x_dtype} activations{', Q8_0-coded expert inputs' if act_quant == 'q8_0' else ''}, "
                    f"{'decode' if T <= 32 else 'prefill'} T={T}",
        "act_quant": act_quant,
        "layers": layers, "tokens_per_step": T, "d": w.d, "E": w.E, "k": w.k, "f": w.f, "act": w.act,
        "weights": w.wfmt, "activations": w.x_dtype,
        **({"routing": "supplied (router skipped): k distinct experts per token drawn with probability "
                       "proportional to rank^-1.1 over a seeded permutation of the experts; weights a softmax of "
                       "seeded normals; one draw per rotated input, the same for every layer"} if routed(w) else {}),
    }


# ====================================================================== oracle timing
def oracle_sample(w, T, layers, max_units, time_budget_s, warmup_units=0, cache=None, with_unit_time=False,
                  act_q8=False):
    """Time the CPU oracle on a bounded sample of the workload.

    A unit is the oracle's forward of one layer of the stack (router, top-k, softmax,
    permutation, every routed expert: dequantise + gate.up + activation + down, combine;
    fp64) on up to 8 of the step's tokens.  Units cycle through the stack's layers; the
    experts a layer routes to are drawn and quantised once (untimed) and cached (in `cache`
    when given, so that a second sample reuses them).
    Returns (seconds per stack step, units timed, threads, description)."""
    import numpy as np
    import torch

    import oracle
    from quantized_routed_expert_softmax_gb300 import synth

    have_cuda = torch.cuda.is_available()
    act = oracle.ACT_SWIGLU if w.act == "swiglu" else oracle.ACT_RELU2
    fmt = {"q8_0": oracle.W_Q8_0, "nvfp4": oracle.W_NVFP4, "int8pc": oracle.W_INT8PC}[w.wfmt]
    tu = min(T, 8)
    cache = {} if cache is None else cache

    def layer_obj(layer):
        if layer in cache:
            return cache[layer]
        x = synth.tokens(w, tu, layer, tag="cpu")
        W = synth.router_weight(w, layer)
        if routed(w):
            idx, wts = synth.zipf_routing(tu, w.E, w.k, seed_tag=f"cpu{layer}")
        else:
            idx, wts = oracle.topk_softmax(oracle.router_logits(x, W), w.k)[0], None
        gu, dn = [None] * w.E, [None] * w.E
        gts, dts = np.ones(w.E, np.float32), np.ones(w.E, np.float32)
        for e in sorted(set(int(v) for v in idx.ravel())):
            if have_cuda:
                a = synth.expert_stack_cuda(w, layer, "gate_up", [e])[0].cpu().numpy()
                b = synth.expert_stack_cuda(w, layer, "down", [e])[0].cpu().numpy()
            else:
                a, b = synth.expert_weights(w, layer, e)
            if w.wfmt == "q8_0":
                gu[e], dn[e] = oracle.q8_0_quantize(a), oracle.q8_0_quantize(b)
            elif w.wfmt == "int8pc":
                gu[e], dn[e] = oracle.int8pc_quantize(a), oracle.int8pc_quantize(b)
            else:
                gu[e], gts[e] = oracle.nvfp4_quantize(a)
                dn[e], dts[e] = oracle.nvfp4_quantize(b)
        L = oracle.Layer(w.d, w.f, w.E, w.k, act, fmt, W, gu, dn,
                         gts if w.wfmt == "nvfp4" else None, dts if w.wfmt == "nvfp4" else None)
        cache[layer] = (L, x, (idx, wts) if routed(w) else (None, None))
        return cache[layer]

    times = []
    units = 0
    spent = 0.0
    while units < max_units + warmup_units and (spent < time_budget_s or units < warmup_units + 1):
        L, x, (ii, ww) = layer_obj(units % layers)
        t0 = time.perf_counter()
        L.forward(x, idx_in=ii, w_in=ww, act_q8=act_q8)
        dt = time.perf_counter() - t0
        if units >= warmup_units:
            times.append(dt)
            spent += dt
        units += 1
    per_token_layer = statistics.mean(times) / tu
    step_s = per_token_layer * T * layers
    what = ("supplied routing, permutation" if routed(w) else "router, top-k, softmax, permutation")
    desc = (f"{len(times)} oracle forwards of single layers of the stack on {tu} token(s) each ({what}, every "
            f"routed expert dequantised and evaluated in fp64, combine), cycling over the {layers} layers; "
            f"per-step time = mean per token-layer x {T} token(s) x {layers} layers")
    if with_unit_time:
        return step_s, len(times), oracle.num_threads(), desc, statistics.mean(times)
    return step_s, len(times), oracle.num_threads(), desc


def single_core_baseline(w, T, layers, threads_all, cache, budget_s=8.0):
    """The same oracle sample on one thread (about budget_s of timed work), then the oracle's
    thread count restored.  A failure here is recorded, never raised: the bench line stands."""
    import oracle
    try:
        oracle.set_num_threads(1)
        step_s, n, _, _ = oracle_sample(w, T, layers, max_units=4 * layers, time_budget_s=budget_s, warmup_units=1,
                                        cache=cache)
        return {"value": round(T / step_s, 6), "cores": 1, "units_timed": n}
    except Exception as exc:
        return {"error": f"{type(exc).__name__}: {exc}"}
    finally:
        try:
            oracle.set_num_threads(threads_all)
        except Exception:
            pass


# ====================================================================== GPU arm
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = str(gpu_index)
        try:
            import torch
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        except Exception:
            pass
        self.proc = None
        # the samples only feed the summary in the JSON line: a scratch file suffices
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}_rank{gpu_index}.csv")
        self.fh = None

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def build_stack(w, T, layers, local_rank, host_weights="none"):
    import torch

    from quantized_routed_expert_softmax_gb300 import layers as L
    from quantized_routed_expert_softmax_gb300 import synth
    stack = [L.build_layer(w, layer=l, host_weights=host_weights) for l in range(layers)]
    for l, layer in enumerate(stack):   # each layer warms L2 with the next one's router weights
        layer.set_l2_prefetch(stack[(l + 1) % layers].router_w)
    inputs = [synth.tokens_cuda(w, T, layer=0, tag=f"bench{r}") for r in range(N_ROTATE)]
    torch.cuda.synchronize()
    return stack, inputs


def build_routings(w, T):
    """Supplied routing per rotated input (device idx [T,k] int32, w [T,k] fp32), or None
    when the stack routes itself."""
    import torch

    from quantized_routed_expert_softmax_gb300 import synth
    if not routed(w):
        return None
    out = []
    for r in range(N_ROTATE):
        idx, wts = synth.zipf_routing(T, w.E, w.k, seed_tag=f"bench{r}")
        out.append((torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda()))
    return out


def capture_graphs(stack, inputs, T, w, stage_events=None, stack_obj=None, routings=None):
    """One CUDA graph per rotated input; each runs the whole stack (with stack_obj: one
    moe_stack_forward call; stage_events then holds two events per input, around it).
    routings: supplied (idx, w) per rotated input, given to every layer."""
    import torch

    from quantized_routed_expert_softmax_gb300 import native
    dev = torch.device("cuda")
    if stack_obj is not None:
        outs_all = torch.empty((len(stack), w.d), dtype=torch.float32, device=dev)
        ws = stack_obj.workspace()
        graphs = []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            stack_obj.forward(inputs[0], outs=outs_all, workspace=ws)   # warm outside capture
            torch.cuda.current_stream().synchronize()
            for g_i, x0 in enumerate(inputs):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    ev = None if stage_events is None else stage_events[g_i]
                    if ev is not None:
                        ev[0].record()
                    stack_obj.forward(x0, outs=outs_all, workspace=ws)
                    if ev is not None:
                        ev[1].record()
                graphs.append(g)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        return graphs, [outs_all[l:l + 1] for l in range(len(stack))]
    outs = [torch.empty((T, w.d), dtype=torch.float32, device=dev) for _ in stack]
    nxt = [torch.empty((T, w.d), dtype=torch.bfloat16, device=dev) for _ in stack]
    wss = [layer.workspace(T) for layer in stack]
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # warm the kernels once outside capture (per-device attribute setup happens here)
        x = inputs[0]
        ri, rw = routings[0] if routings else (None, None)
        for li, layer in enumerate(stack):
            layer.forward(x, idx_in=ri, w_in=rw, out=outs[li], workspace=wss[li])
            native.rmsnorm_bf16(outs[li], out=nxt[li])
            x = nxt[li]
        torch.cuda.current_stream().synchronize()
        for g_i, x0 in enumerate(inputs):
            g = torch.cuda.CUDAGraph()
            ri, rw = routings[g_i] if routings else (None, None)
            with torch.cuda.graph(g, stream=s):
                x = x0
                for li, layer in enumerate(stack):
                    ev = None if stage_events is None else stage_events[g_i][li]
                    layer.forward(x, idx_in=ri, w_in=rw, out=outs[li], workspace=wss[li], stage_events=ev)
                    native.rmsnorm_bf16(outs[li], out=nxt[li])
                    x = nxt[li]
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return graphs, outs


def run_ours(args, rank, world, local_rank, prebuilt=None):
    """Time one workload (args.workload, args.tokens, args.layers) for args.steps steps.
    prebuilt: layers of the same workload built earlier (a secondary line reuses the headline
    stack's weights with other token inputs).  Returns (JSON object on rank 0, (w, T, layers),
    the layers)."""
    import torch
    import torch.distributed as dist

    from quantized_routed_expert_softmax_gb300 import native, synth
    from quantized_routed_expert_softmax_gb300 import build as B
    B.build()
    torch.cuda.set_device(local_rank)
    w = synth.WORKLOADS[args.workload]
    if getattr(args, "experts", 0):
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}_e{args.experts}", E=args.experts)
    T = args.tokens
    layers = args.layers or default_layers(w)
    if prebuilt is not None and len(prebuilt) == layers:
        stack = prebuilt
        inputs = [synth.tokens_cuda(w, T, layer=0, tag=f"bench{r}") for r in range(N_ROTATE)]
        torch.cuda.synchronize()
    else:
        stack, inputs = build_stack(w, T, layers, local_rank, host_weights=getattr(args, "host_weights", "none"))
    aq = getattr(args, "act_quant", "none")
    for layer in stack:   # the activation-quantised path is a flag of the same weights
        layer.desc.act_quant = native.ACT_QUANT[aq]
    routings = build_routings(w, T)
    supplied = routings is not None
    # One token on layers the library runs as one kernel per layer: the whole stack as ONE
    # kernel (moe_stack_forward), the RMS-norm between layers inside it.
    stack_obj = native.MoEStack(stack) if T == 1 and not supplied else None
    if stack_obj is not None and stack_obj.launches() != 1:
        stack_obj = None
    graphs, outs = capture_graphs(stack, inputs, T, w, stack_obj=stack_obj, routings=routings)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- headline: K graph replays, round robin over the rotated inputs
    for i in range(args.warmup):
        graphs[i % N_ROTATE].replay()
    barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.15)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        graphs[i % N_ROTATE].replay()
    e1.record()
    barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    ms_step = ms_total / args.steps
    tokens_per_s = job_throughput(T * args.steps, world, ms_total)

    # ---- active-expert bytes of one step (from the routing the stack actually took)
    tr_bytes = active_expert_bytes(stack, inputs, T, w, routings)

    # ---- dominant kernel (gate.up): live CUDA events recorded inside the graphs
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in stack] for _ in inputs]
    for g in evs:
        for lay in g:
            for ev in lay:
                ev.record()
    torch.cuda.synchronize()
    n_ev_steps = max(N_ROTATE, min(args.steps, 400))
    gu_ms, dn_ms, rt_ms, cb_ms = [], [], [], []
    timing_how = "CUDA events recorded as graph nodes at the stage boundaries of every layer"
    if stack_obj is not None:   # one kernel per step: events around it
        try:   # events that are real record nodes under capture
            sev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)] for _ in inputs]
        except TypeError:
            sev = None
        if sev is not None:
            timing_how = "CUDA events recorded as graph nodes around the one-kernel stack"
            for pair in sev:
                for ev in pair:
                    ev.record()
            torch.cuda.synchronize()
            graphs_ev, _ = capture_graphs(stack, inputs, T, w, stage_events=sev, stack_obj=stack_obj)
            for i in range(args.warmup):
                graphs_ev[i % N_ROTATE].replay()
            torch.cuda.synchronize()
            for i in range(n_ev_steps):
                graphs_ev[i % N_ROTATE].replay()
                if i % N_ROTATE == N_ROTATE - 1:
                    torch.cuda.synchronize()
                    rt_ms.extend(pair[0].elapsed_time(pair[1]) for pair in sev)
        else:   # this torch cannot record external events under capture: time eager launches
            timing_how = "CUDA events around eager launches of the one-kernel stack"
            e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            outs_e = torch.empty((layers, w.d), dtype=torch.float32, device="cuda")
            for i in range(max(args.warmup, 3)):
                stack_obj.forward(inputs[i % N_ROTATE], outs=outs_e)
            for i in range(n_ev_steps):
                e_a.record()
                stack_obj.forward(inputs[i % N_ROTATE], outs=outs_e)
                e_b.record()
                e_b.synchronize()
                rt_ms.append(e_a.elapsed_time(e_b))
        torch.cuda.synchronize()
    try:
        if stack_obj is not None:
            raise StopIteration
        graphs_ev, _ = capture_graphs(stack, inputs, T, w, stage_events=evs, routings=routings)
        for i in range(args.warmup):
            graphs_ev[i % N_ROTATE].replay()
        torch.cuda.synchronize()
        for i in range(n_ev_steps):
            graphs_ev[i % N_ROTATE].replay()
        torch.cuda.synchronize()
        for g in evs:
            for lay in g:
                rt_ms.append(lay[0].elapsed_time(lay[1]))
                gu_ms.append(lay[1].elapsed_time(lay[2]))
                dn_ms.append(lay[2].elapsed_time(lay[3]))
                cb_ms.append(lay[3].elapsed_time(lay[4]))
    except StopIteration:
        pass
    except Exception as exc:   # graph event nodes refused: time the same launches eagerly
        timing_how = f"CUDA events around eager launches of the stack (graph events unavailable: {exc})"
        gu_ms, dn_ms, rt_ms, cb_ms = [], [], [], []
        outs_e = [torch.empty((T, w.d), dtype=torch.float32, device="cuda") for _ in stack]
        for r in range(N_ROTATE):
            x = inputs[r]
            ri, rw = routings[r] if routings else (None, None)
            for li, layer in enumerate(stack):
                lay = evs[r][li]
                layer.forward(x, idx_in=ri, w_in=rw, out=outs_e[li], workspace=layer.workspace(T), stage_events=lay)
                x = native.rmsnorm_bf16(outs_e[li])
            torch.cuda.synchronize()
            for lay in evs[r]:
                rt_ms.append(lay[0].elapsed_time(lay[1]))
                gu_ms.append(lay[1].elapsed_time(lay[2]))
                dn_ms.append(lay[2].elapsed_time(lay[3]))
                cb_ms.append(lay[3].elapsed_time(lay[4]))
    # One token on the one-kernel formats runs as ONE kernel per layer (the library reports one
    # launch): then that kernel is the one measured, between the first two boundaries (the
    # later boundaries coincide with the second), with all the layer's bytes as its work.
    one_kernel = stack[0].launches(T, supplied) == 1
    peak, peak_src = hbm_peak()
    host_w = getattr(args, "host_weights", "none")
    host_w = None if host_w in (False, None, "none") else host_w
    if host_w == "all":   # every weight byte crosses the host link: its measured copy rate is the bound
        peak, peak_src = host_link_peak()
    elif host_w == "down":   # gate.up (and the router) from HBM, then the down bytes over the link
        link, link_src = host_link_peak()
        per_layer = tr_bytes["layer_per_launch"]
        dn_b = tr_bytes["step"] / layers - tr_bytes["gate_up_per_layer"]
        t_bound = (per_layer - dn_b) / (peak * 1e9) + dn_b / (link * 1e9)
        peak_src = (f"derived: the layer's HBM bytes at {peak} GB/s, then its down bytes at the host link's "
                    f"{link} GB/s ({link_src}); peak = all bytes / that time")
        peak = round(per_layer / t_bound / 1e9, 1)
    if stack_obj is not None:   # the one-kernel stack: a launch processes every layer
        gu_ms = list(rt_ms)
        gu_us = statistics.mean(gu_ms) * 1e3
        gu_bytes = tr_bytes["layer_per_launch"] * layers
        gu_flops = 2 * T * w.k * (w.rows_gu * w.d + w.d * w.f) * layers
    elif one_kernel:
        gu_ms = list(rt_ms)
        gu_us = statistics.mean(gu_ms) * 1e3
        gu_bytes = tr_bytes["layer_per_launch"]
        gu_flops = 2 * T * w.k * (w.rows_gu * w.d + w.d * w.f)   # useful FLOP of the whole layer
    else:
        gu_us = statistics.mean(gu_ms) * 1e3
        gu_bytes = tr_bytes["gate_up_per_layer"]
        gu_flops = 2 * T * w.k * w.rows_gu * w.d                # useful gate.up FLOP per layer
    achieved = gu_bytes / (gu_us * 1e-6) / 1e9
    # (the captures cover the plain configurations only: uncoded inputs, device-resident weights)
    captured = aq == "none" and not host_w
    traffic = measured_traffic(args.workload, T, layers) if captured and (stack_obj is not None or not one_kernel) \
        else None
    # Which expert kernels run (the library's AUTO rule): the tensor-core GEMMs when an expert
    # sees at least 8 tokens on average and the shape allows them, else the GEMVs.
    gemm = (T * w.k >= 8 * w.E and w.f % 64 == 0 and (w.act == "swiglu" or w.f % 128 == 0))
    pk = peaks() or {}
    tc_peak = float(pk.get("bf16_tflops_sustained") or 1700.0)
    tc_src = ("measured (MEASURED_PEAKS.json bf16_tflops_sustained: cuBLAS bf16, seconds-long loop; "
              "f16 kind::f16 runs at the bf16 rate)" if pk.get("bf16_tflops_sustained") else "fallback 1.7 PFLOP/s")
    tc_achieved = gu_flops / (gu_us * 1e-6) / 1e12

    # ---- end to end: host x in pinned memory -> device, the stack, out -> host
    # (supplied routing is an input of the step too: idx and w are copied with x)
    x_host = [inp.cpu().pin_memory() for inp in inputs]
    r_host = [(ri.cpu().pin_memory(), rw.cpu().pin_memory()) for ri, rw in routings] if routings else None
    out_host = torch.empty((T, w.d), dtype=torch.float32).pin_memory()
    e2e_steps = max(N_ROTATE, min(args.steps, 500))

    def h2d(r):
        inputs[r].copy_(x_host[r], non_blocking=True)
        if r_host:
            routings[r][0].copy_(r_host[r][0], non_blocking=True)
            routings[r][1].copy_(r_host[r][1], non_blocking=True)

    for i in range(min(args.warmup, 10)):
        h2d(i % N_ROTATE)
        graphs[i % N_ROTATE].replay()
        out_host.copy_(outs[-1], non_blocking=True)
    barrier()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for i in range(e2e_steps):
        h2d(i % N_ROTATE)
        graphs[i % N_ROTATE].replay()
        out_host.copy_(outs[-1], non_blocking=True)
    a1.record()
    barrier()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), world)
    e2e_value = job_throughput(T * e2e_steps, world, e2e_ms)

    launches_per_step = (1 if stack_obj is not None else
                         sum(layer.launches(T, supplied) + 1 for layer in stack))   # + the RMS-norm glue
    result = None
    if rank == 0:
        step_bytes = tr_bytes["step"]
        cfg = workload_config(w, T, layers, aq)
        if host_w:
            cfg["workload"] += (", down experts" if host_w == "down" else ", all expert weights") + \
                " in page-locked host memory read in place"
            cfg["weights_location"] = ("down stack" if host_w == "down" else "both stacks") + \
                " in host memory (page-locked; read in place over the host link)"
        cfg.update({
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"per-step weight working set {step_bytes / 1e9:.2f} GB > 129 MB L2; {N_ROTATE} token inputs "
                  f"{'and routings ' if supplied else ''}rotate so consecutive steps route to different experts",
            "graph": "one CUDA graph per rotated input covers the whole stack",
            "layer_us": round(ms_step * 1e3 / layers, 3),
            "layer_tokens_per_s": round(tokens_per_s * layers, 1),
            "active_expert_bytes_per_step": step_bytes,
            "active_expert_gbs": round(step_bytes * world / (ms_step * 1e-3) / 1e9, 1),
            "active_expert_frac_of_measured_hbm": round(step_bytes / (ms_step * 1e-3) / 1e9 / peak, 4),
            "active_expert_frac_of_8tbs": round(step_bytes / (ms_step * 1e-3) / 1e9 / 8000.0, 4),
            "stage_us_mean": ({"stack_kernel": round(gu_us, 2), "per_layer": round(gu_us / layers, 3)}
                              if stack_obj is not None else {"layer_kernel": round(gu_us, 2)} if one_kernel else
                              {"routing": round(statistics.mean(rt_ms) * 1e3, 2), "gate_up": round(gu_us, 2),
                               "down": round(statistics.mean(dn_ms) * 1e3, 2),
                               "combine": round(statistics.mean(cb_ms) * 1e3, 2)}),
        })
        if stack_obj is not None:
            cfg["layer_kernel"] = ("decode_layer_kernel over the whole stack (moe_stack_forward): router, top-k, "
                                   "softmax, gate.up + SwiGLU, down, combine and the RMS-norm glue of every layer in "
                                   "one cooperative launch per step (one CTA per SM)")
            cfg["graph"] = "one CUDA graph per rotated input holds the single stack launch"
        elif one_kernel:
            cfg["layer_kernel"] = (("decode_layer_kernel with the supplied routing: gate.up + activation, down and "
                                    "combine" if supplied else
                                    "decode_layer_kernel: router, top-k, softmax, gate.up + activation, down and combine")
                                   + " in one cooperative launch per layer (one CTA per SM)")
        result = {
            "metric": METRIC, "value": round(tokens_per_s, 2), "unit": f"tokens/s through the {layers}-layer stack",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; random-init weights of the workload's shapes)",
            "config": cfg,
            "roofline": {"bound": "host-link" if host_w else "hbm",
                         "kernel": ("decode_layer_kernel (the whole stack in one launch: every layer's routed "
                                    "experts' gate.up + down bytes and router weights)" if stack_obj is not None else
                                    ("decode_layer_kernel (the whole layer: routed experts' gate.up + down "
                                     "bytes" + (")" if supplied else " and the router weights)")) if one_kernel else
                                    "expert_gemm_kernel (gate.up + activation, tcgen05)" if gemm
                                    else "gate_up_gemv (gate.up + activation + group mask)"),
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": gu_bytes, "launch_us_mean": round(gu_us, 3),
                         "launches_timed": len(gu_ms), "timing": timing_how, "peak_source": peak_src,
                         "tensor": {"useful_flop_per_launch": gu_flops, "achieved": round(tc_achieved, 2),
                                    "peak": tc_peak, "unit": "TFLOP/s", "frac": round(tc_achieved / tc_peak, 4),
                                    "peak_source": tc_src,
                                    "note": ("useful FLOP only (2*T*k*rows*d); the Q8_0 path issues a second "
                                             "MMA per weight for the exact lo part" if gemm else
                                             "GEMV path: exact code-to-f16 conversion, mma.sync for the dot "
                                             "products")},
                         "bytes_time_us": round(gu_bytes / (peak * 1e9) * 1e6, 2),
                         "flop_time_us": round(gu_flops / (tc_peak * 1e12) * 1e6, 2)},
            "e2e": {"value": round(e2e_value, 2), "unit": f"tokens/s through the {layers}-layer stack",
                    "h2d_bytes_per_step": int(x_host[0].numel() * x_host[0].element_size() +
                                              (sum(t.numel() * t.element_size() for t in r_host[0]) if r_host else 0)),
                    "d2h_bytes_per_step": int(out_host.numel() * out_host.element_size()),
                    "how": ("pinned host x (and the supplied idx, w) -> device copy, " if supplied else
                            "pinned host x -> device copy, ") +
                           "graph replay of the stack, out -> pinned host, all on the stream inside the timed region"},
            "clocks": clk,
            "gpu_launches": launches_per_step * args.steps,
        }
    return result, (w, T, layers), stack


def active_expert_bytes(stack, inputs, T, w, routings=None):
    """Unique active-expert bytes of one step, from the routing each layer took
    (gate.up bytes of every selected expert + down bytes of its active groups).  The router
    weights count toward a layer's launch only when the layer runs its router."""
    import torch

    from quantized_routed_expert_softmax_gb300 import native
    gu_b = stack[0].gate_up.shape[1]
    dn_b = stack[0].down.shape[1]
    x = inputs[0]
    ri, rw = routings[0] if routings else (None, None)
    step = 0
    gu_layer, layer_bytes = [], []
    for layer in stack:
        tr = {}
        out = layer.forward(x, idx_in=ri, w_in=rw, trace=tr)
        experts = torch.unique(tr["idx"]).numel()
        gu_layer.append(experts * gu_b)
        if w.act == "relu2":   # the down projection reads only 16-neuron groups with a non-zero h
            h = tr["h"]
            off = tr["offsets"].cpu().numpy()
            act_groups = 0
            for e in range(w.E):
                if off[e + 1] > off[e]:
                    hh = h[off[e]:off[e + 1]].reshape(off[e + 1] - off[e], -1, 16)
                    act_groups += int((hh != 0).any(dim=2).any(dim=0).sum().item())
            expert_bytes = experts * gu_b + act_groups * (dn_b // (w.f // 16))
        else:
            expert_bytes = experts * (gu_b + dn_b)
        step += expert_bytes
        layer_bytes.append(expert_bytes + (0 if routings else layer.router_w.numel() * 4))
        x = native.rmsnorm_bf16(out)
    torch.cuda.synchronize()
    return {"step": int(step), "gate_up_per_layer": int(statistics.mean(gu_layer)),
            "layer_per_launch": int(statistics.mean(layer_bytes))}


def kernel_source_sha(files=("gemv.cu", "gemm.cu", "common.cuh", "decode.cu", "gemv_core.cuh")):
    import hashlib
    csrc = os.path.join(ROOT, "quantized_routed_expert_softmax_gb300", "csrc")
    blob = b"".join(open(os.path.join(csrc, f), "rb").read() for f in files)
    return hashlib.sha1(blob).hexdigest()[:12]


def measured_traffic(workload, T, layers):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, while the
    kernel's own source files (the entry's "sources") are unchanged since the capture; else None.
    An entry for a whole-stack launch (it names its "layers") scales to this run's stack depth:
    every layer of a stack moves the same bytes."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        entry = json.load(open(p)).get(f"{workload}_T{T}")
    except (OSError, ValueError):
        return None
    if not entry or entry.get("source_sha1_12") != kernel_source_sha(tuple(entry.get("sources", ()))):
        return None
    if "layers" in entry:
        return int(round(entry["bytes"] * layers / entry["layers"]))
    return entry.get("bytes")


# ====================================================================== reference arm
def run_reference(args, rank, world):
    """The oracle as it stands on the host cores.  A step is one bounded sample of the
    workload: one oracle forward of one layer of the stack on up to 8 of the step's tokens;
    the line's value extrapolates those samples to tokens per second through the whole stack
    (mean time per token and layer x tokens x layers), and ms_per_step is the measured time
    of one such sample, so steps x ms_per_step is the time actually spent."""
    from quantized_routed_expert_softmax_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    T = args.tokens
    layers = args.layers or default_layers(w)
    budget = 120.0
    t0 = time.perf_counter()
    step_s, n, threads, desc, unit_s = oracle_sample(w, T, layers, max_units=max(1, args.steps),
                                                     time_budget_s=budget, warmup_units=min(args.warmup, 1),
                                                     with_unit_time=True)
    wall = time.perf_counter() - t0
    value = T / step_s
    cfg = workload_config(w, T, layers)
    cfg["parallelism"] = "host cores"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6),
        "unit": f"tokens/s through the {layers}-layer stack", "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": round(unit_s * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded; random-init weights of the workload's shapes)", "config": cfg,
        "step_is": (f"one bounded sample: the oracle's forward of one layer of the {layers}-layer stack on "
                    f"{min(T, 8)} token(s)"),
        "units_timed": n, "stack_step_ms_extrapolated": round(step_s * 1e3, 3),
        "cpu_baseline": {"value": round(value, 6), "unit": f"tokens/s through the {layers}-layer stack",
                         "cores": threads, "kind": "oracle", "sample": desc, "wall_s": round(wall, 1)},
        "e2e": {"value": round(value, 6), "unit": f"tokens/s through the {layers}-layer stack",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# Further configurations measured by the default run, each with its own workload, roofline and
# oracle baseline: prefill on the headline stack's own weights (Gemma shape, T = 512) and its
# activation-quantised decode, per-channel int8 experts on the Gemma shape (T = 1 and 64), the
# Nemotron-shaped NVFP4 ReLU^2 stack at one token (and, 8 layers deep, with its experts in
# page-locked host memory read in place), and MiniMax-shaped prefill (T = 4096), plain and
# activation-quantised.
SECONDARY = [("gemma", 512, 30, 20, "none", "none"), ("gemma", 1, 30, 400, "q8_0", "none"),
             ("gemma_int8pc", 1, 8, 400, "none", "none"), ("gemma_int8pc", 64, 8, 100, "none", "none"),
             ("nemotron", 1, 40, 400, "none", "none"), ("nemotron", 1, 8, 200, "none", "down"),
             ("nemotron", 1, 8, 200, "none", "all"),
             ("minimax", 4096, 8, 10, "none", "none"), ("minimax", 4096, 8, 10, "q8_0", "none"),
             ("zipf_nvfp4", 1, 4, 400, "none", "none"), ("zipf_nvfp4", 64, 4, 100, "none", "none")]


def cpu_baseline(w, T, layers, budget_s, single_core_s=8.0, single=True, act_q8=False):
    import oracle
    cache = {}
    step_s, n, threads, desc = oracle_sample(w, T, layers, max_units=10 * layers, time_budget_s=budget_s,
                                             warmup_units=1, cache=cache, act_q8=act_q8)
    out = {"value": round(T / step_s, 6), "unit": f"tokens/s through the {layers}-layer stack", "cores": threads,
           "kind": "oracle", "sample": desc}
    if single:
        out["single_core"] = single_core_baseline(w, T, layers, threads, cache, budget_s=single_core_s)
    return out


def main():
    args = parse()
    rank, world, local_rank = dist_info()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    result, (w, T, layers), stack = run_ours(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, T, layers, 15.0, act_q8=args.act_quant == "q8_0")
    if args.secondary and args.workload == "gemma" and args.tokens == 1 and not args.layers and not args.experts:
        import torch
        secondary = []
        w_prev = w
        for name, t2, n2, steps2, aq2, hw2 in SECONDARY:
            a2 = argparse.Namespace(**vars(args))
            a2.workload, a2.tokens, a2.layers, a2.act_quant, a2.host_weights = name, t2, n2, aq2, hw2
            a2.steps, a2.warmup = steps2, max(3, min(args.warmup, 5))
            reuse = (stack if stack is not None and name == w_prev.name and n2 == len(stack) and
                     hw2 == getattr(stack[0], "host_resident", "none") else None)
            if reuse is None:
                stack = None
                torch.cuda.empty_cache()
            r2, (w2, _, _), built = run_ours(a2, rank, world, local_rank, prebuilt=reuse)
            stack = built
            if rank == 0:
                if not args.no_cpu_baseline:
                    r2["cpu_baseline"] = cpu_baseline(w2, t2, n2, 5.0, single=False, act_q8=aq2 == "q8_0")
                for key in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data"):
                    r2.pop(key, None)
                secondary.append(r2)
            w_prev = w2
            del built, r2
            torch.cuda.empty_cache()
        if rank == 0:
            result["secondary"] = secondary
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
