#!/usr/bin/env python
"""Throughput of one MoE layer, forward + backward, on GB300.

One step = the whole hot path over one batch of synthetic tokens: router,
deterministic dispatch, grouped-GEMM SwiGLU experts, fixed-order combine,
and the backward (input and weight gradients).  The workload is the
DeepSeek-V2-Lite-like layer (T=8192 tokens, d=2048, f=1408, 64 routed
experts top-6, 2 shared experts); its weights (1.15 GB) and activations are
far larger than the 129 MB L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs an independent replica on its own batch
(weak scaling, no collective on the data path); the barrier-bracketed time
is the max over ranks and `value` counts the tokens of all ranks.
`--impl reference` times the CPU fp64 oracle on the host cores instead.
"""
import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s (fwd+bwd, 1xGB300)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dsv2lite_T8192_d2048_f1408_E64_k6_S2")
    ap.add_argument("--megakernel", type=int, default=-1, help="1: forward MegaKernel, 0: kernel chain, "
                    "-1: the faster of the two, timed during set-up (same bits)")
    ap.add_argument("--bwd-megakernel", type=int, default=-1, help="1: backward input part as one MegaKernel, "
                    "0: kernel chain, -1: the faster of the two (same bits)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=256)
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller captures for profiling)")
    ap.add_argument("--gemm-pair-kinds", type=int, default=-1,
                    help="bit mask of grouped-GEMM kinds run on CTA pairs (-1: the library default)")
    ap.add_argument("--no-bwd-overlap", action="store_true",
                    help="run the backward's weight-gradient GEMMs on the caller's stream (no B/W overlap)")
    ap.add_argument("--no-route-fusion", action="store_true",
                    help="run the router, scan and scatter as three kernels instead of one cooperative launch")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step's kernels from the host instead of replaying one captured CUDA graph")
    ap.add_argument("--no-autotune", action="store_true",
                    help="skip the library's measured GEMM autotuner (run during set-up, untimed)")
    return ap.parse_args()


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's `value` (the slowest replica sets the
    time); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms_per_step / 1000.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, k)
                elif isinstance(o, (int, float)):
                    flat[pre] = float(o)
            walk(d)
            if "bf16_tflops" in flat or "hbm_gbs" in flat:
                return flat, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms; only the
    samples taken inside the timed window count."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        self.proc = None
        self.window = None

    def start(self):
        """Starts sampling and returns once the first sample is written (at
        most 3 s), so the timed window that follows is covered."""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(self.gpu_index)], stdout=self.tmp,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t_end = time.time() + 3.0
        while time.time() < t_end and os.path.getsize(self.tmp.name) == 0:
            time.sleep(0.01)

    def mark(self, t0, t1):
        """Host wall-clock bounds of the timed window."""
        self.window = (t0, t1)

    def _rows(self):
        rows = []
        for line in open(self.tmp.name):
            r = [c.strip() for c in line.strip().split(", ")]
            if len(r) < 10 or not r[2].replace(".", "").isdigit():
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            rows.append((ts, r))
        return rows

    def stop(self):
        if self.proc is None:
            return None
        if self.window is not None:  # a window shorter than a period: let one sample after its start land
            t_end = time.time() + 0.5
            while time.time() < t_end and not any(ts is not None and ts >= self.window[0] for ts, _ in self._rows()):
                time.sleep(0.02)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        rows = self._rows()
        os.unlink(self.tmp.name)
        inside = rows
        if self.window is not None:
            t0, t1 = self.window
            inside = [x for x in rows if x[0] is not None and t0 <= x[0] <= t1]
            if not inside:  # a window shorter than the sampling period: the first sample after it began
                after = [x for x in rows if x[0] is not None and x[0] >= t0]
                inside = after[:1]
        if not inside:
            return None
        sm = [float(r[2]) for _, r in inside]
        mx = [float(r[3]) for _, r in inside if r[3].replace(".", "").isdigit()]
        reasons = sorted({self.REASONS[i] for _, r in inside for i in range(4) if r[6 + i] == "Active"})
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(sm), "period_ms": 50}
        if self.window is not None:
            out["window_ms"] = round(1000 * (self.window[1] - self.window[0]), 1)
        return out


def workload_cfg(name, tokens=0):
    from combine_fp32_softmax_gb300.configs import BY_NAME
    cfg = BY_NAME[name]
    if tokens:
        cfg = cfg.with_(T=tokens, name=cfg.name.replace(f"T{cfg.T}_", f"T{tokens}_"))
    return cfg


def gemm_flops_per_launch(cfg):
    """Algorithmic flops of one launch of each grouped GEMM (2 flops per
    multiply-add; every routed and shared row, no padding)."""
    dfr = 2 * cfg.d * cfg.f * cfg.Rs
    return {"gemm1_swiglu": 2 * dfr, "gemm2_scale": dfr, "gemm_dh": dfr, "gemm_dx": 2 * dfr,
            "gemm_dw13": 2 * dfr, "gemm_dw2": dfr,
            # the MegaKernels run two GEMMs each (with the gather and the token sums in the same launch)
            "megakernel": 3 * dfr, "megakernel_bwd": 3 * dfr}


def memory_bytes_per_launch(cfg):
    """Algorithmic DRAM bytes of one launch of each memory-bound kernel
    (what the method must read and write once; index reads included)."""
    T, d, E, k, R, Rs = cfg.T, cfg.d, cfg.E, cfg.k, cfg.R, cfg.Rs
    nt = -(-cfg.f // 256)
    rows_copy = T * d * 2 + R * d * 2 + R * 4           # each x (dy) row read once, written to its k rows
    rows_sum = Rs * d * 4 + T * d * 4 + R * 4           # fp32 rows read once, one fp32 row per token written
    return {"gather": rows_copy, "combine_bwd": rows_copy, "combine": rows_sum, "dispatch_bwd": rows_sum,
            "route_tables": T * E * 4 + T * k * 8 + R * 12,  # logits in; top-k out; dest, row_token, row_slot
            "route_bwd": T * E * 8 + T * k * 12,             # logits in, dlogits out; idx, w, dw in
            "dw_reduce": R * nt * 4 + R * 4 + T * k * 4}


def traffic_from_profiles(kernel, workload, cta_group=None):
    """Per-launch DRAM bytes recorded from an ncu capture in profiles/, as
    (bytes or None, note).  A line `traffic_bytes_per_launch[cta_group=N]: B`
    is specific to one tile shape of a grouped GEMM and is preferred when that
    shape ran; `traffic_bytes_per_launch: B` holds for any.  The capture names
    the kernel build it measured (`source_sha256:`); bytes of another build
    are not reported."""
    from combine_fp32_softmax_gb300.build import source_digest
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None, "no ncu capture of this kernel and workload in profiles/"
    lines = [ln.strip() for ln in open(path)]
    built = [ln.split(":", 1)[1].strip() for ln in lines if ln.startswith("source_sha256:")]
    if not built or built[0] != source_digest():
        return None, f"ncu capture in profiles/ is of another build of the kernels ({built[0] if built else '?'})"
    keys = ([f"traffic_bytes_per_launch[cta_group={cta_group}]:"] if cta_group else []) + ["traffic_bytes_per_launch:"]
    for key in keys:
        for line in lines:
            if line.startswith(key):
                try:
                    return float(line.split(":", 1)[1].strip().split()[0]), f"ncu capture {os.path.relpath(path, ROOT)}"
                except ValueError:
                    return None, "unreadable traffic line"
    return None, "no traffic line for this tile shape"


# ------------------------------------------------------------ oracle timing
def oracle_step_time(cfg, inp, ntok):
    """Seconds of the fp64 oracle for forward + backward of the same layer on
    the first `ntok` tokens (a bounded sample of the batch)."""
    from oracle import moe_oracle as O
    x, z, dy = inp.x[:ntok], inp.logits[:ntok], inp.dy[:ntok]
    t0 = time.perf_counter()
    fw = O.layer_fwd(x, z, inp.W1, inp.W3, inp.W2, k=cfg.k, S=cfg.S, renorm=cfg.renorm)
    O.layer_bwd(fw, dy, x, inp.W1, inp.W3, inp.W2, renorm=cfg.renorm)
    return time.perf_counter() - t0


def cpu_baseline(cfg, inp, ntok, reps=1):
    times = [oracle_step_time(cfg, inp, ntok) for _ in range(reps)]
    t = min(times)
    return {"value": ntok / t, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of the same layer on the first {ntok} of {cfg.T} tokens "
                      f"(all experts' weight gradients included), best of {reps}"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    cfg = workload_cfg(args.workload, args.tokens)
    from combine_fp32_softmax_gb300.inputs import make_layer_inputs
    inp = make_layer_inputs(cfg, seed=0)
    ntok = args.cpu_sample_tokens
    for _ in range(args.warmup):
        oracle_step_time(cfg, inp, ntok)
    times = [oracle_step_time(cfg, inp, ntok) for _ in range(args.steps)]
    total = sum(times)
    value = ntok * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg, None),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: fp64 oracle fwd+bwd on the first {ntok} of {cfg.T} tokens"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(cfg, megakernel):
    return {"workload": cfg.name, "T": cfg.T, "d_model": cfg.d, "d_ff": cfg.f, "E": cfg.E, "k": cfg.k,
            "n_shared": cfg.S, "renorm": cfg.renorm, "megakernel": megakernel,
            "l2": "inputs larger than L2 (no flush): weights 1.15 GB + activations per step",
            "parallelism": "replicas"}


# --------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    from combine_fp32_softmax_gb300 import moe
    from combine_fp32_softmax_gb300.inputs import make_layer_inputs

    rank, world, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload_cfg(args.workload, args.tokens)
    inp = make_layer_inputs(cfg, seed=rank)
    g = {k: getattr(inp, k).to(dev) for k in ("x", "logits", "W1", "W3", "W2", "dy")}
    ws = moe.alloc_workspace(cfg, dev)
    if args.gemm_pair_kinds >= 0:
        moe.moe_set_gemm_pair_kinds(args.gemm_pair_kinds)
    if args.no_bwd_overlap:
        moe.moe_set_bwd_overlap(False)
    if args.no_route_fusion:
        moe.moe_set_route_fusion(False)
    f32 = torch.float32
    nexp = cfg.E + cfg.S
    out = dict(y=torch.empty(cfg.T, cfg.d, dtype=f32, device=dev),
               idx=torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev),
               w=torch.empty(cfg.T, cfg.k, dtype=f32, device=dev),
               dx=torch.empty(cfg.T, cfg.d, dtype=f32, device=dev),
               dz=torch.empty(cfg.T, cfg.E, dtype=f32, device=dev),
               dW1=torch.empty(nexp, cfg.f, cfg.d, dtype=f32, device=dev),
               dW3=torch.empty(nexp, cfg.f, cfg.d, dtype=f32, device=dev),
               dW2=torch.empty(nexp, cfg.d, cfg.f, dtype=f32, device=dev))
    def device_ms(fn, min_ms=20.0, max_iters=400):
        """Device time per call of fn: 2 untimed calls, then enough timed calls
        for at least min_ms of work (a short layer's 5 calls are launch noise)."""
        for _ in range(2):
            fn()
        iters, ms = 5, 0.0
        while True:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(iters):
                fn()
            b.record()
            b.synchronize()
            ms = a.elapsed_time(b)
            if ms >= min_ms or iters >= max_iters:
                return ms / iters
            iters = min(max_iters, max(iters + 1, int(iters * 1.2 * min_ms / max(ms, 1e-3))))

    def fwd_ms(use_mk):
        """Device time of the forward alone (kernel chain or MegaKernel)."""
        return device_ms(lambda: moe.moe_layer_fwd(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], out["y"],
                                                   out["idx"], out["w"], ws, use_megakernel=use_mk))

    def best_of(time_one):
        """Chain and MegaKernel timed alternately twice; the faster time of each."""
        t = {"chain": [], "megakernel": []}
        for _ in range(2):
            t["chain"].append(time_one(0))
            t["megakernel"].append(time_one(1))
        return {k: min(v) for k, v in t.items()}

    # Set-up, untimed: the library's measured autotuner picks each grouped
    # GEMM's tile shape and L2 prefetch depth on this very layer.
    tuning = None
    if not args.no_autotune:
        tuning = moe.moe_autotune(cfg, g["logits"], g["x"], g["W1"], g["W3"], g["W2"], g["dy"], out["y"], out["idx"],
                                  out["w"], out["dx"], out["dz"], out["dW1"], out["dW3"], out["dW2"], ws)
        for v in tuning["kinds"].values():
            v["us"] = round(v["us"], 1)
        tuning["fwd_us"] = [round(v, 1) for v in tuning["fwd_us"]]
        tuning["bwd_us"] = [round(v, 1) for v in tuning["bwd_us"]]
    pair_kinds = moe.moe_set_gemm_pair_kinds(moe.ALL_PAIR_KINDS)
    moe.moe_set_gemm_pair_kinds(pair_kinds)

    mk = args.megakernel
    fwd_times = None
    if mk < 0:  # the faster forward of the two (same bits either way)
        fwd_times = best_of(fwd_ms)
        mk = 1 if fwd_times["megakernel"] < fwd_times["chain"] else 0

    def bwd_ms(use_mk):
        """Device time of the backward alone (kernel chain or MegaKernel input part)."""
        which = 3 | (moe.MOE_BWD_MEGAKERNEL if use_mk else 0)
        return device_ms(lambda: moe.moe_layer_bwd(cfg, g["dy"], g["logits"], g["x"], g["W1"], g["W3"], g["W2"],
                                                   out["idx"], out["w"], ws, out["dx"], out["dz"], out["dW1"],
                                                   out["dW3"], out["dW2"], which=which))

    bmk = args.bwd_megakernel
    bwd_times = None
    if bmk < 0:
        bwd_times = best_of(bwd_ms)
        bmk = 1 if bwd_times["megakernel"] < bwd_times["chain"] else 0
    bwd_which = 3 | (moe.MOE_BWD_MEGAKERNEL if bmk else 0)

    def step(src=g):
        moe.moe_layer_fwd(cfg, src["logits"], src["x"], g["W1"], g["W3"], g["W2"], out["y"], out["idx"], out["w"],
                          ws, use_megakernel=mk)
        moe.moe_layer_bwd(cfg, src["dy"], src["logits"], src["x"], g["W1"], g["W3"], g["W2"], out["idx"], out["w"],
                          ws, out["dx"], out["dz"], out["dW1"], out["dW3"], out["dW2"], which=bwd_which)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    code, info = moe.moe_get_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error {code} ({info}) during warm-up")

    # The timed steps replay the step as one CUDA graph (the library's
    # launches, including the cooperative routing launch, the CTA-pair
    # launches and the fork/join of the weight-gradient stream, captured once):
    # the same kernels on the same buffers, without a host launch per kernel.
    run_step = step
    graph_state = "off (--no-graph)" if args.no_graph else "replayed"
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                step()
            run_step = graph.replay
            for _ in range(2):
                run_step()
            barrier()
        except Exception as exc:  # a capture the driver refuses: measure with host launches instead
            graph_state = f"capture failed, host launches: {str(exc).splitlines()[0][:120]}"
            run_step = step
            torch.cuda.synchronize()
            for _ in range(2):
                step()
            barrier()
        code, info = moe.moe_get_device_error(ws)
        if code != 0:
            raise RuntimeError(f"device error {code} ({info}) after the graph capture")

    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e0.record(stream)
    for i in range(args.steps):
        run_step()
        step_ev[i].record(stream)
    e1.record(stream)
    barrier()
    sampler.mark(t_host0, time.time())
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    per_step = [e0.elapsed_time(step_ev[0])] + [step_ev[i - 1].elapsed_time(step_ev[i]) for i in range(1, args.steps)]
    ms_median = max_over_ranks(statistics.median(per_step), dev)
    value = job_tokens_per_s(cfg.T, world, ms)

    # ---- per-kernel times: the library's CUDA events around each launch, on
    # the stream it is launched on, over as many more steps.  The backward's
    # B/W overlap is switched off for this pass: with it on, the events of a
    # weight-gradient GEMM on the second stream would also span its wait for
    # the SMs that dX holds.  Nothing else differs from the timed steps.
    overlap = moe.moe_set_bwd_overlap(False)
    moe.moe_trace_reset()
    moe.moe_trace_enable(True)
    t_trace = time.time()
    for _ in range(args.steps):
        step()
    barrier()
    trace_wall_s = time.time() - t_trace
    moe.moe_trace_enable(False)
    trace = moe.moe_trace_read()
    moe.moe_set_bwd_overlap(overlap)

    # ---- end to end through the C ABI with host buffers: every step uploads
    # its inputs (x, logits, dy) from pinned host memory and reads its
    # results (y, dx, dlogits) back.  Uploads and downloads run on two more
    # streams (the two directions use separate copy engines), double
    # buffered, so step i+1's upload and step i's download overlap compute.
    e2e = None
    if not args.no_e2e:
        pin = {k: getattr(inp, k).pin_memory() for k in ("x", "logits", "dy")}
        srcs = [{k: torch.empty_like(g[k]) for k in pin} for _ in range(2)]
        outs = [{k: torch.empty_like(out[k]) for k in ("y", "dx", "dz")} for _ in range(2)]
        hosts = [{k: torch.empty(out[k].shape, dtype=out[k].dtype, pin_memory=True) for k in ("y", "dx", "dz")}
                 for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in hosts[0].values())
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(nsteps, start_evt=None, end_evt=None):
            if start_evt is not None:
                start_evt.record(stream)
                up.wait_event(start_evt)
                down.wait_event(start_evt)
            with torch.cuda.stream(up):
                for k in pin:
                    srcs[0][k].copy_(pin[k], non_blocking=True)
                in_ready[0].record(up)
            for i in range(nsteps):
                b = i & 1
                stream.wait_event(in_ready[b])
                if i >= 2:
                    stream.wait_event(out_free[b])  # step i-2's download has read that output buffer
                o = outs[b]
                moe.moe_layer_fwd(cfg, srcs[b]["logits"], srcs[b]["x"], g["W1"], g["W3"], g["W2"], o["y"],
                                  out["idx"], out["w"], ws, use_megakernel=mk)
                moe.moe_layer_bwd(cfg, srcs[b]["dy"], srcs[b]["logits"], srcs[b]["x"], g["W1"], g["W3"], g["W2"],
                                  out["idx"], out["w"], ws, o["dx"], o["dz"], out["dW1"], out["dW3"], out["dW2"],
                                  which=bwd_which)
                done[b].record(stream)
                if i + 1 < nsteps:
                    with torch.cuda.stream(up):
                        if i >= 1:
                            up.wait_event(done[1 - b])  # step i-1 no longer reads that input buffer
                        for k in pin:
                            srcs[1 - b][k].copy_(pin[k], non_blocking=True)
                        in_ready[1 - b].record(up)
                with torch.cuda.stream(down):
                    down.wait_event(done[b])
                    for k in hosts[b]:
                        hosts[b][k].copy_(o[k], non_blocking=True)
                    out_free[b].record(down)
            stream.wait_stream(up)
            stream.wait_stream(down)
            if end_evt is not None:
                end_evt.record(stream)

        e2e_steps(max(3, args.warmup))
        barrier()
        e2e_steps(args.steps, e0, e1)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
        e2e = {"value": job_tokens_per_s(cfg.T, world, ems), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "overlap": "uploads and downloads on two more streams, double-buffered"}

    code, info = moe.moe_get_device_error(ws)
    if code != 0:
        raise RuntimeError(f"device error {code} ({info}) in the timed region")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # ---- roofline of every kernel, and of the dominant one (largest share of
    # device time).  GEMMs against the measured bf16 peak, memory-bound kernels
    # against the measured copy rate.  The kernels were timed one launch at a
    # time over a pass well under a second: the burst figure applies; only a
    # pass of a second or more under the power cap is compared with the
    # sustained figure.
    peaks, peak_src = load_peaks()
    flops = gemm_flops_per_launch(cfg)
    mem = memory_bytes_per_launch(cfg)
    capped = bool(clocks and "sw_power_cap" in clocks.get("reasons", []))
    sustained = trace_wall_s >= 1.0 and capped
    bf16_peak = peaks.get("bf16_tflops_sustained" if sustained else "bf16_tflops",
                          FALLBACK_PEAKS["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    peak_kind = (f"bf16 {'sustained' if sustained else 'burst'} ({peak_src}; per-kernel pass "
                 f"{trace_wall_s:.2f} s, power cap {'seen' if capped else 'not seen'} in the timed window)")
    total_ms = sum(v[0] for v in trace.values())
    per_kernel = {}
    for name, (tot, n) in trace.items():
        ms_launch = tot / n
        if name in flops:
            a = flops[name] / (ms_launch / 1000.0) / 1e12
            per_kernel[name] = {"bound": "tensor", "achieved": a, "peak": bf16_peak, "unit": "TFLOP/s",
                                "frac": a / bf16_peak, "us": 1000 * ms_launch, "work": flops[name]}
        elif name in mem:
            a = mem[name] / (ms_launch / 1000.0) / 1e9
            per_kernel[name] = {"bound": "hbm", "achieved": a, "peak": hbm_peak, "unit": "GB/s",
                                "frac": a / hbm_peak, "us": 1000 * ms_launch, "work": mem[name]}
    dom = max(trace, key=lambda k: trace[k][0])
    roof = dict(per_kernel.get(dom, {"bound": "hbm", "achieved": None, "peak": hbm_peak, "unit": "GB/s",
                                     "frac": None}))
    roof["kernel"] = dom
    roof["peak_source"] = peak_kind if roof["bound"] == "tensor" else f"HBM copy, {peak_src}"
    gemm_kind = {"gemm1_swiglu": 0, "gemm2_scale": 1, "gemm_dh": 2, "gemm_dx": 3, "gemm_dw13": 4, "gemm_dw2": 5}
    cta_group = 1 + ((pair_kinds >> gemm_kind[dom]) & 1) if dom in gemm_kind else None
    roof["traffic"], roof["traffic_source"] = traffic_from_profiles(dom, cfg.name, cta_group)
    if cta_group:
        roof["cta_group"] = cta_group
    roof["share"] = trace[dom][0] / total_ms
    roof["per_kernel"] = {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()
                              if kk in ("achieved", "frac", "unit", "us")} for k, v in per_kernel.items()}
    kernels = {k: {"ms_per_launch": v[0] / v[1], "launches": v[1], "share": v[0] / total_ms} for k, v in trace.items()}
    # every GEMM flop of the step over the time of the launches that ran GEMMs
    gemm_ms = sum(trace[k][0] for k in flops if k in trace) / args.steps
    step_flops = 18 * cfg.d * cfg.f * cfg.Rs
    all_gemm_tflops = step_flops / (gemm_ms / 1000.0) / 1e12 if gemm_ms else None
    roof["all_gemms"] = {"achieved": all_gemm_tflops, "frac": all_gemm_tflops / bf16_peak if all_gemm_tflops else None,
                         "unit": "TFLOP/s"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_median,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(cfg, mk),
            "e2e": e2e, "gpu_launches": int(sum(v[1] for v in trace.values())),
            "roofline": roof, "clocks": clocks,
            "gemm_tflops_all": all_gemm_tflops, "fwd_ms": fwd_times, "bwd_ms": bwd_times,
            "bwd_megakernel": bmk, "kernels": kernels,
            "tuning": {"gemm_pair_kinds": pair_kinds, "autotune": tuning, "bwd_overlap": overlap,
                       "route_fusion": not args.no_route_fusion, "cuda_graph": graph_state},
            "kernel_timing": "per-launch CUDA events on the launching stream over --steps further steps run with "
                             "the backward's B/W overlap off (the timed steps run with it on)"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, args.cpu_sample_tokens)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
