"""Benchmark: decode MoE-layer tokens/s and expert-weight HBM GB/s.

Workload (default): the 35B-like decode stack -- d_model 2048, E=256 routed
experts, K=4, expert ffn 512, one always-on shared expert, unfused LoRA r=16
on the shared expert, prerouter heads 2560->512->256, 40 layers, batch 1 --
on seeded synthetic weights and inputs.  One step = one decode token through
all 40 layers: per layer the routed + shared expert FFN, the fused combine +
residual (+ RMS for the next layer's input), the prerouter head of the next
layer and its top-K router (layer 0 routes with its own router).  Steady-state
steps are replayed from captured CUDA graphs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 35b]
    python bench.py --config batched-T4096 ...   # one layer over T tokens
    python bench.py --impl reference ...   # the CPU oracle, same metric

Prints one JSON line (rank 0).  N > 1 runs N independent replicas (the layer
does not shard across GPUs in this build), one per GPU, launched by torchrun.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode MoE-layer tokens/s and expert-weight HBM GB/s vs GB300 peak (1 GPU)"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps; default 2400 for the decode stack (about a second, "
                         "so that the clock sampler sees it), 256 for a batched layer, 16 "
                         "oracle layer passes for --impl reference")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="35b")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=40,
                    help="layer samples the oracle baseline times (native arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-tier", action="store_true",
                    help="decode with the routed experts in pinned host memory, gathered into "
                         "HBM a token ahead, against the HBM-resident stack")
    ap.add_argument("--cache-slots", type=int, default=64,
                    help="--host-tier with --path chain: HBM cache slots per layer")
    ap.add_argument("--free-sms", type=int, default=0,
                    help="--host-tier with --path chain: SMs the chained step leaves to the copies")
    ap.add_argument("--side-streams", type=int, default=1,
                    help="--host-tier with --path chain: streams the layers' cache updates use")
    ap.add_argument("--route-agreement", action="store_true",
                    help="measure how often the predicted routes agree with the layers' own "
                         "routers (seeded decode steps)")
    ap.add_argument("--lora-merge", action="store_true",
                    help="time merging the shared-expert adapters into the int4 weights "
                         "(moe_merge_lora) and report the retained delta")
    ap.add_argument("--engine", default="auto", choices=["auto", "mma_sync", "tcgen05"],
                    help="batched configs: the grouped-GEMM engine (auto: the library's "
                         "default, the register engine)")
    ap.add_argument("--path", default="chain", choices=["chain", "cluster", "fused", "per-call"],
                    help="chain: two kernels per layer chained by programmatic dependent "
                         "launch; cluster: the same step with one cluster kernel per layer "
                         "(h exchanged in distributed shared memory); fused: one persistent "
                         "kernel per step; per-call: the four calls per layer")
    ap.add_argument("--no-l2-prefetch", action="store_true",
                    help="cluster path: no L2 prefetch of the down rows in the prologue")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_traffic(cfg, path: str):
    """DRAM bytes (read + write) of one whole decode step of cfg on `path`
    ("fused", "chain" or "cluster"), scaled from the ncu capture of the 4-layer 35B-like
    stack summarised under profiles/ (per-layer bytes x layers + the step's
    fixed launches); None for other layer shapes, or when the kernel sources
    have changed since that capture."""
    from int4_expert_gemv_gb300.configs import MOE35B
    if (cfg.d, cfg.E, cfg.K, cfg.F, cfg.shared, cfg.bits, cfg.H, cfg.lora_r) != (
            MOE35B.d, MOE35B.E, MOE35B.K, MOE35B.F, MOE35B.shared, MOE35B.bits, MOE35B.H,
            MOE35B.lora_r):
        return None
    layers = cfg.depth
    import hashlib
    import re
    name = {"fused": "decode_step_35b_L4.md", "chain": "decode_chain_35b_L4.md",
            "cluster": "decode_cluster_35b_L4.md"}.get(path)
    p = os.path.join(ROOT, "profiles", name) if name else ""
    if not p or not os.path.exists(p):
        return None
    text = open(p).read()
    per_layer = re.search(r"traffic_bytes_per_layer: (\d+)", text)
    fixed = re.search(r"traffic_bytes_fixed: (\d+)", text)
    files = re.search(r"kernel_sources: (.+)", text)
    digest = re.search(r"kernel_sources_sha256_16: ([0-9a-f]+)", text)
    if not (per_layer and files and digest):
        return None
    h = hashlib.sha256()
    for f in files.group(1).split():
        h.update(open(os.path.join(ROOT, "int4_expert_gemv_gb300", "csrc", f), "rb").read())
    if h.hexdigest()[:16] != digest.group(1):
        return None
    return int(per_layer.group(1)) * layers + (int(fixed.group(1)) if fixed else 0)


# ---------------------------------------------------------------- ranks
def max_over_ranks(v: float, world: int, device: str = "cuda") -> float:
    """The largest of every rank's v: the job takes as long as its slowest
    rank (a collective; every rank calls it)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank decodes `steps` tokens (independent
    replicas, weak scaling) in the slowest rank's `ms`."""
    return world * steps / (ms / 1000.0)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        # nvidia-smi takes a moment to start: the work to be sampled waits
        # for its first line (at most 5 s)
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 5.0 and self.samples() == 0:
            time.sleep(0.05)
        return self

    def samples(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for line in f if line.count(",") >= 8)
        except OSError:
            return 0

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- oracle
def oracle_layer_sampler(cfg, n_layers: int):
    """Host data for n_layers distinct layers and a function timing one layer
    of the oracle (head + top-K + experts + combine) on it."""
    import numpy as np

    import oracle as orc
    from int4_expert_gemv_gb300 import synth

    data = []
    for r in range(min(n_layers, cfg.L)):
        x = synth.step_input(cfg, 10_000 + r)[0].astype(np.float64)
        router = synth.router_host(cfg, r)
        idx, w, _ = orc.topk(orc.head_logits(router, x), cfg.K)
        prev, _, _ = orc.topk(orc.head_logits(router, -x), cfg.K)
        exps = {e: synth.expert_host(cfg, r, e) for e in idx.tolist()}
        any_e = next(iter(exps.values()))
        data.append(dict(x=x, idx=idx, w=w, prev=prev,
                         experts=[exps.get(e, any_e) for e in range(cfg.E)],
                         shared=synth.expert_host(cfg, r, synth.SHARED_EXPERT) if cfg.shared else None,
                         head=synth.head_host(cfg, r)))

    def run_layer(i: int):
        dd = data[i % len(data)]
        z = orc.head_logits(dd["head"], dd["x"], dd["idx"], dd["prev"], cfg.K)
        orc.topk(z, cfg.K)
        y = orc.expert_ffn(dd["experts"], dd["shared"], dd["x"][None], dd["idx"][None])[0]
        orc.combine(y, dd["w"], cfg.shared, dd["x"])

    return run_layer


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_threads() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle_layers(run_layer, layer_samples: int, threads: int) -> float:
    """Seconds for layer_samples oracle layer passes at `threads` threads."""
    import oracle as orc
    orc.set_threads(threads)
    try:
        run_layer(0)
        t0 = time.perf_counter()
        for i in range(layer_samples):
            run_layer(i)
        return time.perf_counter() - t0
    finally:
        orc.set_threads(1)


def cpu_baseline(cfg, layer_samples: int):
    """The oracle on the host cores: layer passes timed at every core (the
    reported value) and on one thread; results are the same bits at both."""
    import oracle as orc
    run_layer = oracle_layer_sampler(cfg, 4)
    n = host_threads() if orc.openmp() else 1
    dt_n = time_oracle_layers(run_layer, layer_samples, n)
    dt_1 = time_oracle_layers(run_layer, layer_samples, 1) if n > 1 else dt_n
    tok = lambda dt: layer_samples / (dt * cfg.depth)
    return {"value": tok(dt_n), "unit": "tokens/s", "cores": n, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "single_thread": {"value": tok(dt_1), "unit": "tokens/s", "cores": 1},
            "sample": f"{layer_samples} layer passes (head, top-K, {cfg.slots} experts, combine) "
                      f"on 4 distinct layers: {dt_n:.1f} s on {n} threads (OpenMP over output "
                      f"rows), {dt_1:.1f} s on 1; extrapolated to a {cfg.depth}-layer token"}


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as orc
    run_layer = oracle_layer_sampler(cfg, 4)
    n = host_threads() if orc.openmp() else 1
    orc.set_threads(n)
    for i in range(args.warmup):
        run_layer(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run_layer(i)
    dt = time.perf_counter() - t0
    orc.set_threads(1)
    v = args.steps / (dt * cfg.depth)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "batch": 1, "layers": cfg.depth},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": n, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step = one layer pass of the plain C oracle "
                                       f"(head, top-K, {cfg.slots} experts, combine) on {n} "
                                       f"threads (OpenMP over output rows); "
                                       f"tokens/s = steps / (time * {cfg.depth} layers)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- native
def path_dtype(cfg, path: str) -> str:
    """What the timed decode path computes in."""
    w = f"int{cfg.bits}-g{cfg.group} weights (fp16 scale, bias)"
    if path in ("chain", "cluster", "fused"):
        return (f"{w} x 16-bit fixed-point activations (power-of-two scale per 16-byte code "
                f"chunk, exact integer chunk dots), fp32 accumulate")
    return f"{w} x f32 activations, fp32 accumulate"


def kernels_per_step(cfg, stack, cluster=False) -> int:
    """Kernel launches of one steady-state step (counted from the calls the
    driver makes; the kernels per call are fixed by the library)."""
    ed = stack.m.layers[0]["experts_desc"]
    heads = cfg.depth if cfg.self_predict else cfg.depth - 1
    if stack.chain and cluster:
        # layer-0 router and its top-K (unless layer 0 follows its own head),
        # one cluster launch per layer, the output sum, one ranking launch
        return (0 if cfg.self_predict else 2) + cfg.depth + 1 + (1 if heads > 0 else 0)
    if stack.chain:
        # layer-0 router (+ its top-K) when layer 0 routes itself or the shared
        # expert carries a gate/up adapter, A and B per layer, one ranking launch
        sh_gu = cfg.shared and any(ed.shared_lora[i].r for i in range(2))
        n = (1 if (not cfg.self_predict or sh_gu) else 0) + (0 if cfg.self_predict else 1)
        return n + 2 * cfg.depth + (1 if heads > 0 else 0)
    if stack.fused:
        return 1
    gu_lora = any(ed.lora[i].r for i in range(2)) or any(ed.shared_lora[i].r for i in range(2))
    ffn = 2 + (1 if gu_lora else 0)
    head = 1 + (1 if cfg.H else 0)
    n = 0
    for N in range(cfg.depth):
        if N == 0 and not cfg.self_predict:
            n += 1 + 1                      # router (H = 0 head) + top-K
        n += ffn + 1                        # experts + combine
        if N + 1 < cfg.depth or cfg.self_predict:
            n += head + 1                   # head + top-K
    return n


def run_native(args, cfg):
    import torch
    import torch.distributed as dist

    from int4_expert_gemv_gb300 import moe, synth
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    import __graft_entry__

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    __graft_entry__.build()

    dm = DeviceModel(cfg)
    moe.moe_decode_step_chain_variant(2 if args.path == "cluster" else 0, not args.no_l2_prefetch)
    st = DecodeStack(dm, fused={"chain": "chain", "cluster": "chain", "fused": True,
                                "per-call": False}[args.path])
    total = args.warmup + args.steps
    xin = torch.from_numpy(synth.gauss(cfg.seed, synth.tag(synth.X_INPUT, 0),
                                       (total + 64, cfg.d), 1.0)).cuda()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # the clock sampler runs from the warm-up to the end of the last timed leg
    clk = ClockSampler(local).__enter__()
    # step 0 (routers everywhere) eagerly, then capture the steady state
    st.step(xin[0])
    st.capture()
    for t in range(1, args.warmup):
        st.step(xin[t])
    torch.cuda.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.nvtx.range_push("timed")
    start.record(stream)
    for t in range(args.warmup, total):
        st.step(xin[t])
    stop.record(stream)
    torch.cuda.nvtx.range_pop()
    barrier()
    ms = max_over_ranks(start.elapsed_time(stop), world)
    tok_s = job_tokens_per_s(args.steps, world, ms)
    ms_step = ms / args.steps

    # ---- per-launch durations of the dominant kernel (instrumented replay of
    # further steps; external events become timing nodes inside the graph)
    t_next = total
    inst = {}
    for rot in range(3):
        g = torch.cuda.CUDAGraph()
        n_ev = 1 if st.fused else cfg.depth
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(n_ev)]
        with torch.cuda.graph(g):
            if st.fused:
                st.enqueue_fused_step(rot if rot else 3, events=evs[0])
            else:
                st.enqueue_step(rot if rot else 3, ffn_events=evs)
        inst[rot] = (g, evs)
    launch_ms = []
    n_inst = min(args.steps, 48)
    for i in range(n_inst):
        t = t_next + i
        st.xin.copy_(xin[t % xin.shape[0]])
        g, evs = inst[t % 3]
        g.replay()
        torch.cuda.synchronize()
        launch_ms += [a.elapsed_time(b) for a, b in evs]
    st.t = t_next + n_inst
    launch_avg_ms = statistics.mean(launch_ms)
    # algorithmic bytes of one timed unit: the expert weights it reads (the
    # chain's unit is the whole step -- events between its PDL-chained kernels
    # would serialise them -- and adds the head weights its kernels stream)
    unit_layers = cfg.depth if st.fused else 1
    launch_bytes = cfg.expert_bytes_per_layer() * unit_layers
    if st.chain:
        launch_bytes += dm.head_bytes_per_token() * cfg.depth

    # ---- end to end through the library: per step, the token's input from
    # pinned host memory (cudaMemcpyAsync), the decode call through the C ABI
    # (moe_decode_step_chain / moe_decode_step, or the per-layer calls),
    # the step's output back to pinned host memory
    pin_in = torch.from_numpy(synth.gauss(cfg.seed, synth.tag(synth.X_INPUT, 1),
                                          (args.steps, cfg.d), 1.0)).pin_memory()
    pin_out = torch.empty((args.steps, cfg.d), dtype=torch.float32).pin_memory()

    def e2e_leg(use_graphs: bool) -> float:
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            st.xin.copy_(pin_in[i], non_blocking=True)
            if use_graphs:
                st.graphs[st.t % 3].replay()
            elif st.fused:
                st.enqueue_fused_step(st.t)
            else:
                st.enqueue_step(st.t)
            st.t += 1
            pin_out[i].copy_(st.stream, non_blocking=True)
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), world)

    e2e_ms = e2e_leg(False)
    e2e_graph_ms = e2e_leg(True)
    # short runs: keep the GPU under the same load until the sampler has seen
    # at least ten samples (untimed)
    t_end = time.time() + 3.0
    while clk.samples() < 10 and time.time() < t_end:
        for _ in range(64):
            st.graphs[st.t % 3].replay()
            st.t += 1
        torch.cuda.synchronize()
    clk.__exit__(None, None, None)

    if rank == 0:
        hbm, hbm_kind = peaks()
        ffn_bytes = cfg.expert_bytes_per_layer()
        expert_gbs = ffn_bytes * cfg.depth / (ms_step / 1000.0) / 1e9
        achieved = launch_bytes / (launch_avg_ms / 1000.0) / 1e9
        head_bytes = dm.head_bytes_per_token()
        cluster = args.path == "cluster"
        if st.chain and cluster:
            kname = ("chain_c_kernel, one 16-CTA-cluster launch per layer (whole step: experts, "
                     f"combine, heads; {kernels_per_step(cfg, st, True)} PDL-chained launches)")
        elif st.chain:
            kname = ("chain_a_kernel + chain_b_kernel (whole step: experts, combine, heads; "
                     f"{kernels_per_step(cfg, st)} PDL-chained launches)")
        elif st.fused:
            kname = "decode_step_kernel (whole step: experts, combine, heads, top-K)"
        else:
            kname = "moe_expert_ffn_int4 (gate/up+SwiGLU, down)"
        line = {
            "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": path_dtype(cfg, args.path), "data": "synthetic",
            "config": {
                "workload": cfg.name, "batch": 1, "layers": cfg.depth, "d_model": cfg.d,
                "experts": cfg.E, "top_k": cfg.K, "expert_ffn": cfg.F,
                "shared_expert": cfg.shared, "weight_bits": cfg.bits, "group": cfg.group,
                "head_hidden": cfg.H, "head_prec": cfg.head_prec,
                "lora": f"r{cfg.lora_r} alpha{cfg.lora_alpha:g} {cfg.lora_on}" if cfg.lora_r else "none",
                "l2": (f"no flush: each step reads {cfg.depth * (ffn_bytes + head_bytes) / 1e6:.0f} MB "
                       f"of weights ({'>' if cfg.depth * (ffn_bytes + head_bytes) > L2_BYTES else '<'}"
                       f" {L2_BYTES / 1e6:.0f} MB L2); routed experts change every step"),
                "graphs": "steady-state steps replayed from captured CUDA graphs",
                "path": args.path,
            },
            "total_weight_gbs": (ffn_bytes + head_bytes) * cfg.depth / (ms_step / 1000.0) / 1e9,
            "expert_weight_gbs": expert_gbs,
            "expert_weight_frac_of_hbm": expert_gbs / hbm,
            "roofline": {"bound": "hbm", "kernel": kname,
                         "achieved": achieved, "peak": hbm, "peak_kind": hbm_kind,
                         "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": measured_traffic(cfg, args.path) if st.fused else None,
                         "bytes_per_launch": launch_bytes,
                         "avg_launch_us": launch_avg_ms * 1000.0,
                         "timing": (f"CUDA events around each whole step in {n_inst} "
                                    if st.fused else
                                    f"CUDA events around each layer's call in {n_inst} ")
                              + "instrumented graph replays after the timed region"},
            "e2e": {"value": job_tokens_per_s(args.steps, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": cfg.d * 4, "d2h_bytes_per_step": cfg.d * 4,
                    "how": "per step: cudaMemcpyAsync of x0 from pinned host memory, "
                           + ("one moe_decode_step_chain call" if st.chain else
                              "one moe_decode_step call" if st.fused else
                              "the per-layer C-ABI calls")
                           + " through the C ABI (no graph), out back to pinned host memory",
                    "graph_replay": {"value": job_tokens_per_s(args.steps, world, e2e_graph_ms),
                                     "unit": "tokens/s",
                                     "how": "the same copies around a replay of the step's "
                                            "captured CUDA graph"}},
            "gpu_launches": kernels_per_step(cfg, st, args.path == "cluster") * args.steps,
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_layers)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def grouped_kernels_per_call(cfg) -> int:
    """Kernels one batched expert-FFN call launches: sort (count, scatter),
    NaN fill, sums of x, [LoRA A x], gate/up GEMM, sums of h, [LoRA A_d h],
    down GEMM."""
    gu = cfg.lora_r and cfg.lora_on == "shared_all"
    dn = bool(cfg.lora_r)
    return 7 + (1 if gu else 0) + (1 if dn else 0)


def run_batched(args, cfg):
    """One step = one MoE layer over T tokens (bf16 input): the prerouter
    head and top-K over T rows, the expert FFN grouped by expert, and the
    combine + residual.  Replayed from a captured CUDA graph; L2 is flushed
    before every timed step (a small T touches fewer expert bytes than L2
    holds), each step timed by its own events."""
    import torch

    from int4_expert_gemv_gb300 import synth
    from int4_expert_gemv_gb300.model import BatchedLayer, DeviceModel
    import __graft_entry__

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    T = cfg.T
    from int4_expert_gemv_gb300 import moe
    moe.moe_debug_batched_engine({"auto": 0, "mma_sync": 1, "tcgen05": 2}[args.engine])
    dm = DeviceModel(cfg)
    bl = BatchedLayer(dm, T)
    x0 = torch.from_numpy(synth.gauss(cfg.seed, synth.tag(synth.X_INPUT, 0), (T, cfg.d), 1.0))
    bl.x.copy_(x0.cuda().to(torch.bfloat16))
    bl.res.copy_(x0.cuda())
    bl.route_own()
    torch.cuda.synchronize()
    cur = bl.cur_idx.cpu().numpy()
    distinct = len(set(cur.ravel().tolist()))

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bl.enqueue()
    ev = (torch.cuda.Event(enable_timing=True, external=True),
          torch.cuda.Event(enable_timing=True, external=True))
    gi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gi):
        bl.enqueue(ffn_events=ev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()

    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for a, b in pairs:
            flush.fill_(1)
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in pairs)
    ms_step = ms / args.steps
    tok_s = world * T * args.steps / (ms / 1000.0)

    # the FFN call alone (events inside an instrumented graph), L2 flushed
    ffn_ms = []
    for _ in range(min(args.steps, 32)):
        flush.fill_(1)
        gi.replay()
        torch.cuda.synchronize()
        ffn_ms.append(ev[0].elapsed_time(ev[1]))
    ffn_avg = statistics.mean(ffn_ms)

    # end to end: x (bf16) and the residual from pinned host memory, the
    # step, the layer output back to pinned host memory
    pin_x = bl.x.cpu().pin_memory()
    pin_r = bl.res.cpu().pin_memory()
    pin_o = torch.empty((T, cfg.d), dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        bl.x.copy_(pin_x, non_blocking=True)
        bl.res.copy_(pin_r, non_blocking=True)
        g.replay()
        pin_o.copy_(bl.out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    if rank == 0:
        hbm, hbm_kind = peaks()
        pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
        pk = json.load(open(pk_path)) if os.path.exists(pk_path) else {}
        tensor_peak = float(pk.get("bf16_tflops", 1900.0))
        tensor_kind = "measured" if "bf16_tflops" in pk else "fallback"
        ffn_bytes = (distinct + (1 if cfg.shared else 0)) * cfg.expert_bytes()
        ffn_flops = 2.0 * T * cfg.slots * 3 * cfg.d * cfg.F
        t_hbm = ffn_bytes / (hbm * 1e9)
        t_tc = ffn_flops / (tensor_peak * 1e12)
        tensor_bound = t_tc > t_hbm
        if tensor_bound:
            achieved, peak, unit = ffn_flops / (ffn_avg / 1000.0) / 1e12, tensor_peak, "TFLOP/s"
        else:
            achieved, peak, unit = ffn_bytes / (ffn_avg / 1000.0) / 1e9, hbm, "GB/s"
        head_k = 1 + (1 if cfg.H else 0)
        line = {
            "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": (f"int{cfg.bits}-g{cfg.group} weights (codes as exact bf16 on the tensor "
                      f"cores) x bf16 activations, fp32 accumulate"), "data": "synthetic",
            "config": {
                "workload": cfg.name, "batch": T, "layers": 1, "d_model": cfg.d,
                "experts": cfg.E, "top_k": cfg.K, "expert_ffn": cfg.F,
                "shared_expert": cfg.shared, "weight_bits": cfg.bits, "group": cfg.group,
                "head_hidden": cfg.H,
                "lora": f"r{cfg.lora_r} alpha{cfg.lora_alpha:g} {cfg.lora_on}" if cfg.lora_r else "none",
                "distinct_experts": distinct,
                "l2": "flushed (2x L2 written) before every timed step",
                "graphs": "each step replayed from a captured CUDA graph",
                "engine": args.engine,
            },
            "expert_weight_gbs": ffn_bytes / (ms_step / 1000.0) / 1e9,
            "ffn_tflops": ffn_flops / (ffn_avg / 1000.0) / 1e12,
            "roofline": {"bound": "tensor" if tensor_bound else "hbm",
                         "kernel": "moe_expert_ffn_int4, grouped (sort, gate/up GEMM, down GEMM)",
                         "achieved": achieved, "peak": peak,
                         "peak_kind": tensor_kind if tensor_bound else hbm_kind,
                         "unit": unit, "frac": achieved / peak, "traffic": None,
                         "bytes_per_launch": ffn_bytes, "flops_per_launch": ffn_flops,
                         "avg_launch_us": ffn_avg * 1000.0,
                         "timing": "CUDA events around the FFN call in an instrumented graph, "
                                   "L2 flushed before each"},
            "e2e": {"value": world * T * args.steps / (e2e_ms / 1000.0), "unit": "tokens/s",
                    "h2d_bytes_per_step": T * cfg.d * (2 + 4),
                    "d2h_bytes_per_step": T * cfg.d * 4},
            "gpu_launches": (head_k + 1 + grouped_kernels_per_call(cfg) + 1) * args.steps,
            "clocks": clk.summary(),
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(cfg, min(args.cpu_layers, 16))
        print(json.dumps(line), flush=True)


def run_merge(args, cfg):
    """One step = merging every layer's shared-expert adapters (gate, up,
    down) into its int4 weights and requantising them (moe_merge_lora, one
    launch per projection) into a second set of blobs; L2 is flushed before
    every timed step, each step timed by its own events.  Also reports the
    retention of layer 0's adapter delta through the merge."""
    import torch

    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DeviceModel, expert_sections, lora_merge_retention
    import __graft_entry__

    local = int(os.environ.get("LOCAL_RANK", "0"))
    rank = int(os.environ.get("RANK", "0"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    if not (cfg.shared and cfg.lora_r and cfg.lora_on == "shared_all"):
        raise SystemExit(f"--lora-merge needs a config with shared-expert adapters, not {cfg.name}")
    dm = DeviceModel(cfg, heads=False)
    secs = expert_sections(cfg)
    jobs = []          # (src, dst, row stride, rows, cols, LoraDesc)
    outs = [torch.empty_like(ly["shared"]) for ly in dm.layers]
    for ly, out in zip(dm.layers, outs):
        ed = ly["experts_desc"]
        for (off, stride, rows, cols), i in zip(secs, range(3)):
            l = ed.shared_lora[i]
            jobs.append((ly["shared"].data_ptr() + off, out.data_ptr() + off, stride, rows, cols, l))

    # the merges are independent: spread them over four streams (forked from
    # and joined back into the current one)
    lanes = [torch.cuda.Stream() for _ in range(4)]

    def step():
        main = torch.cuda.current_stream()
        for ls in lanes:
            ls.wait_stream(main)
        for i, (src, dst, stride, rows, cols, l) in enumerate(jobs):
            moe.moe_merge_lora(src, stride, rows, cols, cfg.bits, l.A, l.B, l.r, l.scale, dst, stride,
                               lanes[i % len(lanes)])
        for ls in lanes:
            main.wait_stream(ls)

    # algorithmic bytes: every record read and written once, A and B read once
    nbytes = sum(2 * rows * moe.moe_record_bytes(cols, cfg.bits) + 2 * l.r * (cols + rows)
                 for _, _, _, rows, cols, l in jobs)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    step()                                   # eager once, then one graph per step
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for a, b in pairs:
            flush.fill_(1)
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in pairs)
    ms_step = ms / args.steps
    gbs = nbytes / (ms_step / 1000.0) / 1e9
    ret = lora_merge_retention(dm, 0, 16)
    if rank == 0:
        hbm, hbm_kind = peaks()
        line = {
            "metric": "LoRA merge into the int4 weights (requantised per 64-group): GB/s",
            "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{cfg.name}: shared-expert adapters of {len(dm.layers)} layers "
                                   f"(r{cfg.lora_r}, gate/up/down)",
                       "l2": "flushed before every timed step",
                       "bytes_per_step": nbytes},
            "roofline": {"bound": "hbm", "kernel": "merge_lora_kernel", "achieved": gbs,
                         "peak": hbm, "peak_kind": hbm_kind, "unit": "GB/s", "frac": gbs / hbm,
                         "traffic": None, "bytes_per_launch": nbytes / len(jobs),
                         "timing": "CUDA events around each step (one graph of all launches "
                                   "of the step, spread over four streams)"},
            "retention": {k: v for k, v in ret.items() if k != "merged_blob"},
            "gpu_launches": len(jobs) * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)


def run_host_tier_chain(args, cfg):
    """Chained decode steps (captured graphs) with the routed experts in
    pinned host memory behind an LRU cache of --cache-slots experts per layer
    in HBM (HostTierChain), against the HBM-resident chained step; plus, per
    layer, when its cache update finishes against when the layer starts."""
    import torch

    from int4_expert_gemv_gb300 import synth
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel, HostTierChain
    import __graft_entry__

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    if int(os.environ.get("RANK", "0")) != 0:
        return
    dm = DeviceModel(cfg)
    stacks = {"hbm": DecodeStack(dm, fused="chain"),
              "host": HostTierChain(dm, args.cache_slots, args.free_sms, args.side_streams)}
    total = args.warmup + args.steps
    xin = torch.from_numpy(synth.gauss(cfg.seed, synth.tag(synth.X_INPUT, 0),
                                       (total + 1, cfg.d), 1.0)).cuda()
    stream = torch.cuda.current_stream()
    res = {}
    tier = stacks["host"]
    with ClockSampler(local) as clk:
        for name, st in stacks.items():
            st.step(xin[0])
            st.capture()
            for t in range(1, args.warmup + 1):
                st.step(xin[t])
            torch.cuda.synchronize()
            if st is tier:
                tier.stats.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for t in range(args.warmup + 1, total + 1):
                st.step(xin[t])
            b.record(stream)
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) / args.steps
        hits, misses = tier.stats.sum(0).tolist()
        # when each layer's update finishes (instrumented replays), against
        # the layer's start in the HBM-resident step (N x its per-layer time)
        n_rep = 8
        fin = [[] for _ in range(cfg.depth)]
        for r in range(n_rep):
            ev = (torch.cuda.Event(enable_timing=True, external=True),
                  [torch.cuda.Event(enable_timing=True, external=True) for _ in range(cfg.depth)])
            g = torch.cuda.CUDAGraph()
            t = tier.t
            with torch.cuda.graph(g):
                tier.enqueue_fused_step(t, update_events=ev)
            tier.xin.copy_(xin[r])
            g.replay()
            tier.t += 1
            torch.cuda.synchronize()
            for N in range(1, cfg.depth):
                fin[N].append(ev[0].elapsed_time(ev[1][N]))
    per_layer = res["hbm"] / cfg.depth
    slack = [N * per_layer - statistics.mean(fin[N]) for N in range(1, cfg.depth)]
    hidden = sum(1 for x in slack if x >= 0)
    moved = misses * tier.blob
    print(json.dumps({
        "metric": "decode tokens/s with the routed experts in host memory behind an HBM cache",
        "value": 1000.0 / res["host"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["host"], "higher_is_better": True,
        "data": "synthetic",
        "config": {"workload": cfg.name, "path": "chained step, captured graphs",
                   "cache_slots_per_layer": args.cache_slots, "free_sms": args.free_sms,
                   "side_streams": args.side_streams,
                   "cache_bytes": tier.cache.numel(),
                   "host_pool_bytes": sum(h.numel() for h in tier.host_pools)},
        "hbm_resident": {"ms_per_step": res["hbm"], "tokens_per_s": 1000.0 / res["hbm"]},
        "cache": {"hits": hits, "misses": misses, "hit_rate": hits / max(1, hits + misses),
                  "c2c_bytes_per_step": moved / args.steps,
                  "c2c_gbs": moved / (res["host"] * args.steps / 1000.0) / 1e9},
        "prefetch": {"layers_hidden": hidden, "layers": cfg.depth - 1,
                     "slack_ms_min": min(slack), "slack_ms_mean": statistics.mean(slack),
                     "note": "slack = layer N's start in the HBM-resident step (N x its per-layer "
                             "time) minus when layer N's cache update finished, from the step's "
                             "start, mean of 8 instrumented replays; >= 0: the copies hide"},
        "clocks": clk.summary()}), flush=True)


def run_host_tier(args, cfg):
    """Per-call decode steps (captured graphs) with the routed experts
    resident in HBM and with them in pinned host memory, gathered into HBM
    slots a token ahead from the predicted routes (HostTierStack); plus the
    gather alone (host -> HBM over NVLink-C2C)."""
    import torch

    from int4_expert_gemv_gb300 import moe, synth
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel, HostTierStack
    import __graft_entry__

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    __graft_entry__.build()
    if int(os.environ.get("RANK", "0")) != 0:
        return
    dm = DeviceModel(cfg)
    stacks = {"hbm": DecodeStack(dm), "host": HostTierStack(dm)}
    total = args.warmup + args.steps
    xin = torch.from_numpy(synth.gauss(cfg.seed, synth.tag(synth.X_INPUT, 0),
                                       (total + 1, cfg.d), 1.0)).cuda()
    stream = torch.cuda.current_stream()
    res = {}
    with ClockSampler(local) as clk:
        for name, st in stacks.items():
            st.step(xin[0])
            st.capture()
            for t in range(1, args.warmup + 1):
                st.step(xin[t])
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for t in range(args.warmup + 1, total + 1):
                st.step(xin[t])
            b.record(stream)
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) / args.steps
        # the gathers of one step alone (every layer's K experts), repeated
        tier = stacks["host"]
        reps = 8
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            for N in range(cfg.depth):
                tier.gather(N, tier.t - 1, stream)
        b.record(stream)
        torch.cuda.synchronize()
    g_ms = a.elapsed_time(b) / reps
    g_bytes = cfg.depth * cfg.K * tier.blob
    print(json.dumps({
        "metric": "decode tokens/s with the routed experts in host memory, gathered a token ahead",
        "value": 1000.0 / res["host"], "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["host"], "higher_is_better": True,
        "data": "synthetic",
        "config": {"workload": cfg.name, "path": "per-call kernels, captured graphs",
                   "host_pool_bytes": sum(h.numel() for h in tier.host_pools),
                   "gather_bytes_per_step": g_bytes},
        "hbm_resident": {"ms_per_step": res["hbm"], "tokens_per_s": 1000.0 / res["hbm"]},
        "gather_alone": {"ms_per_step": g_ms, "gbs": g_bytes / (g_ms / 1000.0) / 1e9,
                         "note": "host pinned memory -> HBM slots, read by the GPU over C2C"},
        "clocks": clk.summary()}), flush=True)


def run_agreement(args, cfg):
    """Predicted routes against the layers' own routers over seeded decode
    steps (per-call path): one JSON line with the agreement statistics."""
    import torch

    from int4_expert_gemv_gb300.model import DeviceModel, prediction_agreement
    import __graft_entry__

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    __graft_entry__.build()
    if int(os.environ.get("RANK", "0")) != 0:
        return
    res = prediction_agreement(DeviceModel(cfg, heads=True), steps=args.steps)
    print(json.dumps({"metric": "predicted route vs the layer's own router: mean K-set overlap",
                      "value": res["mean_overlap"], "unit": "fraction", "n_gpus": 1,
                      "steps": args.steps, "higher_is_better": True, "data": "synthetic",
                      "config": {"workload": cfg.name, "note": "random synthetic heads: "
                                 "a consistency measurement, no quality claim"},
                      "agreement": res}), flush=True)


def main():
    args = parse()
    from int4_expert_gemv_gb300.configs import ALL
    cfg = ALL[args.config]
    if args.steps is None:
        args.steps = (16 if args.impl == "reference" or args.lora_merge or args.route_agreement
                      else 200 if args.host_tier else (256 if cfg.T > 1 else 2400))
    if args.lora_merge:
        run_merge(args, cfg)
    elif args.route_agreement:
        run_agreement(args, cfg)
    elif args.host_tier:
        (run_host_tier_chain if args.path == "chain" else run_host_tier)(args, cfg)
    elif args.impl == "reference":
        import oracle
        oracle.build()
        run_reference(args, cfg)
    elif cfg.T > 1:
        run_batched(args, cfg)
    else:
        run_native(args, cfg)


if __name__ == "__main__":
    main()
