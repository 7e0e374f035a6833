"""Benchmark of the fused denoising-sampler step on GB300.

Workload: one 256-position canvas over V = 262,144 vocabulary entries with hidden
size d = 2,816 (synthetic, seeded; the shapes of the DiffusionGemma sampler).  A step
is one dg_sampler_step call: row statistics, entropy-bound acceptance and the
self-conditioning soft embedding.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle as it stands on the host cores, one whole canvas
(all 256 positions, full V and d) per step (the pages ship no runnable reference).

--gpus N > 1 runs one replica per GPU (independent canvases, no collective on the data
path): under torchrun (WORLD_SIZE set) each rank is one replica; without it the script
starts torchrun itself on 127.0.0.1.  --gpus must equal WORLD_SIZE.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "canvas positions/sec per fused sampler step (V=262144,d=2816); % of roofline"
UNIT = "positions/s"
WORKLOAD = "canvas256"
# kernels one timed step launches: the single pass's product, statistics merge, and reduce
# (which also runs the acceptance); the two-pass step: statistics, product, acceptance, reduce
KERNELS_PER_STEP = 3
KERNELS_PER_STEP_TWO_PASS = 4
# the tensor-bound workloads timed after the headline one (their own step, single pass and
# two passes)
DEFAULT_ALSO = "batch8,late_batch32"
# the denoising loop timed beside the step: a graph of 16 steps (the pages report 11 to 24
# denoising steps per canvas), convergence after two stable steps below 1 nat of mean
# entropy or at 24 steps
LOOP_STEPS = 16
LOOP_STABLE_STEPS = 2
LOOP_THRESHOLD = 1.0
LOOP_STEP_LIMIT = 24


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def config_of(wl) -> dict:
    """The workload a line is measured on; identical for the native and the reference arm."""
    return {"workload": f"{wl.name}: {wl.n_req} request x {wl.L_c} positions, V={wl.V}, d={wl.d}, "
                        f"fp32 logits, bf16 W, gamma={wl.gamma}",
            "rows": wl.R, "V": wl.V, "d": wl.d,
            "budget_nats": list(wl.budget) if isinstance(wl.budget, tuple) else wl.budget,
            "l2": "no flush: each step reads 1.62 GiB of logits and W, 13x the 129 MB L2"}


def source_sha(files=("soft_embed.cu", "dg_common.cuh")) -> str:
    """Hash of the soft-embed kernel's code (comments and blank space left out), so that
    stored ncu counters are used only for the kernel they were taken on."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "denoising_sampler_step_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def stored_traffic() -> dict:
    """The ncu DRAM traffic per call kept in profiles/, if it was taken on the current kernel
    source (else empty: the counters describe another kernel)."""
    tpath = os.path.join(ROOT, "profiles", "soft_embed_traffic.json")
    if not os.path.exists(tpath):
        return {}
    with open(tpath) as f:
        tj = json.load(f)
    return tj if tj.get("kernel_source_sha") == source_sha() else {}


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.proc = None
        self.gpu = gpu_index
        self.period_ms = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                pw.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None,
                "window": "from warm-up start to the end of the end-to-end loop"}


# --------------------------------------------------------------------------- CPU oracle legs

def oracle_seconds(x, Wb, wl, rows, budget):
    """Times the oracle on `rows` canvas positions: their statistics, their acceptance
    as one request, and their soft embeddings over the full vocabulary."""
    import numpy as np
    from oracle import entropy_accept, row_stats, soft_embed
    t0 = time.perf_counter()
    st = row_stats(x[rows])
    entropy_accept(st["H"], st["kappa"], 1, len(rows), np.array([budget], np.float32))
    soft_embed(x[rows], st["lse"], 0, wl.V, Wb, wl.gamma)
    return time.perf_counter() - t0


def cpu_baseline(x, Wb, wl, min_seconds: float = 10.0) -> dict:
    """Whole-canvas passes of the oracle, repeated until about min_seconds have passed."""
    import numpy as np
    rows = np.arange(wl.R)
    total, passes = 0.0, 0
    while passes == 0 or (total < min_seconds and passes < 8):
        total += oracle_seconds(x, Wb, wl, rows, float(wl.budget))
        passes += 1
    return {"value": passes * wl.R / total, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{passes} whole-canvas pass(es) of {wl.name} ({wl.R} positions, full V and d): fp64 "
                      f"statistics, acceptance and soft embedding, {total:.1f} s; numpy BLAS and the "
                      f"oracle's row pool on all host cores"}


def run_reference(args) -> None:
    """The oracle as it stands, one whole canvas per step (statistics, acceptance and the
    soft embedding of all 256 positions over the full vocabulary) on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from denoising_sampler_step_gb300 import inputs
    wl = inputs.WORKLOADS[WORKLOAD]
    x = inputs.logits(wl)
    Wb = inputs.embedding_bf16(wl)
    import numpy as np
    rows = np.arange(wl.R)
    for _ in range(args.warmup):
        oracle_seconds(x, Wb, wl, rows, float(wl.budget))
    times = [oracle_seconds(x, Wb, wl, rows, float(wl.budget)) for _ in range(args.steps)]
    total = sum(times)
    value = wl.R * args.steps / total
    sample = (f"{args.steps} whole-canvas steps of {wl.name} ({wl.R} positions each, full V and d): fp64 "
              f"statistics, acceptance and soft embedding, {total:.1f} s; numpy BLAS and the oracle's row "
              f"pool on all host cores")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm

def other_configs(args, dev, B, inputs, SamplerStep, cost) -> dict:
    """The step at further workloads (fresh inputs each): ms per step, the product's tensor
    rate and the fraction of the step roofline, single pass and two passes."""
    import numpy as np
    import torch
    pk = peaks()
    res = {}
    for name in [n for n in args.also.split(",") if n]:
        wl = inputs.WORKLOADS[name]
        xd = torch.from_numpy(inputs.logits(wl)).to(dev)
        Wd = torch.from_numpy(inputs.embedding_bf16(wl).view(np.int16)).to(dev).view(torch.bfloat16)
        bd = torch.from_numpy(inputs.budgets(wl)).to(dev)
        sc = cost.StepCost(rows=wl.R, V=wl.V, d=wl.d, vocab=wl.V)
        t_roof = sc.roofline_seconds(pk["hbm_gbs"], pk["bf16_tflops"])
        t_roof_sus = sc.roofline_seconds(pk["hbm_gbs"], pk["bf16_tflops_sustained"] or pk["bf16_tflops"])
        n = max(3, min(args.steps, int(2000 // max(1, wl.R // 256))))
        out = {"rows": wl.R, "steps": n, "t_roof_us": t_roof * 1e6,
               "bound": "tensor" if sc.flops / (pk["bf16_tflops"] * 1e12) >= t_roof * 0.999 else "hbm",
               "config": config_of(wl)}
        for mode in ("single_pass", "two_pass"):
            st = SamplerStep(Wd, wl.n_req, wl.L_c, wl.V, wl.gamma, device=dev, two_pass=mode == "two_pass")
            for _ in range(3):
                st(xd, bd)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                st(xd, bd)
            e1.record()
            torch.cuda.synchronize(dev)
            B.dg_get_device_status()
            ms = e0.elapsed_time(e1) / n
            out[mode] = {"ms_per_step": ms, "positions_per_s": wl.R / (ms * 1e-3),
                         "tflops": sc.flops / (ms * 1e-3) / 1e12,
                         "frac": t_roof / (ms * 1e-3), "frac_sustained_peak": t_roof_sus / (ms * 1e-3)}
            del st
        res[name] = out
        del xd, Wd
        torch.cuda.empty_cache()
    return res


def run_sharded(args) -> None:
    """The vocabulary-parallel step (calvarado04.com, "The fix" and "Why not just all-gather the
    weights"): rank r of N holds the logit columns and W rows of vocabulary shard r; per step
    it summarises its rows, all-gathers the 16-byte summaries, combines them in shard order,
    accepts, forms its partial embedding against the global lse and all-gathers the partials,
    which every rank adds in shard order.  One canvas per step over all ranks (strong scaling);
    N = 1 runs the same code over a one-rank NCCL group."""
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{args.master_port}", rank=0, world_size=1,
                                device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build()
    from denoising_sampler_step_gb300 import binding as B
    from denoising_sampler_step_gb300 import inputs
    from denoising_sampler_step_gb300.vocab_parallel import ShardedStep, TorchComm, shard_bounds

    wl = inputs.WORKLOADS[WORKLOAD]
    dev = torch.device("cuda", local)
    s, e = shard_bounds(wl.V, world)[rank]
    x = inputs.logits(wl)  # every rank draws the same canvas and keeps its columns
    Wb = inputs.embedding_bf16(wl)
    shard = torch.from_numpy(np.ascontiguousarray(x[:, s:e])).to(dev)
    Wsh = torch.from_numpy(np.ascontiguousarray(Wb[s:e]).view(np.int16)).to(dev).view(torch.bfloat16)
    bd = torch.from_numpy(inputs.budgets(wl)).to(dev)
    del x, Wb
    comm = TorchComm()
    st = ShardedStep(wl.n_req, wl.L_c, wl.gamma)
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        st.rank_step(shard, s, Wsh, bd, comm)
    torch.cuda.synchronize(dev)
    dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        st.rank_step(shard, s, Wsh, bd, comm)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    # the same rank step, 16 of them captured in one CUDA graph (NCCL collectives included) and
    # replayed: the eager loop above issues each step's launches and collectives from Python,
    # which at one rank takes about as long as the GPU work itself
    gms = None
    graph_error = None
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            st.rank_step(shard, s, Wsh, bd, comm)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for _ in range(LOOP_STEPS):
                st.rank_step(shard, s, Wsh, bd, comm)
        g.replay()
        torch.cuda.synchronize(dev)
        dist.barrier()
        reps = max(1, -(-args.steps // LOOP_STEPS))
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
        gm = torch.tensor([g0.elapsed_time(g1) / (reps * LOOP_STEPS)], device=dev)
        dist.all_reduce(gm, op=dist.ReduceOp.MAX)
        gms = gm.item()
        del g
    except Exception as ex:  # report, do not hide the eager number
        graph_error = str(ex)[:200]
    clk = clocks.stop()
    mx = torch.tensor([t0.elapsed_time(t1)], device=dev)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    ms = mx.item()
    B.dg_get_device_status()
    if rank == 0:
        line = {
            "metric": METRIC, "value": wl.R * args.steps / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "mode": "sharded",
            "dtype": "f32 statistics, bf16 x bf16 -> f32 tensor-core product", "data": "synthetic",
            "config": config_of(wl),
            "parallelism": f"vocabulary-parallel over {world} rank(s): shard [{s}, {e}) on rank 0; NCCL "
                           "all-gathers of the row summaries and of the partial embeddings",
            "all_gather_bytes_per_rank_per_step": {"row_summaries": world * wl.R * 16,
                                                    "partial_embeddings": world * wl.R * wl.d * 4},
            "gpu_launches": 6 * args.steps,
            "clocks": clk,
            "graph": ({"ms_per_step": gms, "value": wl.R / (gms * 1e-3),
                       "how": f"{LOOP_STEPS} rank steps (their NCCL all-gathers included) captured in one "
                              "CUDA graph and replayed; max over ranks"}
                      if gms is not None else {"ms_per_step": None, "error": graph_error}),
        }
        print(json.dumps(line))
    dist.destroy_process_group()


def spawn_ranks(args) -> int:
    """--gpus N > 1 without torchrun: start torchrun on 127.0.0.1 with N ranks running this
    script (same arguments) and return its exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(args.master_port), os.path.abspath(__file__)]
    cmd += sys.argv[1:]
    return subprocess.call(cmd)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--also", default=DEFAULT_ALSO,
                    help="comma-separated further workloads whose step is timed after the main one and "
                         "reported under other_configs (single pass and two passes); '' for none")
    ap.add_argument("--master-port", type=int, default=29531,
                    help="rendezvous port when --gpus N > 1 starts its own ranks")
    ap.add_argument("--only", choices=["soft_embed", "step", "soft_embed_e4m3", "step_e4m3"], default=None,
                    help="profiling target: run only this call (warm-up, then --steps calls) and print "
                         "its mean duration; no JSON line")
    ap.add_argument("--mode", default="replicas", choices=["replicas", "sharded"],
                    help="replicas: each rank steps its own canvas (the driver's line); sharded: the "
                         "vocabulary-parallel step over all ranks, one canvas per step (NCCL all-gathers)")
    ap.add_argument("--sustained", type=float, default=0.0,
                    help="also run the step and the soft-embed call back to back for this many seconds "
                         "each, sampling clocks and power every 20 ms")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args))
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if world_env != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world_env}: start one rank per GPU")
    if args.impl == "reference":
        run_reference(args)
        return
    if args.mode == "sharded":
        run_sharded(args)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    import __graft_entry__
    __graft_entry__.build()
    from denoising_sampler_step_gb300 import binding as B
    from denoising_sampler_step_gb300 import cost, inputs, replicas
    from denoising_sampler_step_gb300.step import SamplerStep

    # each rank serves its own canvases (independent requests: weak scaling)
    wl = replicas.rank_workload(inputs.WORKLOADS[WORKLOAD], rank)
    x = inputs.logits(wl)
    Wb = inputs.embedding_bf16(wl)
    budgets = inputs.budgets(wl)
    dev = torch.device("cuda", local)
    xd = torch.from_numpy(x).to(dev)
    Wd = torch.from_numpy(Wb.view(np.int16)).to(dev).view(torch.bfloat16)
    bd = torch.from_numpy(budgets).to(dev)
    step = SamplerStep(Wd, wl.n_req, wl.L_c, wl.V, wl.gamma, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.only:
        # a short, fixed launch sequence for a profiler: warm-up calls, then --steps calls
        if args.only == "soft_embed":
            lse = B.dg_row_stats(xd)["lse"]
            call = lambda: B.dg_soft_embed(xd, lse, 0, wl.V, Wd, wl.gamma, out=step.out["E"], ws=step.ws)
        elif args.only in ("soft_embed_e4m3", "step_e4m3"):
            # the 8-bit table: the bf16 table quantised per row once (before the calls)
            Qd, sd = B.dg_quantize_e4m3(Wd)
            ws8 = B.workspace_e4m3(wl.R, wl.V, wl.d, dev)
            lse = B.dg_row_stats(xd)["lse"]
            if args.only == "soft_embed_e4m3":
                call = lambda: B.dg_soft_embed_e4m3(xd, lse, 0, wl.V, Qd, sd, wl.gamma, out=step.out["E"], ws=ws8)
            else:
                call = lambda: B.dg_sampler_step_e4m3(xd, wl.n_req, wl.L_c, Qd, sd, wl.gamma, bd, ws=ws8)
        else:
            call = lambda: step(xd, bd)
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize(dev)
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        for _ in range(args.steps):
            call()
        o1.record(stream)
        torch.cuda.synchronize(dev)
        B.dg_get_device_status()
        if rank == 0:
            print(f"{args.only}: {o0.elapsed_time(o1) / args.steps * 1e3:.1f} us per call "
                  f"({args.warmup} warm-up + {args.steps} calls)", flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step(xd, bd)
    B.dg_get_device_status()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(xd, bd)
    ev1.record(stream)
    barrier()
    ms = ev0.elapsed_time(ev1)
    B.dg_get_device_status()

    # each step timed on its own (events around every call, no synchronisation between
    # calls): the median and the minimum the timing protocol asks for beside the mean
    pairs = []
    for _ in range(min(args.steps, 50)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(xd, bd)
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize(dev)
    per = sorted(a.elapsed_time(b) for a, b in pairs)
    per_step = {"n": len(per), "median_ms": per[len(per) // 2], "min_ms": per[0], "max_ms": per[-1]}

    # the same step captured once in a CUDA graph and replayed (launches replayed as one
    # graph, the overlaps kept as programmatic edges)
    graph = {"ms_per_step": None}
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step(xd, bd)  # warm the capture stream
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(xd, bd)
        for _ in range(3):
            g.replay()
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        barrier()
        gms = replicas.max_over_ranks([g0.elapsed_time(g1)], device=dev)[0]
        B.dg_get_device_status()
        graph = {"ms_per_step": gms / args.steps,
                 "value": world * wl.R * args.steps / (gms * 1e-3),
                 "how": "one dg_sampler_step captured in a CUDA graph, replayed K times"}
    except Exception as ex:  # report, do not hide the eager numbers
        graph = {"ms_per_step": None, "error": str(ex)[:200]}

    # the denoising loop: LOOP_STEPS loop steps (the step over the eligible positions,
    # then the loop-state update) captured in one CUDA graph and replayed; the loop state
    # advances across replays, the work per step does not change.  Timed twice: with the
    # argmax on the canvas, and with candidates drawn at temperature 1 (the statistics and
    # the draw in one pass over the logits)
    def time_loop(temperature):
        from denoising_sampler_step_gb300.step import SamplerLoop
        lp = SamplerLoop(Wd, wl.n_req, wl.L_c, wl.V, wl.gamma, LOOP_STABLE_STEPS, LOOP_THRESHOLD,
                         LOOP_STEP_LIMIT, temperature=temperature, seed=1, min_accept=1, device=dev)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            lp(xd, bd)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)
        lg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(lg, stream=cap):
            for _ in range(LOOP_STEPS):
                lp(xd, bd)
        lp.reset()
        lg.replay()
        barrier()
        reps = max(1, -(-args.steps // LOOP_STEPS))
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        for _ in range(reps):
            lg.replay()
        l1.record(stream)
        barrier()
        lms = replicas.max_over_ranks([l0.elapsed_time(l1)], device=dev)[0]
        B.dg_get_device_status()
        n_loop = reps * LOOP_STEPS
        res = {"ms_per_step": lms / n_loop, "steps": n_loop,
               "value": world * wl.R * n_loop / (lms * 1e-3),
               "converged_requests": int(lp.state["converged"].sum().item()),
               "params": {"stable_steps": LOOP_STABLE_STEPS, "entropy_threshold": LOOP_THRESHOLD,
                          "step_limit": LOOP_STEP_LIMIT, "min_accept": 1, "temperature": temperature},
               "how": f"{LOOP_STEPS} dg_sampler_loop_step calls captured in one CUDA graph, replayed "
                      f"{reps} times on the same logits"}
        del lp, lg
        return res

    loop, loop_sampled = {"ms_per_step": None}, {"ms_per_step": None}
    try:
        loop = time_loop(0.0)
        loop_sampled = time_loop(1.0)
    except Exception as ex:
        err = {"ms_per_step": None, "error": str(ex)[:200]}
        loop = loop if loop.get("ms_per_step") else err
        loop_sampled = err

    # per-call durations on the launching stream: each entry point called back to back
    # (same inputs, same shapes), the mean over the loop
    out = step.out
    nrep = max(args.steps, 10)
    sample_out = {"candidate": torch.empty(wl.R, dtype=torch.int32, device=dev),
                  "log_p": torch.empty(wl.R, dtype=torch.float32, device=dev)}
    calls = {
        "row_stats": lambda: B.dg_row_stats(xd, stream=stream, out=out),
        "accept": lambda: B.dg_entropy_accept(out["H"], out["kappa"], wl.n_req, wl.L_c, bd,
                                              stream=stream, out=out),
        "soft_embed": lambda: B.dg_soft_embed(xd, out["lse"], 0, wl.V, Wd, wl.gamma, out=out["E"],
                                              ws=step.ws, stream=stream),
        # the stochastic-candidate pass (not part of the argmax step; reported alongside)
        "row_sample": lambda: B.dg_row_sample(xd, 1.0, seed=1, offset=0, stream=stream, out=sample_out),
        # the statistics and the draw in one pass (the sampling loop's first kernel)
        "row_stats_sample": lambda: B.dg_row_stats_sample(xd, 1.0, seed=1, offset=0, stream=stream,
                                                          out=dict(sample_out, **{k: out[k] for k in
                                                                                  ("m", "lse", "H", "kappa",
                                                                                   "argmax")})),
    }
    comp = {}
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, call in calls.items():
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        k0.record(stream)
        for _ in range(nrep):
            call()
        k1.record(stream)
        torch.cuda.synchronize(dev)
        comp[name] = k0.elapsed_time(k1) / nrep

    # the same step and product over the 8-bit table (the bf16 table quantised per row to
    # E4M3 on the device): half the table's bytes, block-scaled E4M3 MMAs
    e4m3 = {"ms_per_step": None}
    try:
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        Qd, sd = B.dg_quantize_e4m3(Wd, stream=stream)
        q1.record(stream)
        torch.cuda.synchronize(dev)
        ws8 = B.workspace_e4m3(wl.R, wl.V, wl.d, dev)
        o8 = {k: torch.empty_like(v) for k, v in out.items()}
        e4calls = {
            "step": lambda: B.dg_sampler_step_e4m3(xd, wl.n_req, wl.L_c, Qd, sd, wl.gamma, bd, out=o8, ws=ws8,
                                                   stream=stream),
            "soft_embed": lambda: B.dg_soft_embed_e4m3(xd, out["lse"], 0, wl.V, Qd, sd, wl.gamma, out=o8["E"],
                                                       ws=ws8, stream=stream),
        }
        t8 = {}
        for name, call in e4calls.items():
            for _ in range(3):
                call()
            torch.cuda.synchronize(dev)
            k0.record(stream)
            for _ in range(nrep):
                call()
            k1.record(stream)
            torch.cuda.synchronize(dev)
            t8[name] = k0.elapsed_time(k1) / nrep
        B.dg_get_device_status()
        sc8 = cost.StepCost(rows=wl.R, V=wl.V, d=wl.d, vocab=wl.V)
        pk8 = peaks()
        a8 = sc8.e4m3_gemm_bytes / (t8["soft_embed"] * 1e-3) / 1e9
        tr8 = stored_traffic().get("e4m3_traffic_bytes_per_launch")
        e4m3 = {"ms_per_step": t8["step"], "value": world * wl.R / (t8["step"] * 1e-3), "unit": UNIT,
                "soft_embed_us": t8["soft_embed"] * 1e3,
                "roofline": {"kernel": "soft_embed over the 8-bit table (block-scaled E4M3 product + reduce)",
                             "bound": "hbm", "achieved": a8, "peak": pk8["hbm_gbs"], "unit": "GB/s",
                             "frac": a8 / pk8["hbm_gbs"], "traffic": tr8,
                             "algorithmic_bytes_per_launch": sc8.e4m3_gemm_bytes,
                             "note": "the high/low split of A gives each vocabulary block the MMA time of a "
                                     "bf16 block; the product is bound by the tensor pipe sharing the SM with "
                                     "the rest of the pipeline, not by its bytes"},
                # the tensor pipe's view: the high and low E4M3 parts make the MMA work twice the
                # product's 2 R V d, at the E4M3 rate (the measured bf16 peak times the nominal
                # E4M3 : bf16 ratio of 2)
                "roofline_tensor": {"kernel": "soft_embed over the 8-bit table: its block-scaled E4M3 MMAs",
                                    "bound": "tensor", "mma_flops_per_launch": 2 * sc8.flops,
                                    "achieved": 2 * sc8.flops / (t8["soft_embed"] * 1e-3) / 1e12,
                                    "peak": 2 * pk8["bf16_tflops"], "unit": "TFLOP/s",
                                    "frac": 2 * sc8.flops / (t8["soft_embed"] * 1e-3) / 1e12
                                            / (2 * pk8["bf16_tflops"]),
                                    "peak_source": pk8["source"] + " bf16 x 2 (nominal E4M3 : bf16)"},
                "table_bytes": sc8.e4m3_table_bytes, "bf16_table_bytes": sc8.w_bytes,
                "quantize_ms": q0.elapsed_time(q1),
                "how": "dg_sampler_step_e4m3 (single pass) and dg_soft_embed_e4m3 called back to back, "
                       "mean over the loop; the table quantised once by dg_quantize_e4m3 (timed)"}
        del Qd, sd, ws8, o8
    except Exception as ex:  # report, do not hide the other numbers
        e4m3 = {"ms_per_step": None, "error": str(ex)[:200]}

    # end to end through the public API: pinned host inputs in, results out, every step
    h = step.host_buffers()
    h["logits"].copy_(torch.from_numpy(x))
    h["budgets"].copy_(torch.from_numpy(budgets))
    step.run_pipelined(h, 3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    step.run_pipelined(h, args.steps)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    clk = clocks.stop()

    ms, e2e_ms = replicas.max_over_ranks([ms, e2e_ms], device=dev)

    # sustained operation: the clock the power cap allows when a call runs for seconds
    sustained = None
    if args.sustained > 0:
        sustained = {}
        for name, call, t_ms in (("step", lambda: step(xd, bd), ms / args.steps),
                                 ("soft_embed", calls["soft_embed"], comp["soft_embed"])):
            n = max(10, int(args.sustained * 1e3 / t_ms))
            sampler = ClockSampler(local, period_ms=20)
            sampler.start()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(n):
                call()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            c = sampler.stop()
            sustained[name] = {"ms_per_call": s0.elapsed_time(s1) / n, "calls": n, "sm_mhz": c["sm_mhz"],
                               "power_w": c["power_w"], "reasons": c["reasons"], "samples": c["samples"]}
        B.dg_get_device_status()

    pk = peaks()
    sc = cost.StepCost(rows=wl.R, V=wl.V, d=wl.d, vocab=wl.V)
    t_roof = sc.roofline_seconds(pk["hbm_gbs"], pk["bf16_tflops"])
    ms_step = ms / args.steps
    # the kernels one step runs (the single pass: the product with the statistics folded, the
    # statistics merge, the redo pass, the split-K reduce, the acceptance), timed together as
    # the step, against the step's algorithmic bytes; the plain product call beside it
    achieved_step = sc.step_bytes / (ms_step * 1e-3) / 1e9
    achieved = sc.gemm_bytes / (comp["soft_embed"] * 1e-3) / 1e9
    tj = stored_traffic()
    traffic, traffic_step = tj.get("traffic_bytes_per_launch"), tj.get("step_traffic_bytes")
    line = {
        "metric": METRIC,
        "value": replicas.whole_job_rate(wl.R, args.steps, world, ms),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 statistics, bf16 x bf16 -> f32 tensor-core product",
        "data": "synthetic",
        "config": config_of(wl),
        "parallelism": f"replicas x{world} (independent canvases per GPU, no collective on the data path)",
        "step_roofline": {"t_roof_us": t_roof * 1e6, "t_step_us": ms_step * 1e3,
                          "frac": t_roof / (ms_step * 1e-3), "peaks": pk["source"]},
        "roofline": {"kernel": "dg_sampler_step, single pass: soft_embed_kernel<0> with the statistics "
                               "folded (the dominant kernel), the statistics merge, the split-K reduce with "
                               "the acceptance in its first CTA; one call", "bound": "hbm",
                     "achieved": achieved_step, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_step / pk["hbm_gbs"], "traffic": traffic_step,
                     "algorithmic_bytes_per_launch": sc.step_bytes, "launch_us": ms_step * 1e3,
                     "peak_source": pk["source"], "timed": "CUDA events around the timed steps"},
        "roofline_product": {"kernel": "dg_soft_embed (soft_embed_kernel<0> + split-K reduce), statistics given",
                             "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                             "algorithmic_bytes_per_launch": sc.gemm_bytes,
                             "launch_us": comp["soft_embed"] * 1e3, "peak_source": pk["source"]},
        "kernel_us": {k: v * 1e3 for k, v in comp.items()},
        "e2e": {"value": replicas.whole_job_rate(wl.R, args.steps, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": step.h2d_bytes(h), "d2h_bytes_per_step": step.d2h_bytes(),
                "ms_per_step": e2e_ms / args.steps,
                "how": "SamplerStep.run_pipelined: each step uploads its logits from pinned host memory "
                       "(overlapping the previous step's kernels) and reads every result back"},
        "per_step": per_step,
        "graph": graph,
        "loop": loop,
        "loop_sampled": loop_sampled,
        "e4m3_table": e4m3,
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clk,
    }
    if sustained is not None:
        line["sustained"] = sustained
    if args.also and not args.sustained:
        line["other_configs"] = other_configs(args, dev, B, inputs, SamplerStep, cost)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x, Wb, wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
