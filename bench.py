#!/usr/bin/env python
"""Benchmark of the quantized MoE layer forward (ds4moe) on GB300.

One step = one full forward (router, bucketing, gate/up + SwiGLU, down, combine, shared
expert) over one batch of synthetic tokens, inputs resident in HBM. L2 is flushed between
steps (a write of twice the L2 size, outside the timed events). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

--config picks the headline workload (default 4: prefill of 4096 tokens, d=4096, 256 experts,
top-8, f=2048, Q2_K routed + Q8_0 shared, the first 1024 tokens table-routed: the largest
single-GPU workload, tensor-core bound). Every other workload (tiny-q8, decode-1, decode-16,
prefill-512) is timed in the same run and reported under detail.per_config, each with its own
roofline (HBM for decode). Under torchrun each rank runs an independent replica on its own
tokens (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")  # the CPU baseline is the single-threaded oracle

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "MoE layer tok/s; decode weight GB/s vs HBM peak; prefill TFLOP/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            pk = json.load(fh)
        return dict(hbm=float(pk["hbm_gbs"]), bf16=float(pk["bf16_tflops"]),
                    bf16_sus=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sus=1700.0, src="fallback")


def workload_name(spec: synthetic.Spec) -> str:
    s = spec
    txt = (f"{s.name}: {s.n_tokens} tokens, d={s.d}, {s.n_experts} experts top-{s.top_k}, f={s.f}, "
           f"{s.fmt_gate_up}/{s.fmt_down} routed, {s.n_shared} {s.fmt_shared} shared f={s.f_shared}")
    if s.bias:
        txt += f", {s.bias} router bias"
    if s.n_hash:
        txt += f", first {s.n_hash} table-routed"
    return txt


# ------------------------------------------------------------------ algorithmic work

def weight_bytes(spec, distinct: int) -> dict:
    mgu = synthetic.row_bytes(spec.fmt_gate_up, spec.d) * spec.f
    md = synthetic.row_bytes(spec.fmt_down, spec.f) * spec.d
    shared = 0
    if spec.n_shared:
        shared = 2 * synthetic.row_bytes(spec.fmt_shared, spec.d) * spec.f_shared + \
            synthetic.row_bytes(spec.fmt_shared, spec.f_shared) * spec.d
    router = spec.n_experts * spec.d * 4 if spec.n_tokens > spec.n_hash else 0
    return dict(routed_gateup=distinct * 2 * mgu, routed_down=distinct * md, shared=shared, router=router,
                x=spec.n_tokens * spec.d * 2, out=spec.n_tokens * spec.d * 4)


def forward_flops(spec) -> float:
    per_pair = 2.0 * spec.d * spec.f * 3
    shared = 2.0 * spec.d * spec.f_shared * 3 if spec.n_shared else 0.0
    learned = spec.n_tokens - spec.n_hash
    return spec.n_tokens * (spec.top_k * per_pair + shared) + learned * 2.0 * spec.n_experts * spec.d


# Source files that decide each timed kernel's code: a recorded DRAM traffic figure stays valid
# while these files are unchanged.
KERNEL_SOURCES = {
    "decode": ("decode.cu", "mma_units.cuh", "common.cuh"),
    "gemm": ("gemm_tc.cu", "tc_ptx.cuh", "common.cuh"),
}
TRAFFIC_FAMILY = {"route": "decode", "gateup": "decode", "down_combine": "decode",
                  "routed_gateup": "gemm", "shared_gateup": "gemm", "routed_down": "gemm", "shared_down": "gemm"}


def kernel_source_hash(family: str | None = None) -> str:
    """sha256 prefix over the CUDA sources: all of csrc, or one kernel family's files."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_moe_gb300", "csrc")
    names = KERNEL_SOURCES[family] if family else sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = rec.get(f"{workload}:{kernel}")
    fam = TRAFFIC_FAMILY.get(kernel)
    if not ent or not fam or ent.get("source_hash") != kernel_source_hash(fam):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.tmp.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.tmp.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU baseline (oracle)

def oracle_token(problem, spec, xb, n):
    """fp64 oracle forward of token n of the batch xb (table-routed when n < n_hash)."""
    from oracle import moe
    nh = 1 if n < spec.n_hash else 0
    tid = problem.token_ids[n:n + 1] if nh else None
    return moe.forward(problem, x_bits=xb[n:n + 1], token_ids=tid, n_hash=nh)


def oracle_sample(spec, problem, seconds: float, min_tokens: int = 1):
    """Runs the fp64 oracle on successive tokens of the workload until `seconds` elapse."""
    xb = synthetic.activations(spec, max(spec.n_tokens, 256))
    n = 0
    t0 = time.perf_counter()
    while n < min_tokens or time.perf_counter() - t0 < seconds:
        if n >= xb.shape[0]:
            break
        oracle_token(problem, spec, xb, n)
        n += 1
    dt = time.perf_counter() - t0
    return n, dt


def run_reference(args, spec, rank):
    if rank != 0:
        return
    problem = synthetic.make_problem(spec)
    xb = synthetic.activations(spec, max(spec.n_tokens, 256))
    # one step = one token of the workload through the oracle (bounded sample)
    tok = 0

    def step():
        nonlocal tok
        oracle_token(problem, spec, xb, tok % xb.shape[0])
        tok += 1

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(spec), "sample": "one token per step"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} single-token forwards of the workload, fp64 numpy, 1 thread"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks (host logic)

def batch_seed(spec: synthetic.Spec, rank: int, batch: int, batches: int) -> int:
    """Seed of input batch `batch` on `rank`: every rank draws its own tokens (replicas share weights)."""
    return spec.seed + 7919 * (rank * batches + batch + 1)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's value (timings are reduced with MAX; world 1 returns the value)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_step: int, steps: int, seconds: float) -> float:
    """Tokens per second of all ranks together: every rank runs `steps` steps of its own tokens."""
    return world * tokens_per_step * steps / seconds


# ------------------------------------------------------------------ GPU arm

def kernel_work(spec, distinct: float) -> dict:
    """Algorithmic work of each timed phase: bytes (decode path, HBM-bound) or FLOPs (expert GEMMs)."""
    wb = weight_bytes(spec, distinct)
    pair = 2.0 * spec.d * spec.f
    nb = {"routed_gateup": wb["routed_gateup"] + wb["x"], "routed_down": wb["routed_down"],
          "shared_gateup": wb["shared"] * 2 / 3 + wb["x"], "shared_down": wb["shared"] / 3,
          "router_logits": wb["router"] + wb["x"], "combine": wb["out"],
          # decode path: route; gate/up of the touched and the shared experts; down + combine
          "route": wb["router"] + wb["x"],
          "gateup": wb["routed_gateup"] + wb["shared"] * 2 / 3 + wb["x"],
          "down_combine": wb["routed_down"] + wb["shared"] / 3 + wb["out"]}
    fl = {"routed_gateup": spec.n_tokens * spec.top_k * 2 * pair, "routed_down": spec.n_tokens * spec.top_k * pair,
          "shared_gateup": spec.n_tokens * 2 * 2.0 * spec.d * spec.f_shared,
          "shared_down": spec.n_tokens * 2.0 * spec.d * spec.f_shared}
    return dict(bytes=nb, flops=fl, weights=wb)


def measure(api, spec, args, dev, stream, rank, world, peaks, l2_mode, with_e2e=True):
    """Creates the workload's handle (and, in `layer` mode, a second layer), times K forwards with
    CUDA events (L2 prepared between steps, outside the events), then a profiled pass (per-launch
    times) and the end-to-end host-buffer pass. Returns a dict of raw measurements."""
    import torch

    problem = synthetic.make_problem(spec)
    shapes = api.make_shapes(spec.d, spec.f, spec.f_shared, spec.n_experts, spec.top_k, spec.n_shared,
                             spec.fmt_gate_up, spec.fmt_down, spec.fmt_shared, problem.router_b is not None,
                             spec.hash_vocab, spec.n_tokens, dev.index)
    arrays = [problem.router_w, problem.router_b, problem.gate.full(), problem.up.full(), problem.down.full(),
              problem.shared_gate, problem.shared_up, problem.shared_down, problem.hash_table]
    h = api.ds4moe_create(api.make_weights(*arrays), shapes)
    del arrays
    # A second layer of the same shape with its own weights: between timed steps it runs once
    # after the L2 flush, as the previous layer of a model would, so the kernels' code is warm
    # while every byte of the timed layer's data is cold.
    h_prev = None
    if l2_mode == "layer":
        pp = synthetic.make_problem(spec.with_(seed=spec.seed + 1000003))
        arrays = [pp.router_w, pp.router_b, pp.gate.full(), pp.up.full(), pp.down.full(), pp.shared_gate,
                  pp.shared_up, pp.shared_down, pp.hash_table]
        h_prev = api.ds4moe_create(api.make_weights(*arrays), shapes)
        del arrays, pp

    # per-rank input batches (different tokens per step, and per rank)
    xs, tids = [], []
    for b in range(args.batches):
        sb = spec.with_(seed=batch_seed(spec, rank, b, args.batches))
        xs.append(torch.from_numpy(synthetic.activations(sb).view(np.int16)).to(dev))
        if spec.n_hash:
            r = np.random.default_rng(sb.seed)
            tids.append(torch.from_numpy(r.integers(0, spec.hash_vocab, spec.n_hash).astype(np.int32)).to(dev))
    out = torch.empty((spec.n_tokens, spec.d), dtype=torch.float32, device=dev)
    out_prev = torch.empty_like(out)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)

    def fwd(i, handle=None, o=None):
        b = i % args.batches
        api.ds4moe_forward_ex(handle or h, xs[b].data_ptr(), spec.n_tokens,
                              tids[b].data_ptr() if spec.n_hash else None, spec.n_hash,
                              (o if o is not None else out).data_ptr(), stream.cuda_stream)

    def cool(i):
        flush_buf.zero_()  # evicts everything from L2
        if h_prev is not None:
            fwd(i + 1, h_prev, out_prev)  # the previous layer: other weights, same kernels

    def time_steps(n, prep):
        st = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            prep(i)
            st[i].record(stream)
            fwd(i)
            en[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(st, en)]

    for i in range(args.warmup):
        cool(i)
        fwd(i)
    torch.cuda.synchronize()

    # timed region: each step timed alone with events on the launching stream
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
    step_ms = time_steps(args.steps, cool)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(float(sum(step_ms)), world, dev)

    # per-launch times of the same workload: events recorded between the launches (this
    # serialises the launches, so it runs after the timed region, over the same inputs)
    flush_only_ms = time_steps(args.steps, lambda i: flush_buf.zero_())  # code cold as well
    api.ds4moe_set_profiling(h, True)
    phase_ms: dict[str, list] = {}
    distinct = []
    for i in range(args.steps):
        cool(i)
        fwd(i)
        for name, ms in api.ds4moe_get_phase_times(h):  # waits for this step
            phase_ms.setdefault(name, []).append(ms)
        distinct.append(api.ds4moe_get_stats(h)["distinct_experts"])
    api.ds4moe_set_profiling(h, False)

    # end to end through the host entry point: pinned host input, copies inside the timed region
    e2e_total = None
    if with_e2e:
        x_host = torch.empty((spec.n_tokens, spec.d), dtype=torch.int16, pin_memory=True)
        x_host.copy_(xs[0].cpu())
        out_host = torch.empty((spec.n_tokens, spec.d), dtype=torch.float32, pin_memory=True)
        tid_host = tids[0].cpu().pin_memory() if spec.n_hash else None
        e2e_s = []
        for i in range(args.warmup + args.steps):
            cool(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            api.ds4moe_forward_host(h, x_host.data_ptr(), spec.n_tokens,
                                    tid_host.data_ptr() if tid_host is not None else None,
                                    spec.n_hash, out_host.data_ptr(), stream.cuda_stream)
            if i >= args.warmup:
                e2e_s.append(time.perf_counter() - t0)
        e2e_total = max_over_ranks(float(sum(e2e_s)), world, dev)

    launches = api.ds4moe_launches_per_forward(h, spec.n_tokens) * args.steps
    api.ds4moe_destroy(h)
    if h_prev is not None:
        api.ds4moe_destroy(h_prev)
    del xs, tids, out, out_prev, flush_buf
    torch.cuda.empty_cache()
    return dict(problem=problem, step_ms=step_ms, total_ms=total_ms, flush_only_ms=flush_only_ms,
                phase_ms={k: float(np.mean(v)) for k, v in phase_ms.items()}, distinct=float(np.mean(distinct)),
                e2e_total=e2e_total, launches=launches, clocks=clocks, l2_layer=h_prev is not None)


def summarize(spec, m, args, world, peaks) -> dict:
    """Throughput and roofline fractions of one measured workload."""
    ms_per_step = m["total_ms"] / args.steps
    work = kernel_work(spec, m["distinct"])
    mean_phase = m["phase_ms"]
    top = max(mean_phase, key=mean_phase.get)
    fwd_bytes = sum(work["weights"].values())
    flops = forward_flops(spec)
    hbm_bound = spec.n_tokens <= 64 or top not in work["flops"]
    if hbm_bound:
        alg = work["bytes"].get(top, 0.0)
        achieved = alg / (mean_phase[top] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                "frac": achieved / peaks["hbm"], "peak_source": f"{peaks['src']} hbm_gbs",
                "algorithmic_bytes_per_launch": alg, "traffic": recorded_traffic(top, spec.name)}
    else:
        alg = work["flops"][top]
        achieved = alg / (mean_phase[top] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": top, "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16"],
                "peak_source": f"{peaks['src']} bf16_tflops (burst; the fp16 dense rate equals bf16's)",
                "algorithmic_flops_per_launch": alg, "traffic": recorded_traffic(top, spec.name)}
    tot = sum(mean_phase.values())
    return dict(
        ms_per_step=ms_per_step,
        value=whole_job_rate(world, spec.n_tokens, args.steps, m["total_ms"] / 1e3),
        e2e=None if m["e2e_total"] is None else whole_job_rate(world, spec.n_tokens, args.steps, m["e2e_total"]),
        roofline=roof,
        detail={"step_ms_p10_p50_p90": [float(np.percentile(m["step_ms"], q)) for q in (10, 50, 90)],
                "ms_per_step_flush_only": float(np.mean(m["flush_only_ms"])),
                "phase_ms": mean_phase, "phase_share": {k: v / tot for k, v in mean_phase.items()},
                "distinct_experts_mean": m["distinct"],
                "forward_algorithmic_bytes": fwd_bytes, "forward_gbs": fwd_bytes / (ms_per_step / 1e3) / 1e9,
                "forward_hbm_frac": fwd_bytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm"],
                "forward_flops": flops, "forward_tflops": flops / (ms_per_step / 1e3) / 1e12,
                "forward_tensor_frac": flops / (ms_per_step / 1e3) / 1e12 / peaks["bf16"]})


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4,
                    help="headline workload (default 4: prefill-4096, the largest single-GPU workload)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time only the headline workload")
    ap.add_argument("--batches", type=int, default=8, help="distinct input batches cycled over the steps")
    ap.add_argument("--l2-mode", choices=["layer", "flush"], default="layer",
                    help="between steps: flush L2 then run a second layer (default), or flush only")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    spec = synthetic.CONFIGS[args.config]

    if args.impl == "reference":
        run_reference(args, spec, rank)
        return

    import torch
    import torch.distributed as dist
    from quantized_moe_gb300 import ds4moe as api

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    m = measure(api, spec, args, dev, stream, rank, world, peaks, args.l2_mode)
    head = summarize(spec, m, args, world, peaks)
    per_config = {}
    if not args.no_per_config:
        for c in sorted(synthetic.CONFIGS):
            if c == args.config:
                continue
            cs = synthetic.CONFIGS[c]
            mc = measure(api, cs, args, dev, stream, rank, world, peaks, args.l2_mode)
            sc = summarize(cs, mc, args, world, peaks)
            per_config[cs.name] = {"workload": workload_name(cs), "value": sc["value"], "unit": "tok/s",
                                   "ms_per_step": sc["ms_per_step"], "e2e_tok_s": sc["e2e"],
                                   "roofline": sc["roofline"], "gpu_launches": mc["launches"],
                                   "clocks": mc["clocks"], **sc["detail"]}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n_done, dt = oracle_sample(spec, m["problem"], args.cpu_seconds)
        cpu = {"value": n_done / dt, "unit": "tok/s", "cores": 1, "kind": "oracle",
               "sample": f"first {n_done} token(s) of the workload, one at a time, fp64 numpy oracle, 1 thread "
                         f"of {os.cpu_count()} host cores, {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": head["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 mma, f32 accumulate", "data": "synthetic",
        "config": {"workload": workload_name(spec),
                   "l2": ("flushed between steps (write of 2x L2), then one forward of a second layer with its own "
                          "weights (kernel code warm, every byte of the timed layer cold)"
                          if m["l2_layer"] else "flushed between steps (write of 2x L2)"),
                   "parallelism": f"replicas x{world}", "batches": args.batches},
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "e2e": {"value": head["e2e"], "unit": "tok/s",
                "h2d_bytes_per_step": spec.n_tokens * spec.d * 2 + spec.n_hash * 4,
                "d2h_bytes_per_step": spec.n_tokens * spec.d * 4},
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
        "detail": {**head["detail"], "kernel_source_hash": kernel_source_hash(), "peaks": peaks,
                   "per_config": per_config},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
