"""Benchmark of the W4A16 routed-MoE block on GB300: single-token decode at production width
(hidden 2048, 256 experts top-8, expert/shared intermediate 512, int4 experts, int8 router/shared, g64).

A step is one forward call: one token through one whole block (router -> top-8 -> experts -> shared ->
combine). Steps rotate over --layers distinct weight sets (default 40, 18.3 GB) and a pool of distinct tokens,
so that no call finds its weights in the 129 MB L2. One JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs independent replicas on its own GPU (the block has no exchange step);
value = tokens of all ranks / max elapsed over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w4a16_top_mixture_gb300 import synth  # noqa: E402

METRIC = "MoE-block tokens/s at 2048/256x512 top-8 W4A16; achieved HBM GB/s vs peak"
WORKLOAD = ("decode T=1: hidden 2048, 256 experts top-8 renormalised, expert intermediate 512, shared expert "
            "intermediate 512 with sigmoid gate; int4 g64 affine experts, int8 g64 router+shared; x fp16 ~N(0,1); "
            "uniform routing")
SEED = 1


def rank_env():
    """(world size, rank, local rank) from the torchrun environment; 1 / 0 / 0 without it."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank):
    """Each replica draws its own weights and tokens."""
    return SEED + 1000 * rank


def max_over_ranks(v):
    """Largest value of v over the process group (v itself without one): the slowest rank sets the time."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(v)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, steps, elapsed_ms):
    """Tokens per second of the whole job: every rank processes `steps` tokens in at most `elapsed_ms`."""
    return world * steps / (elapsed_ms * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_record():
    """DRAM bytes per launch from a committed ncu summary, valid only if the kernel source is unchanged."""
    rec = os.path.join(ROOT, "profiles", "k_decode1_prod_t1.json")
    if not os.path.exists(rec):
        return None
    d = json.load(open(rec))
    if d.get("kernel_src_sha256") != kernel_sha():
        return None
    return d.get("dram_bytes_per_launch")


# k_decode1's sources
KERNEL_SOURCES = ("decode1.cu", "decode_dev.cuh", "topk.cuh", "decode.cuh", "layout.cuh", "ptx.cuh")


def kernel_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a16_top_mixture_gb300", "csrc")
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()


class ClockSampler:
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(seconds=12.0, layer_seed=SEED):
    """The float64 oracle, as it stands, on a bounded sample of the same workload (T=1 tokens through one
    production block), single-threaded in a child process. Returns tokens/s and the sample description."""
    code = f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
import oracle.moe_oracle as O
from w4a16_top_mixture_gb300 import synth
cfg = synth.PROD
w = synth.gen_layer(cfg, {layer_seed}, 0)
n, t0 = 0, time.perf_counter()
while time.perf_counter() - t0 < {seconds}:
    x = synth.gen_token(cfg, 12345, n)[None, :]
    O.block_forward(w, x, cfg.top_k)          # fresh dequantisation of the selected experts every token
    n += 1
el = time.perf_counter() - t0
print(json.dumps({{"tokens": n, "seconds": el}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["tokens"] / d["seconds"], d


def run_reference(args):
    """Reference arm: the float64 oracle on the host cores, same metric/unit; each step = one token."""
    _, rank, _ = rank_env()
    if rank != 0:
        return
    budget = float(os.environ.get("MOE_REF_BUDGET_S", "90"))
    code = f"""
import sys, time, json
sys.path.insert(0, {ROOT!r})
import oracle.moe_oracle as O
from w4a16_top_mixture_gb300 import synth
cfg = synth.PROD
w = synth.gen_layer(cfg, {SEED}, 0)
for i in range({args.warmup}):
    O.block_forward(w, synth.gen_token(cfg, 999, i)[None, :], cfg.top_k)
n, t0 = 0, time.perf_counter()
while n < {args.steps} and (n == 0 or time.perf_counter() - t0 < {budget}):
    O.block_forward(w, synth.gen_token(cfg, 12345, n)[None, :], cfg.top_k)
    n += 1
print(json.dumps({{"tokens": n, "seconds": time.perf_counter() - t0}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    v = d["tokens"] / d["seconds"]
    sample = f"{d['tokens']} of {args.steps} steps timed (one token each, {budget:.0f} s budget)"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": 1},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "cpu_count": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _time_graph(fn, reps=10, per=20):
    """Device time per call of fn: CUDA events around each of `reps` replays of a graph of `per` calls, after
    warm-up. Returns (median, list of per-replay times), microseconds per call."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(per):
            fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / per)
    return float(np.median(ts)), ts


def _roofline_entry(cfg, U, T, us, peak):
    """Algorithmic bytes of one call (router, shared expert, U unique experts), achieved GB/s and fractions."""
    b = synth.unique_weight_bytes(cfg, U)
    gbs = b / (us * 1e-6) / 1e9
    return {"unique_experts": int(U), "algorithmic_bytes": int(b), "achieved_gbs": gbs, "frac": gbs / peak,
            "frac_of_8tbs": gbs / 8000.0, "tokens": T}


def extra_configs(stk, blocks, X, peak):
    """The other block configurations, each on seeded synthetic inputs of its shape (device-resident; times are
    device times). Unique experts U come from the call's own routing record; roofline fractions are against
    the measured HBM peak (frac) and against 8 TB/s (frac_of_8tbs)."""
    import torch
    from w4a16_top_mixture_gb300 import lib
    out = {}

    def dev(x):
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.float16)

    def unique(b, T):
        return len(np.unique(b.last_routing(T)["ids"].cpu().numpy()))

    # tiny block, T = 1
    cfg = synth.TINY
    b = lib.MoeBlock.from_config(cfg, max_tokens=1)
    b.load_weights(synth.gen_layer(cfg, 5))
    xd, od = dev(synth.gen_x(cfg, 1, 5)), torch.empty((1, cfg.hidden), dtype=torch.float16, device="cuda")
    us, _ = _time_graph(lambda: b.forward(xd, od))
    out["tiny_T1"] = {"us_per_block": us, "tokens_per_s": 1e6 / us, "note": "L2-resident (one tiny layer)",
                      **_roofline_entry(cfg, unique(b, 1), 1, us, peak)}
    b.close()
    # production block, T = 16, Zipf(1.1) routing, 4 layers rotated
    cfg = synth.PROD
    bs, xs = [], []
    for l in range(4):
        x = synth.gen_x(cfg, 16, 42 + l)
        w = synth.gen_layer(cfg, 42 + l)
        w["router_q"], w["router_s"], w["router_b"] = synth.zipf_router(cfg, x, 42 + l)
        b = lib.MoeBlock.from_config(cfg, max_tokens=16)
        b.load_weights(w)
        bs.append(b)
        xs.append(dev(x))
    od = torch.empty((16, cfg.hidden), dtype=torch.float16, device="cuda")
    Us = []
    for b, x in zip(bs, xs):
        b.forward(x, od)
        torch.cuda.synchronize()
        Us.append(unique(b, 16))
    it = [0]

    def step16():
        i = it[0] % 4
        it[0] += 1
        bs[i].forward(xs[i], od)
    us, _ = _time_graph(step16)
    U = float(np.mean(Us))
    out["batched_T16_zipf"] = {"us_per_block": us, "tokens_per_s": 16e6 / us, "U_per_layer": Us,
                               **_roofline_entry(cfg, U, 16, us, peak)}
    for b in bs:
        b.close()
    # 40 stacked layers with RMSNorm + residual, T = 1: one moe_stack_forward call (one chain of launches)
    # per token through all layers
    h = [X[0:1].clone(), torch.empty_like(X[0:1])]
    us, _ = _time_graph(lambda: stk.forward(h[0], h[1]), reps=10, per=5)
    nl = stk.n_layers
    ent = _roofline_entry(cfg, cfg.top_k, 1, us / nl, peak)
    ent["algorithmic_bytes_per_call"] = ent["algorithmic_bytes"] * nl
    out["stack_T1"] = {"layers": nl, "us_per_token": us, "us_per_block": us / nl, "tokens_per_s": 1e6 / us,
                       "api": "moe_stack_forward", **ent}
    # prompt chunk T = 512, uniform and Zipf routing (tcgen05 grouped-GEMM path)
    for routing, seed in (("uniform", 553), ("zipf", 42)):
        x = synth.gen_x(cfg, 512, seed)
        w = synth.gen_layer(cfg, seed)
        if routing == "zipf":
            w["router_q"], w["router_s"], w["router_b"] = synth.zipf_router(cfg, x, seed)
        b = lib.MoeBlock.from_config(cfg, max_tokens=512)
        b.load_weights(w)
        xd, od = dev(x), torch.empty((512, cfg.hidden), dtype=torch.float16, device="cuda")
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        ts = []
        for r in range(13):
            flush.fill_(r)            # the layer's 0.9 GB of weights exceed L2 anyway; the flush makes sure
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            b.forward(xd, od)
            e1.record()
            torch.cuda.synchronize()
            if r >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        us = float(np.median(ts))
        U = unique(b, 512)
        ent = _roofline_entry(cfg, U, 512, us, peak)
        flops = 2.0 * 512 * cfg.top_k * 3 * cfg.hidden * cfg.expert_inter   # routed work, 2 flops a weight a token
        ent["routed_tflops"] = flops / (us * 1e-6) / 1e12
        out[f"chunk_T512_{routing}"] = {"us_per_block": us, "tokens_per_s": 512e6 / us, **ent}
        b.close()
        del flush
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from w4a16_top_mixture_gb300 import build, lib

    world, rank, local = rank_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.cuda.current_device()
    build.build()
    cfg = synth.PROD
    NL = args.layers
    # The layers live in one stack (it serves the stacked configuration as a whole); the headline steps call
    # its layers one at a time through their own block handles.
    stk = lib.MoeStack(cfg, NL, max_tokens=1, eps=1e-6)
    for l in range(NL):
        stk.load_layer(l, synth.gen_layer(cfg, rank_seed(rank), l, with_gamma=True))   # host arrays: repacked
    blocks = [lib.MoeBlock.borrow(stk, l) for l in range(NL)]
    pool = 4096
    xh = synth.gen_x_fast(cfg, pool, 77 + rank)
    X = torch.from_numpy(xh.view(np.int16)).cuda().view(torch.float16)
    OUT = torch.empty_like(X)

    def step(i):
        b = blocks[i % NL]
        j = i % pool
        b.forward(X[j:j + 1], OUT[j:j + 1])     # current stream (the capture stream inside a graph)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    s, f = stk.status()
    if s != 0:
        raise RuntimeError(f"device status {s} flags {f:#x}")

    # The timed steps are replayed from CUDA graphs (S steps each) so that host launch latency does not
    # leave the GPU idle between the short decode kernels.
    K = args.steps
    S = min(K, 200)

    def capture(n, base):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(n):
                step(base + i)
        return g
    g_main = capture(S, args.warmup)
    g_tail = capture(K % S, args.warmup) if K % S else None
    launches_per_step = 1
    st = torch.cuda.current_stream()
    g_main.replay()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t_start.record(st)
        for _ in range(K // S):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        t_end.record(st)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    launches = K * launches_per_step
    kern_ms = elapsed_ms / K            # per launch, including the gap between graph nodes
    s, f = stk.status()
    if s != 0:
        raise RuntimeError(f"device status {s} flags {f:#x}")
    elapsed_ms = max_over_ranks(elapsed_ms)
    # a longer record of the same step: the median over 50 replays of a 200-step graph (extra field)
    g_med = capture(200, args.warmup + K)
    reps = []
    for _ in range(50):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g_med.replay()
        e1.record(st)
        torch.cuda.synchronize()
        reps.append(e0.elapsed_time(e1) * 1e3 / 200)

    # end-to-end through the C ABI with host buffers (pinned), copies inside the timed region
    Ke = min(K, 2000)
    xpin = torch.from_numpy(xh[:Ke].view(np.int16).copy()).view(torch.float16).pin_memory()
    opin = torch.empty_like(xpin).pin_memory()
    for i in range(min(20, Ke)):
        blocks[i % NL].forward_host(xpin[i:i + 1], opin[i:i + 1], stream=st)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(Ke):
        blocks[i % NL].forward_host(xpin[i:i + 1], opin[i:i + 1], stream=st)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s)

    if rank == 0:
        bytes_call = synth.unique_weight_bytes(cfg, cfg.top_k)
        peak, kind = peaks()
        achieved = bytes_call / (kern_ms * 1e-3) / 1e9
        tr = traffic_record()
        cpu_v, cpu_d = cpu_baseline() if not args.skip_cpu else (None, {"tokens": 0, "seconds": 0.0})
        value = whole_job_value(world, K, elapsed_ms)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": 1, "weight_sets": NL,
                       "weight_bytes_resident": NL * synth.layer_bytes(cfg),
                       "l2": f"inputs larger than L2: {NL} distinct weight sets rotated, a different token each step",
                       "timing": f"CUDA graphs of {S} steps replayed; CUDA events around the replays",
                       "parallelism": f"replicas x{world}", "weights": "int4/int8 g64 affine, fp16 activations"},
            "us_per_block": kern_ms * 1e3,
            "us_per_block_median_50x200": float(np.median(reps)),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": tr, "peak_kind": kind,
                         "frac_of_8tbs": achieved / 8000.0,
                         "algorithmic_bytes_per_launch": bytes_call,
                         "kernel": "k_decode1 (fused single-token decode kernel, one launch per step)"},
            "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": 1, "cpu_count": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{cpu_d['tokens']} T=1 tokens through one production block in "
                                       f"{cpu_d['seconds']:.1f} s, single-threaded float64 numpy"},
            "e2e": {"value": whole_job_value(world, Ke, e2e_s * 1e3), "unit": "tokens/s", "h2d_bytes_per_step": 2 * cfg.hidden,
                    "d2h_bytes_per_step": 2 * cfg.hidden,
                    "how": "moe_block_forward_host: pinned x -> device, forward, out -> host, status word, stream sync, per step"},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        if not args.no_extras:
            line["configs"] = extra_configs(stk, blocks, X, peak)
        print(json.dumps(line), flush=True)
    stk.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=40)
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle leg (profiling runs)")
    ap.add_argument("--no-extras", action="store_true", help="omit the other block configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
