#!/usr/bin/env python3
"""Throughput of the PowerSGD compression step on one GB300 (per rank), as gradient GB/s
and as a fraction of the HBM roofline.

Workload "shard" (the default): one d_model = 3968 resblock shard. The four 1/8-column
weight-gradient matrices qkv 3968x1488, attn-out 3968x496, mlp-in 3968x1984 and mlp-out
15872x496 in fp16, W = 8 simulated workers, rank 112, fp16 error buffers and fp32 Q
state. Gradients are synthetic N(0, 2^-2) fp16 (sigma 2^-12 at scale s_b = 2^10), drawn
once on the device into two gradient sets used on alternate steps. Every step reads 378
MB of gradient and 378 MB of error buffer, more than the 129 MB L2, so L2 is not flushed.

Workload "stack64": 64 such resblock shards in bf16 with W = 4 and rank 112. Block b's
true gradient has std 2^-12 2^(-4b) and its scale is s_b = 2^(4b mod 24), so the raw bf16
values of deep blocks are subnormal or zero; 2 x 3968 fp32 gains/biases per block and
worker. One gradient set (12 GB per step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload shard|stack64]

With N > 1 (torchrun, one rank per GPU) every rank compresses its own resblock shard.
The ranks are independent blocks with no data exchange (weak scaling). The value is the
gradient bytes of all ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SHAPES = ((3968, 1488), (3968, 496), (3968, 1984), (15872, 496))
WORKLOADS = {
    "shard": dict(name="resblock_shard_3968_fp16_w8_r112", blocks=1, workers=8, dtype="f16", unc=0, sets=2),
    "stack64": dict(name="stack64_resblock_shards_3968_bf16_w4_r112", blocks=64, workers=4, dtype="bf16",
                    unc=2 * 3968, sets=1),
}
RANK = 112
METRIC = "PowerSGD step gradient GB/s and % of HBM roofline (rank 112, 1 GB300)"
UNIT = "GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}
SMS, FP32_LANES = 152, 128  # GB300: SMs, FP32 lanes per SM


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0: max(3, steps // 10)")
    ap.add_argument("--workload", default="shard", choices=sorted(WORKLOADS))
    return ap.parse_args()


# The dominant phase's kernel, its committed ncu summary and the file that holds its source.
PROFILED = {"ingest": ("k_ingest_p", "profiles/k_ingest_p_resblock_shard.md"),
            "decomp": ("k_decomp_tc", "profiles/k_decomp_tc_resblock_shard.md"),
            "qgemm": ("k_gemm", "profiles/k_gemm_qgemm_resblock_shard.md")}
KERNEL_SRC = "rank_gradient_compression_gb300/csrc/tc.cu"


def kernel_source_hash(path: str, name: str):
    """sha256 of a kernel's text, from its __global__ to the closing brace of its body."""
    import hashlib
    import re
    try:
        s = open(os.path.join(ROOT, path)).read()
        mt = re.search(r"__global__[^;{]*?\b" + re.escape(name) + r"\(", s)
        if mt is None:
            return None
        i = mt.start()
        j = s.index("{", i)
    except (OSError, ValueError):
        return None
    depth = 0
    for k in range(j, len(s)):
        if s[k] == "{":
            depth += 1
        elif s[k] == "}":
            depth -= 1
            if depth == 0:
                return hashlib.sha256(s[i:k + 1].encode()).hexdigest()
    return None


def profiled_traffic(phase: str):
    """DRAM bytes per launch from the phase kernel's committed ncu summary, or None when
    there is no summary or the kernel's source has changed since it was captured."""
    if phase not in PROFILED:
        return None, None
    kname, md = PROFILED[phase]
    try:
        text = open(os.path.join(ROOT, md)).read()
    except OSError:
        return None, None
    fields = dict(l.split(": ", 1) for l in text.splitlines() if ": " in l and not l.startswith(("|", "#")))
    if fields.get("source_sha256", "").strip() != kernel_source_hash(KERNEL_SRC, kname):
        return None, md
    try:
        return int(fields["traffic_bytes_per_launch"]), md
    except (KeyError, ValueError):
        return None, md


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def numel_per_worker():
    return sum(m * n for m, n in SHAPES)


# ------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU) leg
def oracle_sample(matrices, wk, min_seconds=0.0, block=0):
    """Time the fp64 oracle on steps of the given matrices of one block of the workload:
    one step, or as many consecutive steps (same gradients, evolving state) as it takes to
    spend min_seconds in the oracle. Input generation is outside the timing.
    Returns (gradient bytes processed, seconds, steps)."""
    import numpy as np
    import oracle
    import synth
    Wk = wk["workers"]
    if wk["dtype"] == "bf16":
        wl = synth.with_shapes(synth.stack64(steps=1, workers=Wk, blocks=block + 1), matrices, unc_len=0)
    else:
        wl = synth.with_shapes(synth.resblock_shard(steps=1, workers=Wk), matrices)
    grads = [[synth.grad(wl, 0, block, j, w).double().numpy() for w in range(Wk)] for j in range(len(matrices))]
    st = oracle.BlockState(e=[[np.zeros(s) for _ in range(Wk)] for s in matrices],
                           q=[synth.q0(wl, block, j).double().numpy() for j in range(len(matrices))])
    dt, n = 0.0, 0
    while n == 0 or dt < min_seconds:
        t0 = time.perf_counter()
        oracle.block_step(grads, st, wl.scale(block), wk["dtype"])
        dt += time.perf_counter() - t0
        n += 1
    return n * Wk * sum(m * n_ for m, n_ in matrices) * 2, dt, n


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wk = WORKLOADS[args.workload]
    sample = ((3968, 496),)  # attn-out of block 0, all workers: about a second of fp64 work per step
    for _ in range(args.warmup):
        oracle_sample(sample, wk)
    tot_b, tot_s = 0, 0.0
    for _ in range(args.steps):
        b, s, _ = oracle_sample(sample, wk)
        tot_b += b
        tot_s += s
    val = tot_b / tot_s / 1e9
    smp = f"attn_out 3968x496 of block 0 x {wk['workers']} workers"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wk["name"], "sample": smp},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"one step of the {smp} per timed step"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------- our leg
def make_grads(wk, dev, gen):
    """[B][J][W] raw gradients on the device, drawn with torch's seeded generator."""
    import torch
    dt = torch.float16 if wk["dtype"] == "f16" else torch.bfloat16
    out = []
    for b in range(wk["blocks"]):
        log2_sig = -2 if wk["dtype"] == "f16" else -12 - 4 * b + (4 * b) % 24
        row = []
        for (m, n) in SHAPES:
            ws = []
            for _ in range(wk["workers"]):
                x = torch.randn((m, n), generator=gen, device=dev)
                ws.append((x * 2.0 ** log2_sig).to(dt))
                del x
            row.append(ws)
        out.append(row)
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from rank_gradient_compression_gb300 import dist as pdist
    from rank_gradient_compression_gb300 import psgd

    wk = WORKLOADS[args.workload]
    B, Wk, dtype = wk["blocks"], wk["workers"], wk["dtype"]
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # one workload instance per rank: the blocks of the N-rank job are independent
    assert pdist.shard_blocks(world, rank, world) == [rank]
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    sets = [make_grads(wk, dev, g) for _ in range(wk["sets"])]
    errs = [[[torch.zeros((m, n), dtype=tdt, device=dev) for _ in range(Wk)] for (m, n) in SHAPES]
            for _ in range(B)]
    q = [[torch.randn((n, RANK), generator=g, device=dev) for (m, n) in SHAPES] for _ in range(B)]
    ghat = [[torch.empty((m, n), dtype=torch.float32, device=dev) for (m, n) in SHAPES] for _ in range(B)]
    scales = [2.0 ** 10 if dtype == "f16" else 2.0 ** ((4 * b) % 24) for b in range(B)]
    unc_in = unc_out = None
    if wk["unc"]:
        unc_in = [[(torch.randn(wk["unc"], generator=g, device=dev) * 2.0 ** (-12 - 4 * b + (4 * b) % 24))
                   for _ in range(Wk)] for b in range(B)]
        unc_out = [torch.empty(wk["unc"], dtype=torch.float32, device=dev) for _ in range(B)]
    ps = psgd.PowerSGD(SHAPES, B, Wk, RANK, dtype, unc_len=wk["unc"], device=dev)
    nsets = len(sets)

    def step(i, grads=None, gh=None):
        ps.step(grads if grads is not None else sets[i % nsets], errs, q, scales,
                gh if gh is not None else ghat, unc_in, unc_out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    psgd.psgd_profile_begin(ps.handle, args.steps)
    launches0 = psgd.psgd_launch_count(ps.handle)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    start.record(stream)
    host_s = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        step(i)
        host_s.append(time.perf_counter() - t0)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    launches = psgd.psgd_launch_count(ps.handle) - launches0
    phase_ms, nprof = psgd.psgd_profile_end(ps.handle)
    ms = pdist.max_over_ranks(start.elapsed_time(end) / args.steps, device=dev)

    # ---------------- end to end: pinned host gradients in, G-hat out, every step
    e2e_steps = args.e2e_steps or max(3, args.steps // 10)
    # Step t+1's gradients are copied on their own stream into the other device set while
    # step t runs, and G-hat is read back on a third stream; events order every reuse of
    # a buffer. Each step still copies its own inputs and reads its result inside the
    # timed region. The second device set of a one-set workload is allocated here.
    if nsets == 1:
        sets.append([[[torch.empty_like(t) for t in ws] for ws in row] for row in sets[0]])
    host_g = [[[t.cpu().pin_memory() for t in ws] for ws in row] for row in sets[0]]
    host_gh = [[torch.empty((m, n), dtype=torch.float32).pin_memory() for (m, n) in SHAPES] for _ in range(B)]
    ghat2 = [[torch.empty_like(x) for x in row] for row in ghat]
    gh_sets = [ghat, ghat2]
    h2d = sum(t.numel() * t.element_size() for row in host_g for ws in row for t in ws)
    d2h = sum(t.numel() * t.element_size() for row in host_gh for t in row)
    if unc_in is not None:
        h2d += sum(t.numel() * t.element_size() for row in unc_in for t in row)
    cp_stream, rb_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    inputs_ready, inputs_free = [ev(), ev()], [ev(), ev()]
    gh_ready, gh_free = [ev(), ev()], [ev(), ev()]

    def copy_in(k):
        with torch.cuda.stream(cp_stream):
            cp_stream.wait_event(inputs_free[k])
            for b in range(B):
                for j in range(len(SHAPES)):
                    for w_ in range(Wk):
                        sets[k][b][j][w_].copy_(host_g[b][j][w_], non_blocking=True)
            inputs_ready[k].record(cp_stream)

    def run(nsteps):
        copy_in(0)
        for i in range(nsteps):
            k = i % 2
            if i + 1 < nsteps:
                copy_in(1 - k)
            stream.wait_event(inputs_ready[k])
            stream.wait_event(gh_free[k])
            step(i, sets[k], gh_sets[k])
            inputs_free[k].record(stream)
            gh_ready[k].record(stream)
            with torch.cuda.stream(rb_stream):
                rb_stream.wait_event(gh_ready[k])
                for b in range(B):
                    for j in range(len(SHAPES)):
                        host_gh[b][j].copy_(gh_sets[k][b][j], non_blocking=True)
                gh_free[k].record(rb_stream)
        stream.wait_stream(cp_stream)
        stream.wait_stream(rb_stream)

    run(2)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cp_stream.wait_stream(stream)
    rb_stream.wait_stream(stream)
    run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = pdist.max_over_ranks(e0.elapsed_time(e1) / e2e_steps, device=dev)
    barrier()

    nel = B * numel_per_worker()          # matrix entries per step (all blocks)
    we = Wk * nel                         # worker-elements per step
    grad_bytes = we * 2                   # per rank per step
    value = world * grad_bytes / (ms * 1e-3) / 1e9
    e2e_val = world * grad_bytes / (e2e_ms * 1e-3) / 1e9

    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    # algorithmic bytes per launch and flops per launch, per phase (per rank)
    unc_bytes = 4 * B * wk["unc"] * (Wk + 1)
    alg_bytes = {"ingest": 6 * we, "pgemm": 2 * we, "qgemm": 2 * we, "decomp": 4 * we + 4 * nel,
                 "skip_unc": unc_bytes, "orth": 0, "qreduce": 0}
    flops = {"pgemm": 2 * we * RANK, "qgemm": 2 * we * RANK, "decomp": 2 * nel * RANK}
    per_launch = {k: v / max(nprof, 1) for k, v in phase_ms.items()}
    total_ms = sum(per_launch.values()) or 1.0
    share = {k: v / total_ms for k, v in per_launch.items()}
    dom = max(per_launch, key=per_launch.get)
    if ps.engine == "tcgen05" and dom == "pgemm":
        alg_bytes["pgemm"] = 0
    d_ms = per_launch[dom]
    if alg_bytes.get(dom, 0) and (ps.engine == "tcgen05" or dom in ("ingest", "decomp")):
        ach = alg_bytes[dom] / (d_ms * 1e-3) / 1e9
        traffic, prof = profiled_traffic(dom) if args.workload == "shard" else (None, None)
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": traffic, "kernel": dom, "peak_kind": pk_kind, "profile": prof,
                "alg_bytes": alg_bytes[dom]}
    else:
        ach = flops.get(dom, 0) / (d_ms * 1e-3) / 1e12
        peak = SMS * FP32_LANES * 2 * float(pk.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "frac": ach / peak if peak else None, "traffic": None, "kernel": dom,
                "peak_kind": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"}
    step_bytes = 12 * we + 4 * nel + unc_bytes
    step_gbs = world * step_bytes / (ms * 1e-3) / 1e9

    l2 = (f"inputs larger than L2 ({(4 * we) / 1e6:.0f} MB of gradient and error read per step), no flush")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wk["name"], "shapes": [list(s) for s in SHAPES], "workers": Wk,
                       "rank": RANK, "grad_dtype": dtype, "engine": ps.engine, "blocks_per_rank": B,
                       "unc_len": wk["unc"], "l2": l2,
                       "parallelism": f"independent workload instance per rank x{world}"},
            "roofline": roof,
            "step_roofline": {"alg_bytes_per_step": step_bytes, "achieved": step_gbs, "unit": "GB/s",
                              "frac_of_measured_hbm": step_gbs / hbm / world,
                              "frac_of_8TBs": step_gbs / 8000.0 / world},
            "phases_ms_per_step": {k: round(v, 4) for k, v in per_launch.items()},
            "phase_share": {k: round(v, 4) for k, v in share.items()},
            "clocks": clk, "gpu_launches": launches,
            # host time of one psgd_step call (argument marshalling, table lookup, launches),
            # median over the first timed steps, before the launch queue can fill
            "host_us_per_step": 1e6 * statistics.median(host_s[:10]),
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b_, s_, nst = oracle_sample(SHAPES, wk, min_seconds=10.0)
        if args.workload == "shard":
            smp = f"{nst} consecutive full steps of the workload (all 4 matrices, W=8) in fp64 numpy"
        else:
            smp = (f"{nst} consecutive steps of block 0 (all 4 matrices, W=4, bf16) of the 64 in fp64 "
                   f"numpy; the blocks are alike in cost")
        line["cpu_baseline"] = {"value": b_ / s_ / 1e9, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                                "sample": smp + ", at least 10 s of oracle time", "seconds": s_}
    if rank == 0:
        print(json.dumps(line), flush=True)
    ps.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
