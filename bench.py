"""Benchmark of one inflight-batch layer step (RoPE + append, then paged attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--kv-dtype bf16|fp8|int8]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is the whole hot path over one batch: paged_kv_append_rope + paged_attention_forward
(plan, context tensor-core kernel, split-KV decode, log-sum-exp combine), inputs resident in HBM.
The default workload is the decode-only Llama-7B-like layer (64 requests, 32/32 heads, head_dim
128, KV lengths U[512, 4096], 64-token pages): the KV pool (~2.4 GB) is larger than L2, so no
flush is needed between steps.  With N > 1 (torchrun) every rank runs its own batch of the same
shape (requests are independent, so the path shards with no exchange) and ``value`` is the sum
over ranks of the work divided by the slowest rank's time.

Printed (rank 0): one JSON line with value, e2e (same metric through the public API with the
step's q/k/v copied host->device and the output copied back inside the timed region), the
dominant kernel's roofline, clocks sampled during the timed region and the CPU oracle baseline.
``--impl reference`` times the CPU oracle itself on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn KV GB/s (% of HBM peak); prefill TFLOP/s (% BF16 peak); tokens/s"


# --------------------------------------------------------------------------------------------
# algorithmic work (what the method must move / compute)
# --------------------------------------------------------------------------------------------

def work_of(b) -> dict:
    """Decode KV bytes (each KV head read once per request), context flops (causal part only,
    2 flops per MAC for QK^T and PV), append bytes."""
    esz = 1 if b.kv_dtype != "bf16" else 2
    D, Hq, Hkv = b.head_dim, b.num_q_heads, b.num_kv_heads
    gen = b.request_types == 1
    L = (b.past + b.new_len).astype(np.int64)
    dec_kv = int(np.sum(L[gen]) * 2 * Hkv * D * esz)
    dec_qo = int(np.sum(b.new_len[gen])) * 2 * Hq * D * 2  # q read + out write per generation row
    ctx_flops = 0
    for r in np.nonzero(~gen)[0]:
        n, P = int(b.new_len[r]), int(b.past[r])
        ctx_flops += 4 * D * Hq * (n * P + n * (n + 1) // 2)
    T = b.num_tokens
    append_bytes = T * (Hq + 2 * Hkv) * D * 2 + T * Hq * D * 2 + T * 2 * Hkv * D * esz + T * D // 2 * 8
    return dict(decode_kv_bytes=dec_kv, decode_bytes=dec_kv + dec_qo, ctx_flops=ctx_flops,
                append_bytes=append_bytes, tokens=T)


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if one exists for this kernel and
    workload (profiles/<kernel>__<workload>.md, line 'dram_bytes_per_launch: <int>')."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("dram_bytes_per_launch:"):
            try:
                return int(line.split(":", 1)[1].strip())
            except ValueError:
                return None
    return None


# --------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.25)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# --------------------------------------------------------------------------------------------

class OracleSample:
    """The CPU oracle on one generation request at a time (write image of its token, then fp64
    attention for all its heads), cycling through the batch's generation requests."""

    def __init__(self, b):
        import oracle
        self.oracle = oracle
        self.b = b
        bits = lambda t: (t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
                          if t.dtype == torch.bfloat16 else t.detach().cpu().contiguous().numpy())
        self.pool = bits(b.pool)
        self.q, self.k, self.v = bits(b.q), bits(b.k), bits(b.v)
        self.cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos)
        self.gen = [r for r in range(b.num_requests) if b.request_types[r] == 1]
        self.row_of = np.concatenate([[0], np.cumsum(b.new_len)[:-1]]).astype(np.int64)
        self.gen_row0 = int(b.new_len[:b.num_contexts].sum())
        self.i = 0
        self.esz = 1 if b.kv_dtype != "bf16" else 2

    def step(self) -> int:
        """Process one generation request (all of its tokens); returns the KV bytes it read."""
        b, o = self.b, self.oracle
        r = self.gen[self.i % len(self.gen)]
        self.i += 1
        row, n = int(self.row_of[r]), int(b.new_len[r])
        sl = slice(row, row + n)
        g = slice(row - self.gen_row0, row - self.gen_row0 + n)  # rows of the draft-token arrays
        kw = dict(new_len=b.new_len[r:r + 1], past=b.past[r:r + 1], block_table=b.block_table[r:r + 1],
                  num_q_heads=b.num_q_heads, num_kv_heads=b.num_kv_heads, head_dim=b.head_dim,
                  tokens_per_block=b.tokens_per_block, num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8",
                  kv_int8=b.kv_dtype == "int8")
        st, q_out = o.append_rope_ex(**kw, inv_scale=b.inv_scale, q_bits=self.q[sl], k_bits=self.k[sl],
                                     v_bits=self.v[sl], cs=self.cs, pool=self.pool,
                                     pos_offset=None if b.position_offsets is None else b.position_offsets[g])
        q64 = o.f32_from_bf16(q_out).astype(np.float64)
        o.attention(**kw, kv_scale=b.kv_scale, pool=self.pool, q=q64, softmax_scale=b.softmax_scale,
                    num_contexts=0, gen_mask=None if b.packed_mask is None else b.packed_mask[g])
        L = int(b.past[r]) + n
        return L * 2 * b.num_kv_heads * b.head_dim * self.esz


def cpu_baseline(b, budget_s: float = 12.0) -> dict:
    s = OracleSample(b)
    s.step()  # build / load the oracle outside the timing
    t0, nbytes, n = time.perf_counter(), 0, 0
    while time.perf_counter() - t0 < budget_s and n < 4 * len(s.gen):
        nbytes += s.step()
        n += 1
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": s.oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} generation requests of the workload (all heads each), fp64 oracle "
                      f"write image + attention, {dt:.1f} s wall"}


# --------------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", rank=rank, world_size=world)
    else:
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    """Max over ranks (the slowest rank's time); NCCL reduces on the GPU, gloo on the host."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(work_per_rank: float, ms_total_per_rank: float, steps: int, world: int) -> tuple[float, float]:
    """Weak scaling: every rank processes its own batch of the same shape.  Returns (ms per
    step of the slowest rank, whole-job units per second = world * work / that time)."""
    ms_step = reduce_max(ms_total_per_rank, world) / steps
    return ms_step, world * work_per_rank / (ms_step * 1e-3)


def run_ours(args):
    import paged_kv_cache_rope_gb300 as pk
    from paged_kv_cache_rope_gb300 import workloads as W

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    b = W.workload(args.workload, kv_dtype=args.kv_dtype, device=str(dev), poison=False,
                   seed=args.workload + 1000 * rank, max_gen=args.max_gen)
    work = work_of(b)
    pool = pk.KVPool(b.pool, b.kv_scale, b.inv_scale)
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev)
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, dev)
    step = pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)
    q, k, v = b.q, b.k, b.v

    # launches per step and their names
    step(q, k, v)
    torch.cuda.synchronize()
    fwd_names = pk.last_launch_names()
    names = ["append_rope"] + fwd_names
    launches_per_step = len(names)
    # generation rows run on the narrow and/or the wide decode kernel: together they read the KV
    dec_names = [n for n in ("decode_splitkv", "decode_splitkv_wide", "decode_tc") if n in fwd_names]
    dominant = "+".join(dec_names) if work["decode_kv_bytes"] else "context_attn"

    for _ in range(args.warmup):
        step(q, k, v)
    torch.cuda.synchronize()

    # (1) the step itself, timed as a whole.  (2) the same K steps again with per-kernel events
    # recorded by the library around each launch; while events are set the library keeps every
    # kernel on the caller's stream (no context/generation overlap), so that each pair of events
    # brackets one kernel's own work.
    ev_app = [pk.KernelEvents(1) for _ in range(args.steps)]
    ev_fwd = [pk.KernelEvents(len(fwd_names)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        start.record()
        for i in range(args.steps):
            pk.paged_kv_append_rope(pool, meta, step.Hq, q, k, v, step.q_out, table, step.d_error)
            pk.paged_attention_forward(pool, meta, step.Hq, step.q_out, step.out, step.softmax_scale,
                                       step.workspace, step.d_error)
        stop.record()
        torch.cuda.synchronize()
        barrier(world)
        k0.record()
        for i in range(args.steps):
            with ev_app[i]:
                pk.paged_kv_append_rope(pool, meta, step.Hq, q, k, v, step.q_out, table, step.d_error)
            with ev_fwd[i]:
                pk.paged_attention_forward(pool, meta, step.Hq, step.q_out, step.out, step.softmax_scale,
                                           step.workspace, step.d_error)
        k1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_step, _ = aggregate(1.0, start.elapsed_time(stop), args.steps, world)
    ms_serial, _ = aggregate(1.0, k0.elapsed_time(k1), args.steps, world)
    err = int(step.d_error.item())
    if err:
        raise SystemExit(f"device error word {err} during the timed region")

    kern_ms = {}
    for j, n in enumerate(fwd_names):
        kern_ms[n] = statistics.fmean(e.elapsed_ms(j) for e in ev_fwd)
    kern_ms["append_rope"] = statistics.fmean(e.elapsed_ms(0) for e in ev_app)

    # ---- the same step captured once into a CUDA graph and replayed (launch overhead gone) ----
    graph = None
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            step(q, k, v)
        torch.cuda.current_stream().wait_stream(gs)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            step(q, k, v)
        for _ in range(3):
            cg.replay()
        torch.cuda.synchronize()
        barrier(world)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            cg.replay()
        g1.record()
        torch.cuda.synchronize()
        g_ms, _ = aggregate(1.0, g0.elapsed_time(g1), args.steps, world)
        graph = {"ms_per_step": g_ms, "launches_per_step": launches_per_step}
        del cg
    except Exception as exc:  # capture is a measurement extra, never a reason to fail the bench
        graph = {"error": str(exc)[:200]}

    # ---- e2e through the public API: host q/k/v in pinned memory, output copied back ----
    # Every step copies its q/k/v from pinned host memory and its output back to the host.  The
    # copies run on a second stream, double-buffered, so that step i's output and step i+2's
    # inputs move while step i+1 computes (as a serving loop would run it); two step objects
    # share the pool and own separate output buffers.
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    dbuf = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
    steps2 = [step, pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)]
    hout = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    xs = torch.cuda.Stream()
    cs = torch.cuda.current_stream()
    e2e_steps = max(10, args.steps // 4)

    def run_e2e(n: int) -> None:
        h2d_ev = [torch.cuda.Event(), torch.cuda.Event()]
        done_ev = [torch.cuda.Event(), torch.cuda.Event()]
        with torch.cuda.stream(xs):
            xs.wait_stream(cs)
            for i in range(min(2, n)):
                for d, h in zip(dbuf[i], (hq, hk, hv)):
                    d.copy_(h, non_blocking=True)
                h2d_ev[i].record(xs)
        for i in range(n):
            bi = i & 1
            cs.wait_event(h2d_ev[bi])
            steps2[bi](*dbuf[bi])
            done_ev[bi].record(cs)
            with torch.cuda.stream(xs):
                xs.wait_event(done_ev[bi])
                hout.copy_(steps2[bi].out, non_blocking=True)
                if i + 2 < n:
                    for d, h in zip(dbuf[bi], (hq, hk, hv)):
                        d.copy_(h, non_blocking=True)
                    h2d_ev[bi].record(xs)
        cs.wait_stream(xs)

    run_e2e(3)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    run_e2e(e2e_steps)
    e1.record()
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    e2e_ms = reduce_max(max(e0.elapsed_time(e1) / e2e_steps, wall_ms), world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()

    pk_ = peaks()
    if work["decode_kv_bytes"]:
        value = world * work["decode_kv_bytes"] / (ms_step * 1e-3) / 1e9
        e2e_value = world * work["decode_kv_bytes"] / (e2e_ms * 1e-3) / 1e9
        unit = "GB/s"
    else:
        value = world * work["ctx_flops"] / (ms_step * 1e-3) / 1e12
        e2e_value = world * work["ctx_flops"] / (e2e_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    if graph and "ms_per_step" in graph:
        w = work["decode_kv_bytes"] or work["ctx_flops"]
        graph["value"] = world * w / (graph["ms_per_step"] * 1e-3) / (1e9 if work["decode_kv_bytes"] else 1e12)
        graph["tokens_per_s"] = world * work["tokens"] / (graph["ms_per_step"] * 1e-3)
    if dominant != "context_attn":
        dec_ms = sum(kern_ms[n] for n in dec_names)
        ach = work["decode_bytes"] / (dec_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk_["hbm"], "unit": "GB/s",
                "frac": ach / pk_["hbm"], "kernel": dominant, "peak_source": pk_["src"]}
    else:
        ach = work["ctx_flops"] / (kern_ms["context_attn"] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk_["bf16"], "unit": "TFLOP/s",
                "frac": ach / pk_["bf16"], "kernel": "context_attn", "peak_source": pk_["src"]}
    roof["traffic"] = ncu_traffic(dominant, b.name + ("" if b.kv_dtype == "bf16" else "_" + b.kv_dtype))

    kernels = {}
    for n, ms in kern_ms.items():
        d = {"us": ms * 1e3}
        if n in dec_names and len(dec_names) == 1:
            d["GB/s"] = work["decode_bytes"] / (ms * 1e-3) / 1e9
            d["frac_hbm"] = d["GB/s"] / pk_["hbm"]
        elif n == "context_attn":
            d["TFLOP/s"] = work["ctx_flops"] / (ms * 1e-3) / 1e12
            d["frac_bf16"] = d["TFLOP/s"] / pk_["bf16"]
        elif n == "append_rope":
            d["GB/s"] = work["append_bytes"] / (ms * 1e-3) / 1e9
            d["frac_hbm"] = d["GB/s"] / pk_["hbm"]
        kernels[n] = d

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"bf16": "bf16", "fp8": "fp8-e4m3 KV / bf16 q", "int8": "int8 KV / bf16 q"}[b.kv_dtype],
        "data": "synthetic (seeded N(0,1) q/k/v and cached KV, random page placement)",
        "config": {"workload": b.name, "requests": b.num_requests, "contexts": b.num_contexts,
                   "num_tokens": b.num_tokens, "num_q_heads": b.num_q_heads,
                   "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim,
                   "tokens_per_block": b.tokens_per_block, "kv_dtype": b.kv_dtype,
                   "l2": "inputs larger than L2 (KV pool %.2f GB), no flush" % (
                       b.pool.numel() * b.pool.element_size() / 1e9),
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "tokens_per_s": world * work["tokens"] / (ms_step * 1e-3),
        "pct_of_hbm_peak": 100.0 * value / pk_["hbm"] if unit == "GB/s" else None,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "graph": graph,
        "kernels": kernels,
        "kernels_timed": "second loop of the same K steps, per-kernel events, all kernels on one stream",
        "ms_per_step_serial": ms_serial,
        "roofline": roof,
        "clocks": sampler.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b.to("cpu"))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as the reference arm: rank 0 only, one generation request per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from paged_kv_cache_rope_gb300 import workloads as W

    b = W.workload(args.workload, kv_dtype=args.kv_dtype, device="cpu", poison=False)
    s = OracleSample(b)
    for _ in range(args.warmup):
        s.step()
    t0 = time.perf_counter()
    nbytes = sum(s.step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v and cached KV, random page placement)",
        "config": {"workload": b.name, "kv_dtype": b.kv_dtype,
                   "sample": "one generation request (all heads) per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": s.oracle.num_threads(), "kind": "oracle",
                         "sample": f"{args.steps} generation requests, fp64 write image + attention"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8", "int8"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--max-gen", type=int, default=None,
                    help="keep only the first N generation requests (profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
