"""Benchmark of one inflight-batch layer step (RoPE + append, then paged attention) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--kv-dtype bf16|fp8|int8]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-sub]

A step is the whole hot path over one batch: paged_kv_append_rope + paged_attention_forward
(plan, context tensor-core kernel, split-KV decode, log-sum-exp combine), inputs resident in HBM.
The default workload is the decode-only Llama-7B-like layer (64 requests, 32/32 heads, head_dim
128, KV lengths U[512, 4096], 64-token pages): the KV pool (~2.4 GB) is larger than L2, so no
flush is needed between steps.  With N > 1 (torchrun) every rank runs its own batch of the same
shape (requests are independent, so the path shards with no exchange) and ``value`` is the sum
over ranks of the work divided by the slowest rank's time.

Printed (rank 0): one JSON line with value (decode KV GB/s of the default workload), e2e (same
metric through the public API with the step's q/k/v copied host->device and the output copied
back inside the timed region), the roofline of the kernel that takes the most time, clocks
sampled during the timed region and the CPU oracle baseline.  The default run adds ``sub``: the
same measurement on the other workloads of the metric -- the 16384-token prefill (prefill
TFLOP/s of the context kernel), the inflight mixed batch with bf16 and FP8 pools, the 70B-like
GQA decode with bf16 and FP8 pools, and the tiny mixed batch (launch overhead) -- each with its
per-kernel fractions of the measured and the nominal peaks and its own clocks.
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

# Nominal GB300 figures (context for the measured fractions): HBM3e bandwidth and dense bf16
# tensor throughput per GPU.
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0

# kernels that read the generation requests' KV (together they move the decode bytes)
DECODE_KERNELS = ("decode_splitkv", "decode_splitkv_wide", "decode_tc")


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


def kernel_rates(work: dict, kern_ms: dict, pk_: dict) -> dict:
    """Per-kernel time and, where the kernel has algorithmic work of its own, its rate and its
    fraction of the measured peak (``frac_*``) and of the nominal GB300 peak (``*_nominal``).
    The decode kernels share the decode bytes: each gets a rate only when it is the only one."""
    dec = [n for n in DECODE_KERNELS if n in kern_ms]
    out = {}
    for n, ms in kern_ms.items():
        d = {"us": ms * 1e3}
        if n in dec and len(dec) == 1 and work["decode_kv_bytes"]:
            gbs = work["decode_bytes"] / (ms * 1e-3) / 1e9
            d.update({"GB/s": gbs, "frac_hbm": gbs / pk_["hbm"], "frac_hbm_nominal": gbs / NOMINAL_HBM_GBS})
        elif n == "context_attn" and work["ctx_flops"]:
            tf = work["ctx_flops"] / (ms * 1e-3) / 1e12
            d.update({"TFLOP/s": tf, "frac_bf16": tf / pk_["bf16"], "frac_bf16_sustained": tf / pk_["bf16_sustained"],
                      "frac_bf16_nominal": tf / NOMINAL_BF16_TFLOPS})
        elif n == "append_rope":
            gbs = work["append_bytes"] / (ms * 1e-3) / 1e9
            d.update({"GB/s": gbs, "frac_hbm": gbs / pk_["hbm"], "frac_hbm_nominal": gbs / NOMINAL_HBM_GBS})
        out[n] = d
    return out


def roofline_of(work: dict, kern_ms: dict, pk_: dict, workload: str) -> dict:
    """Roofline of the kernel class that takes the most time in the step: the decode kernels
    (together, HBM), the context kernel (bf16 tensor) or the append (HBM)."""
    classes = {}
    dec = [n for n in DECODE_KERNELS if n in kern_ms]
    if dec and work["decode_kv_bytes"]:
        classes["+".join(dec)] = sum(kern_ms[n] for n in dec)
    if "context_attn" in kern_ms and work["ctx_flops"]:
        classes["context_attn"] = kern_ms["context_attn"]
    if "append_rope" in kern_ms:
        classes["append_rope"] = kern_ms["append_rope"]
    kernel = max(classes, key=classes.get)
    ms = classes[kernel]
    if kernel == "context_attn":
        ach = work["ctx_flops"] / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": pk_["bf16"], "unit": "TFLOP/s", "frac": ach / pk_["bf16"],
                "peak_nominal": NOMINAL_BF16_TFLOPS, "frac_nominal": ach / NOMINAL_BF16_TFLOPS,
                "frac_sustained": ach / pk_["bf16_sustained"]}
    else:
        nbytes = work["append_bytes"] if kernel == "append_rope" else work["decode_bytes"]
        ach = nbytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk_["hbm"], "unit": "GB/s", "frac": ach / pk_["hbm"],
                "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": ach / NOMINAL_HBM_GBS}
    roof.update({"kernel": kernel, "us_per_launch": ms * 1e3, "peak_source": pk_["src"],
                 "share_of_serial_step": ms / sum(kern_ms.values())})
    roof["traffic"] = ncu_traffic(kernel, workload)
    return roof


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
# CPU oracle baseline (bounded samples)
# --------------------------------------------------------------------------------------------

def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


class OracleSample:
    """The CPU oracle on one generation request at a time (write image of its token, then fp64
    attention for all its heads), cycling through the batch's generation requests."""

    def __init__(self, b):
        import oracle
        self.oracle = oracle
        self.b = b
        self.pool = _bits(b.pool)
        self.q, self.k, self.v = _bits(b.q), _bits(b.k), _bits(b.v)
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


def oracle_context_rate(b, stride: int) -> dict:
    """The CPU oracle on the context rows of a batch: the write image of every new token, then
    fp64 attention (all query heads) of every ``stride``-th context row; the rate is the causal
    flops of those rows over the attention's wall time."""
    import oracle as o
    pool = _bits(b.pool).copy()
    cs = o.rope_table(b.rope_base, b.head_dim, b.max_pos)
    kw = dict(new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
              num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
              num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", kv_int8=b.kv_dtype == "int8")
    st, q_out = o.append_rope(**kw, inv_scale=b.inv_scale, q_bits=_bits(b.q), k_bits=_bits(b.k),
                              v_bits=_bits(b.v), cs=cs, pool=pool)
    q64 = o.f32_from_bf16(q_out).astype(np.float64)
    rows, flops, row0 = [], 0, 0
    for r in range(b.num_contexts):
        n, P = int(b.new_len[r]), int(b.past[r])
        for i in range(0, n, stride):
            rows.append(row0 + i)
            flops += 4 * b.head_dim * b.num_q_heads * (P + i + 1)
        row0 += n
    t0 = time.perf_counter()
    o.attention(**kw, kv_scale=b.kv_scale, pool=pool, q=q64, softmax_scale=b.softmax_scale,
                rows=np.array(rows, dtype=np.int64))
    dt = time.perf_counter() - t0
    return {"tflops": flops / dt / 1e12, "rows": len(rows), "seconds": dt, "flops": flops}


def cpu_baseline(b, ctx_batches=(), budget_s: float = 8.0) -> dict:
    """The oracle as it stands on the host cores: generation requests of the main workload
    (``value``, GB/s) and, for each batch in ``ctx_batches`` ((name, batch, row stride)), its
    context rows (TFLOP/s, sampled every stride-th row and extrapolated to the full prefill)."""
    s = OracleSample(b)
    s.step()  # build / load the oracle outside the timing
    t0, nbytes, n = time.perf_counter(), 0, 0
    while time.perf_counter() - t0 < budget_s and n < 40 * len(s.gen):
        nbytes += s.step()
        n += 1
    dt = time.perf_counter() - t0
    res = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": s.oracle.num_threads(), "kind": "oracle",
           "sample": f"{n} generation requests of the workload (all heads each), fp64 oracle "
                     f"write image + attention, {dt:.1f} s wall"}
    ctx = {}
    for name, cb, stride in ctx_batches:
        c = oracle_context_rate(cb, stride)
        full = work_of(cb)["ctx_flops"]
        ctx[name] = {"value": c["tflops"], "unit": "TFLOP/s", "extrapolated": stride > 1,
                     "sample": f"every {stride}th context row ({c['rows']} rows, all {cb.num_q_heads} query "
                               f"heads), fp64 attention over the pool after the write image, "
                               f"{c['seconds']:.1f} s wall",
                     "full_prefill_s_extrapolated": full / (c["tflops"] * 1e12)}
    if ctx:
        res["context"] = ctx
    return res


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


class Ctx:
    def __init__(self, world, rank, local):
        self.world, self.rank, self.local = world, rank, local
        self.dev = torch.device("cuda", local)
        self.gpu_index = torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local


def measure(cx: Ctx, workload: int, kv_dtype: str, steps: int, warmup: int, *, graph: bool = True,
            e2e: bool = False, bucket: bool = False, max_gen: int | None = None) -> dict:
    """Times K steps of one workload: the step as a whole (default streams), the same K steps with
    per-kernel events (every kernel on the caller's stream), optionally graph replay and the
    end-to-end loop through the public API with host inputs.  Returns the raw measurements."""
    import paged_kv_cache_rope_gb300 as pk
    from paged_kv_cache_rope_gb300 import workloads as W

    world, dev = cx.world, cx.dev
    b = W.workload(workload, kv_dtype=kv_dtype, device=str(dev), poison=False,
                   seed=workload + 1000 * cx.rank, max_gen=max_gen)
    work = work_of(b)
    pool = pk.KVPool(b.pool, b.kv_scale, b.inv_scale)
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev,
                        position_offsets=b.position_offsets, packed_mask=b.packed_mask)
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, dev)
    step = pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)
    q, k, v = b.q, b.k, b.v

    # launches per step and their names
    step(q, k, v)
    torch.cuda.synchronize()
    fwd_names = pk.last_launch_names()
    launches_per_step = 1 + len(fwd_names)

    for _ in range(warmup):
        step(q, k, v)
    torch.cuda.synchronize()

    # (1) the step itself, timed as a whole.  (2) the same K steps again with per-kernel events
    # recorded by the library around each launch; while events are set the library keeps every
    # kernel on the caller's stream (no context/generation overlap), so that each pair of events
    # brackets one kernel's own work.
    ev_app = [pk.KernelEvents(1) for _ in range(steps)]
    ev_fwd = [pk.KernelEvents(len(fwd_names)) for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(cx.gpu_index)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        start.record()
        for _ in range(steps):
            pk.paged_kv_append_rope(pool, meta, step.Hq, q, k, v, step.q_out, table, step.d_error)
            pk.paged_attention_forward(pool, meta, step.Hq, step.q_out, step.out, step.softmax_scale,
                                       step.workspace, step.d_error)
        stop.record()
        torch.cuda.synchronize()
        barrier(world)
        k0.record()
        for i in range(steps):
            with ev_app[i]:
                pk.paged_kv_append_rope(pool, meta, step.Hq, q, k, v, step.q_out, table, step.d_error)
            with ev_fwd[i]:
                pk.paged_attention_forward(pool, meta, step.Hq, step.q_out, step.out, step.softmax_scale,
                                           step.workspace, step.d_error)
        k1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_step, _ = aggregate(1.0, start.elapsed_time(stop), steps, world)
    ms_serial, _ = aggregate(1.0, k0.elapsed_time(k1), steps, world)
    err = int(step.d_error.item())
    if err:
        raise SystemExit(f"device error word {err} during the timed region ({b.name})")

    kern_ms = {"append_rope": statistics.fmean(e.elapsed_ms(0) for e in ev_app)}
    for j, n in enumerate(fwd_names):
        kern_ms[n] = statistics.fmean(e.elapsed_ms(j) for e in ev_fwd)

    res = dict(b=b, work=work, ms_step=ms_step, ms_serial=ms_serial, kern_ms=kern_ms, fwd_names=fwd_names,
               launches_per_step=launches_per_step, clocks=sampler.summary(), graph=None, e2e=None,
               bucket_graph=None)

    # ---- the same step captured once into a CUDA graph and replayed (launch overhead gone) ----
    if graph:
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
            for _ in range(steps):
                cg.replay()
            g1.record()
            torch.cuda.synchronize()
            g_ms, _ = aggregate(1.0, g0.elapsed_time(g1), steps, world)
            res["graph"] = {"ms_per_step": g_ms, "launches_per_step": launches_per_step}
            del cg
        except Exception as exc:  # capture is a measurement extra, never a reason to fail the bench
            res["graph"] = {"error": str(exc)[:200]}

    # ---- the same step on a padding bucket: one graph for every batch of the bucket ----
    # The bucket holds this batch's request slots and rows, with the KV-length limit rounded up
    # to a multiple of 1024 tokens; the replays run this batch through it.
    if bucket and graph:
        try:
            B = b.tokens_per_block
            max_kv = int(-(-int(b.kv_lengths.max()) // 1024) * 1024)
            bk = pk.Bucket(context_slots=b.num_contexts, generation_slots=b.num_requests - b.num_contexts,
                           max_tokens=b.num_tokens, max_context_tokens=b.num_ctx_tokens, max_kv_len=max_kv,
                           max_gen_tokens=int(b.new_len[b.num_contexts:].max()) if b.num_requests > b.num_contexts else 1,
                           max_blocks_per_seq=-(-max_kv // B))
            btable = pk.paged_rope_table_build(b.rope_base, b.head_dim, max(max_kv, b.max_pos), dev)
            bstep = pk.PagedAttentionBucketStep(pool, bk, b.num_q_heads, b.head_dim, btable,
                                                draft=b.position_offsets is not None)
            bstep.load(b.request_types, b.new_len, b.past, b.block_table, q, k, v,
                       position_offsets=b.position_offsets, packed_mask=b.packed_mask)
            bstep.capture()
            for _ in range(3):
                bstep.replay()
            torch.cuda.synchronize()
            barrier(world)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record()
            for _ in range(steps):
                bstep.replay()
            g1.record()
            torch.cuda.synchronize()
            if int(bstep.d_error.item()):
                raise RuntimeError(f"device error word {int(bstep.d_error.item())} in the bucket replay")
            g_ms, _ = aggregate(1.0, g0.elapsed_time(g1), steps, world)
            res["bucket_graph"] = {"ms_per_step": g_ms, "max_kv_len": max_kv, "slots": bk.slots,
                                   "max_tokens": bk.max_tokens}
            del bstep
        except Exception as exc:  # a measurement extra, never a reason to fail the bench
            res["bucket_graph"] = {"error": str(exc)[:200]}

    # ---- e2e through the public API: host q/k/v in pinned memory, output copied back ----
    # Every step copies its q/k/v from pinned host memory and its output back to the host.  The
    # copies run on a second stream, double-buffered, so that step i's output and step i+2's
    # inputs move while step i+1 computes (as a serving loop would run it); two step objects
    # share the pool and own separate output buffers.
    if e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        dbuf = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
        steps2 = [step, pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)]
        hout = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
        xs = torch.cuda.Stream()
        cs = torch.cuda.current_stream()
        e2e_steps = max(10, steps // 4)

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
        res["e2e"] = {"ms_per_step": e2e_ms, "h2d": sum(t.numel() * t.element_size() for t in (hq, hk, hv)),
                      "d2h": hout.numel() * hout.element_size()}
        del steps2, dbuf
    del step, pool, meta, table
    return res


def sub_record(m: dict, world: int, pk_: dict) -> dict:
    """The sub-record of one workload: step times, tokens/s, per-kernel rates and fractions, the
    dominant kernel's roofline and the clocks of its timed region."""
    b, work = m["b"], m["work"]
    wname = b.name + ("" if b.kv_dtype == "bf16" else "_" + b.kv_dtype)
    rec = {"workload": b.name, "kv_dtype": b.kv_dtype, "requests": b.num_requests, "contexts": b.num_contexts,
           "num_tokens": b.num_tokens, "ms_per_step": m["ms_step"], "ms_per_step_serial": m["ms_serial"],
           "tokens_per_s": world * work["tokens"] / (m["ms_step"] * 1e-3),
           "kernels": kernel_rates(work, m["kern_ms"], pk_), "roofline": roofline_of(work, m["kern_ms"], pk_, wname),
           "clocks": m["clocks"]}
    if work["ctx_flops"]:
        rec["prefill_TFLOP/s"] = rec["kernels"]["context_attn"]["TFLOP/s"]
        rec["prefill_frac_bf16"] = rec["kernels"]["context_attn"]["frac_bf16"]
    if m["graph"] is not None:
        rec["graph"] = m["graph"]
    if m["bucket_graph"] is not None:
        rec["bucket_graph"] = m["bucket_graph"]
    return rec


# the workloads of the metric besides the default one: (key, workload, kv dtype)
SUB_WORKLOADS = (
    ("prefill_16k", 5, "bf16"),
    ("mixed", 4, "bf16"),
    ("mixed_fp8", 4, "fp8"),
    ("decode_gqa", 3, "bf16"),
    ("decode_gqa_fp8", 3, "fp8"),
    ("draft", 6, "bf16"),
    ("draft_fp8", 6, "fp8"),
    ("draft_int8", 6, "int8"),
    ("tiny", 1, "bf16"),
)


def run_ours(args):
    world, rank, local = dist_setup()
    cx = Ctx(world, rank, local)
    pk_ = peaks()
    m = measure(cx, args.workload, args.kv_dtype, args.steps, args.warmup, graph=True, e2e=True,
                max_gen=args.max_gen)
    b, work = m["b"], m["work"]
    ms_step = m["ms_step"]
    e2e_ms = m["e2e"]["ms_per_step"]
    if work["decode_kv_bytes"]:
        value = world * work["decode_kv_bytes"] / (ms_step * 1e-3) / 1e9
        e2e_value = world * work["decode_kv_bytes"] / (e2e_ms * 1e-3) / 1e9
        unit = "GB/s"
    else:
        value = world * work["ctx_flops"] / (ms_step * 1e-3) / 1e12
        e2e_value = world * work["ctx_flops"] / (e2e_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    graph = m["graph"]
    if graph and "ms_per_step" in graph:
        w = work["decode_kv_bytes"] or work["ctx_flops"]
        graph["value"] = world * w / (graph["ms_per_step"] * 1e-3) / (1e9 if work["decode_kv_bytes"] else 1e12)
        graph["tokens_per_s"] = world * work["tokens"] / (graph["ms_per_step"] * 1e-3)
    wname = b.name + ("" if b.kv_dtype == "bf16" else "_" + b.kv_dtype)

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
        "pct_of_hbm_nominal": 100.0 * value / NOMINAL_HBM_GBS if unit == "GB/s" else None,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": m["e2e"]["h2d"],
                "d2h_bytes_per_step": m["e2e"]["d2h"], "ms_per_step": e2e_ms},
        "gpu_launches": m["launches_per_step"] * args.steps,
        "graph": graph,
        "kernels": kernel_rates(work, m["kern_ms"], pk_),
        "kernels_timed": "second loop of the same K steps, per-kernel events, all kernels on one stream",
        "ms_per_step_serial": m["ms_serial"],
        "roofline": roofline_of(work, m["kern_ms"], pk_, wname),
        "clocks": m["clocks"],
        "peaks": {"hbm_gbs": pk_["hbm"], "bf16_tflops": pk_["bf16"], "bf16_tflops_sustained": pk_["bf16_sustained"],
                  "source": pk_["src"], "hbm_gbs_nominal": NOMINAL_HBM_GBS, "bf16_tflops_nominal": NOMINAL_BF16_TFLOPS},
    }
    del m
    torch.cuda.empty_cache()

    ctx_cpu = []
    if not args.no_sub and args.workload == 2 and args.max_gen is None:
        # the rest of the metric, measured in the same run: the prefill TFLOP/s half on the 16K
        # prefill, the mixed inflight batch, the GQA decode, draft-token verification on the
        # three pool kinds, the tiny batch's launch overhead
        sub_steps = max(3, min(args.steps, 20))
        subs = {}
        for key, wl, kd in SUB_WORKLOADS:
            ms = measure(cx, wl, kd, sub_steps, args.warmup, graph=True, e2e=False, bucket=key in ("tiny", "mixed"))
            subs[key] = sub_record(ms, world, pk_)
            if rank == 0 and world == 1 and not args.no_cpu_baseline and key in ("prefill_16k", "mixed"):
                ctx_cpu.append((key, ms["b"], 16 if key == "prefill_16k" else 2))
            del ms
            torch.cuda.empty_cache()
        line["sub"] = subs
        line["sub_steps"] = sub_steps
        pf = subs["prefill_16k"]["kernels"]["context_attn"]
        line["prefill"] = {"workload": subs["prefill_16k"]["workload"], "TFLOP/s": pf["TFLOP/s"],
                           "frac_bf16": pf["frac_bf16"], "frac_bf16_sustained": pf["frac_bf16_sustained"],
                           "frac_bf16_nominal": pf["frac_bf16_nominal"], "us_per_launch": pf["us"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b.to("cpu"), [(k, cb.to("cpu"), s) for k, cb, s in ctx_cpu])
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
    ap.add_argument("--no-sub", action="store_true", help="only the main workload (no sub-records)")
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
