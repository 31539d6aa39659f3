"""Shared test plumbing: run one batch through the CUDA library (via the C-ABI binding) and
through the CPU oracle, on the same seeded inputs."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

BF16_TOL = 1e-2       # max abs error vs the fp64 oracle, bf16 pool
FP8_TOL = 4e-2        # the FP8-pool bar, taken against the fp64 oracle on the same FP8 pool
FP8_DEQ_TOL = 1e-2    # what the kernels are held to against that oracle (tighter than FP8_TOL);
                      # INT8 pools are held to the same bar against the oracle on the INT8 pool


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


@dataclasses.dataclass
class GpuResult:
    pool: torch.Tensor       # pool after the append (device)
    q_out: torch.Tensor      # rotated q (device)
    out: torch.Tensor        # attention output (device)
    error: int               # device error word
    launches: int


def gpu_run(b: W.Batch, device: str = "cuda", attention: bool = True) -> GpuResult:
    """Append (+ attention) through the C-ABI on a fresh copy of the batch's pool."""
    pool = pk.KVPool(b.pool.to(device).clone(), b.kv_scale, b.inv_scale)
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, device,
                        position_offsets=b.position_offsets, packed_mask=b.packed_mask)
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, device)
    step = pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)
    q, k, v = b.q.to(device), b.k.to(device), b.v.to(device)
    if attention:
        out = step(q, k, v)
    else:
        pk.paged_kv_append_rope(pool, meta, b.num_q_heads, q, k, v, step.q_out, table, step.d_error)
        out = step.out
    torch.cuda.synchronize()
    return GpuResult(pool.data, step.q_out, out, int(step.d_error.item()), step.launches)


@dataclasses.dataclass
class OracleResult:
    pool: np.ndarray         # write image (bits)
    q_out: np.ndarray        # bf16 bits [T, Hq*D]
    out: np.ndarray          # fp64 [T, Hq, D] (NaN for rows not computed)
    status: int


def oracle_run(b: W.Batch, rows=None, unquantised: bool = False) -> OracleResult:
    """O1 + O2 on the batch.  ``unquantised`` runs an 8-bit batch on its bf16 twin pool."""
    use_twin = unquantised and b.kv_dtype != "bf16"
    pool_np = bits(b.pool_bf16 if use_twin else b.pool).copy()
    fp8 = b.kv_dtype == "fp8" and not use_twin
    i8 = b.kv_dtype == "int8" and not use_twin
    cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos)
    args = dict(new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
                num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
                num_blocks=b.num_blocks, kv_fp8=fp8, inv_scale=b.inv_scale, q_bits=bits(b.q),
                k_bits=bits(b.k), v_bits=bits(b.v), cs=cs, pool=pool_np, kv_int8=i8)
    if b.position_offsets is None:
        st, q_out = oracle.append_rope(**args)
    else:  # draft tokens: context rows keep i, generation rows take the batch's offsets
        ctx = [np.arange(int(n), dtype=np.int32) for n in b.new_len[:b.num_contexts]]
        st, q_out = oracle.append_rope_ex(**args, pos_offset=np.concatenate(ctx + [b.position_offsets]))
    q64 = oracle.f32_from_bf16(q_out).astype(np.float64)
    st2, out = oracle.attention(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=fp8, kv_scale=b.kv_scale if (fp8 or i8) else 1.0, pool=pool_np,
        q=q64, softmax_scale=b.softmax_scale, rows=rows, num_contexts=b.num_contexts,
        gen_mask=b.packed_mask, kv_int8=i8)
    return OracleResult(pool_np, q_out, out, st or st2)


def gpu_out_f64(res: GpuResult, b: W.Batch) -> np.ndarray:
    return res.out.float().cpu().numpy().astype(np.float64).reshape(b.num_tokens, b.num_q_heads, b.head_dim)


def bf16_step(x: np.ndarray) -> np.ndarray:
    """Spacing of the bf16 grid at |x|: 2^(e - 7) for |x| in [2^e, 2^(e + 1))."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


# Every max_err call of the running test, for the session's parity report (conftest prints
# it): (test [label], plain max abs error, error as judged, elements that needed the allowance,
# elements).  Label "oracle": a result against the fp64 oracle on the same pool; "unquantised":
# against the oracle on the unquantised values of an 8-bit pool (quantisation error included).
PARITY_LOG: list[tuple[str, float, float, int, int]] = []
CURRENT_TEST = ""


def max_err(gpu: np.ndarray, ref: np.ndarray, rows=None, label: str = "oracle") -> float:
    """Max abs error of bf16 results against the fp64 oracle, read at the bf16 output's own
    resolution.  Where one bf16 step at the reference value is wider than the 1e-2 bar
    (|ref| >= 2: steps of 2^-6 and more), the part of that step beyond the bar is not counted:
    a result one step away from the rounded reference -- an fp32 value a hair on the other side
    of a rounding midpoint -- is the limit of the output format, not of the kernel.  For
    |ref| < 2 this is the plain max abs error."""
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    assert np.all(np.isfinite(ref))
    if not np.all(np.isfinite(gpu)):
        return float("inf")
    if not gpu.size:
        return 0.0
    allowance = np.maximum(0.0, bf16_step(ref) - BF16_TOL)
    diff = np.abs(gpu - ref)
    judged = float(np.max(diff - allowance))
    # elements over the plain 1e-2 bar that the allowance brought back under it
    used = int(np.count_nonzero((diff > BF16_TOL) & (diff - allowance <= BF16_TOL)))
    PARITY_LOG.append((f"{CURRENT_TEST} [{label}]", float(np.max(diff)), judged, used, int(diff.size)))
    return judged
