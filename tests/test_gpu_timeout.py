"""Bounded waits on the GPU: a wait that runs out must set PKV_DEVERR_TIMEOUT, let the kernel
finish (no trap, no hang), free what it holds, and leave the CUDA context usable.

The self-test build of the library (``build_selftest``: the same sources, with the producers of
the two tensor-core kernels -- context and draft-token generation -- issuing no K / V copy and
every bounded wait given about a millisecond) runs a batch's attention: the MMA warp's wait for
the first K tile and the softmax warps' waits for their first S tile can only run out.  The
wait is for copies that are never issued, so no copy is in flight when the kernel tears down
(the producer waits for its Q tile first).  The same step then runs through libpaged_kv.so in
the same process and must match the fp64 oracle.
"""
import ctypes as C
import time

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from helpers import BF16_TOL, max_err, oracle_run
from paged_kv_cache_rope_gb300 import build as pkbuild
from paged_kv_cache_rope_gb300 import workloads as W


def _selftest_lib() -> C.CDLL:
    L = C.CDLL(pkbuild.build_selftest())
    P, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    L.paged_attention_forward.argtypes = [P, P, i32, P, i64, P, C.c_float, P, sz, P, P]
    L.paged_attention_forward.restype = C.c_int
    return L


@pytest.mark.gpu
def test_wait_that_runs_out_sets_timeout_and_context_stays_usable():
    sel = _selftest_lib()
    dev = "cuda"
    b = W.workload(1, device="cpu")
    pool = pk.KVPool(b.pool.to(dev).clone())
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev)
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, dev)
    step = pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)
    q, k, v = b.q.to(dev), b.k.to(dev), b.v.to(dev)
    pk.paged_kv_append_rope(pool, meta, b.num_q_heads, q, k, v, step.q_out, table, step.d_error)
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0

    pc, bc = pool.c(), meta.c()
    t0 = time.perf_counter()
    rc = sel.paged_attention_forward(
        C.byref(pc), C.byref(bc), b.num_q_heads, step.q_out.data_ptr(), step.q_out.stride(0),
        step.out.data_ptr(), float(step.softmax_scale), step.workspace.data_ptr(),
        step.workspace.numel(), step.d_error.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == pk.PKV_OK  # the host sees nothing wrong: the error is the device's to report
    torch.cuda.synchronize()  # returns: every wait of the kernel is bounded
    elapsed = time.perf_counter() - t0
    err = int(step.d_error.item())
    assert err & pk.PKV_DEVERR_TIMEOUT, f"error word {err:#x}: the timeout bit is not set"
    assert err & ~pk.PKV_DEVERR_TIMEOUT == 0, f"error word {err:#x}: unexpected bits"
    assert elapsed < 10.0, f"the stalled launch took {elapsed:.1f} s"

    # the context still works: the same step through the product library, checked against the
    # oracle (the pool already holds this step's tokens; the attention reads it unchanged)
    step.d_error.zero_()
    step.out.fill_(float("nan"))
    pk.paged_attention_forward(pool, meta, b.num_q_heads, step.q_out, step.out, step.softmax_scale,
                               step.workspace, step.d_error)
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0
    ref = oracle_run(b)
    got = step.out.float().cpu().numpy().astype(np.float64).reshape(b.num_tokens, b.num_q_heads, b.head_dim)
    assert max_err(got, ref.out) <= BF16_TOL


@pytest.mark.gpu
def test_generation_kernel_wait_runs_out_and_context_stays_usable():
    """The same on the tensor-core generation kernel: one request verifying an 8-token draft
    tree with 8 query heads per KV head (64 (token, head) rows, beyond the decode kernel's
    columns)."""
    sel = _selftest_lib()
    dev = "cuda"
    b = W.make_batch(name="timeout_gen", ctx=[], gen=[(8, 300), (8, 77)], num_q_heads=16, num_kv_heads=2,
                     head_dim=128, tokens_per_block=32, kv_dtype="bf16", seed=4, draft_tree=True)
    pool = pk.KVPool(b.pool.to(dev).clone())
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev, b.position_offsets, b.packed_mask)
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, dev)
    step = pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)
    q, k, v = b.q.to(dev), b.k.to(dev), b.v.to(dev)
    pk.paged_kv_append_rope(pool, meta, b.num_q_heads, q, k, v, step.q_out, table, step.d_error)
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0
    pk.paged_attention_forward(pool, meta, b.num_q_heads, step.q_out, step.out, step.softmax_scale, step.workspace,
                               step.d_error)
    names = pk.last_launch_names()
    assert "decode_tc" in names, names  # the batch takes the tensor-core generation kernel
    torch.cuda.synchronize()

    pc, bc = pool.c(), meta.c()
    t0 = time.perf_counter()
    rc = sel.paged_attention_forward(
        C.byref(pc), C.byref(bc), b.num_q_heads, step.q_out.data_ptr(), step.q_out.stride(0),
        step.out.data_ptr(), float(step.softmax_scale), step.workspace.data_ptr(),
        step.workspace.numel(), step.d_error.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == pk.PKV_OK
    torch.cuda.synchronize()  # returns: every wait of the kernel is bounded
    elapsed = time.perf_counter() - t0
    err = int(step.d_error.item())
    assert err & pk.PKV_DEVERR_TIMEOUT, f"error word {err:#x}: the timeout bit is not set"
    assert err & ~pk.PKV_DEVERR_TIMEOUT == 0, f"error word {err:#x}: unexpected bits"
    assert elapsed < 10.0, f"the stalled launch took {elapsed:.1f} s"

    step.d_error.zero_()
    step.out.fill_(float("nan"))
    pk.paged_attention_forward(pool, meta, b.num_q_heads, step.q_out, step.out, step.softmax_scale,
                               step.workspace, step.d_error)
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0
    ref = oracle_run(b)
    got = step.out.float().cpu().numpy().astype(np.float64).reshape(b.num_tokens, b.num_q_heads, b.head_dim)
    assert max_err(got, ref.out) <= BF16_TOL
