"""paged_attention_forward_noalloc: the attention entry point for callers that cannot allocate
device memory where they call it (no workspace argument; the library's own static scratch
buffer is used instead).  Its outputs must match the regular entry point's on the same batch,
on two calls in a row (the shared buffer keeps the previous call's contents), and a batch that
needs more scratch than the buffer holds must be refused before anything runs.

This file is collected last on purpose, and passes both alone in a fresh process (the first
call on the device performs the buffer's address lookup) and after the other tests."""
import ctypes as C

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import BF16_TOL

pytestmark = pytest.mark.gpu


def _setup(b: W.Batch):
    pool = pk.KVPool(b.pool.cuda().clone(), b.kv_scale, b.inv_scale)
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, "cuda")
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_out = torch.empty(b.num_tokens, b.num_q_heads * b.head_dim, dtype=torch.bfloat16, device="cuda")
    pk.paged_kv_append_rope(pool, meta, b.num_q_heads, b.q.cuda(), b.k.cuda(), b.v.cuda(), q_out, table, err)
    return pool, meta, q_out, err


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_noalloc_matches_regular_entry_point_twice(kv_dtype):
    # two chunked/fresh contexts and decodes long enough to split
    b = W.make_batch(name="noalloc", ctx=[(300, 64), (37, 0)], gen=[5, 700, 3000, 129], num_q_heads=16, num_kv_heads=4,
                     head_dim=128, tokens_per_block=32, kv_dtype=kv_dtype, seed=21)
    pool, meta, q_out, err = _setup(b)
    ref = torch.empty(b.num_tokens, b.num_q_heads * b.head_dim, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pk.paged_attention_workspace_size(pool, meta, b.num_q_heads), dtype=torch.uint8, device="cuda")
    pk.paged_attention_forward(pool, meta, b.num_q_heads, q_out, ref, b.softmax_scale, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for _ in range(2):  # the second call runs on the scratch the first one left behind
        out = torch.full_like(ref, float("nan"))
        pk.paged_attention_forward_noalloc(pool, meta, b.num_q_heads, q_out, out, b.softmax_scale, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= BF16_TOL, diff
        assert torch.equal(out, ref)  # same kernels, same plan: bit-identical in practice


def test_noalloc_refuses_batches_beyond_its_scratch():
    # 1024 generation requests of 100k tokens need far more than 64 MiB of split partials; the
    # host sizes this from the host lengths and refuses before launching.  The device buffers
    # are real (page 0 everywhere, in range) so nothing could read out of bounds regardless.
    R, L, B, Hq, Hkv, D = 1024, 100_000, 64, 32, 8, 128
    mb = -(-L // B)
    types = np.full(R, pk.PKV_REQ_GENERATION, np.int32)
    meta = pk.BatchMeta(types, np.ones(R, np.int32), np.full(R, L - 1, np.int32), np.zeros((R, mb), np.int32), "cuda")
    pool = pk.KVPool(torch.zeros(4, 2, B, Hkv, D, dtype=torch.bfloat16, device="cuda"))
    need = pk.paged_attention_workspace_size(pool, meta, Hq)
    assert need > pk.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(R, Hq * D, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pc, bc = pool.c(), meta.c()
    code = pk.lib().paged_attention_forward_noalloc(C.byref(pc), C.byref(bc), Hq, q.data_ptr(), q.stride(0),
                                                    out.data_ptr(), C.c_float(D ** -0.5), err.data_ptr(),
                                                    torch.cuda.current_stream().cuda_stream)
    assert code == -6  # PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert err.item() == 0 and torch.count_nonzero(out).item() == 0
