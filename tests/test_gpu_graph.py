"""A whole layer step (append + attention) captured into a CUDA graph and replayed: the entry
points only enqueue work (no allocation, no synchronisation), so capture works and replays
reproduce the direct-launch results bit for bit."""
import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_graph_replay_matches_direct(kv_dtype):
    b = W.make_batch(name="graph", ctx=[(150, 40)], gen=[700, 33, 2000], num_q_heads=16, num_kv_heads=4,
                     head_dim=128, tokens_per_block=32, kv_dtype=kv_dtype, seed=31)
    dev = "cuda"
    table = pk.paged_rope_table_build(b.rope_base, b.head_dim, b.max_pos, dev)
    q, k, v = b.q.to(dev), b.k.to(dev), b.v.to(dev)

    def make():
        pool = pk.KVPool(b.pool.to(dev).clone(), b.kv_scale, b.inv_scale)
        meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev)
        return pk.PagedAttentionStep(pool, meta, b.num_q_heads, b.head_dim, table)

    direct = make()
    direct(q, k, v)
    torch.cuda.synchronize()
    ref_out, ref_pool = direct.out.clone(), direct.pool.data.clone()

    step = make()
    pool0 = step.pool.data.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (first-call set-up per kernel)
        step(q, k, v)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(q, k, v)
    for _ in range(2):
        step.pool.data.copy_(pool0)
        step.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert step.d_error.item() == 0
        assert torch.equal(step.out, ref_out)
        assert np.array_equal(bits(step.pool.data), bits(ref_pool))
