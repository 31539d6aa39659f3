"""The bench's algorithmic-work definitions (the numerators of every reported roofline fraction),
checked against brute-force counts on small batches: context flops count 2 flops per MAC of
QK^T and of PV over the causal part only; decode bytes read each KV head once per generation
request; 8-bit pools move one byte per element."""
import numpy as np

import bench
from paged_kv_cache_rope_gb300 import workloads as W


def _brute(b):
    D, Hq, Hkv = b.head_dim, b.num_q_heads, b.num_kv_heads
    esz = 1 if b.kv_dtype != "bf16" else 2
    flops = 0
    kv_bytes = 0
    for r in range(len(b.new_len)):
        n, past = int(b.new_len[r]), int(b.past[r])
        if b.request_types[r] == 0:  # context: row i sees keys 0 .. past + i
            for i in range(n):
                keys = past + i + 1
                flops += Hq * keys * D * 2 * 2  # QK^T and PV, 2 flops per MAC
        else:  # generation: every key of the request, K and V, each KV head once
            kv_bytes += (past + n) * Hkv * D * 2 * esz
    return flops, kv_bytes


def test_context_flops_and_decode_bytes_match_brute_force():
    b = W.make_batch(name="work", ctx=[(37, 0), (20, 45)], gen=[54, (3, 17), 300], num_q_heads=8,
                     num_kv_heads=2, head_dim=64, tokens_per_block=16, kv_dtype="bf16", seed=3,
                     draft_tree=True)
    flops, kv_bytes = _brute(b)
    w = bench.work_of(b)
    assert w["ctx_flops"] == flops
    assert w["decode_kv_bytes"] == kv_bytes
    gen_rows = int(np.sum(b.new_len[b.request_types == 1]))
    assert w["decode_bytes"] == kv_bytes + gen_rows * 2 * b.num_q_heads * b.head_dim * 2


def test_eight_bit_pools_move_half_the_decode_bytes():
    wb = bench.work_of(W.workload(3, kv_dtype="bf16", poison=False, max_gen=8))
    w8 = bench.work_of(W.workload(3, kv_dtype="fp8", poison=False, max_gen=8))
    wi = bench.work_of(W.workload(3, kv_dtype="int8", poison=False, max_gen=8))
    assert 2 * w8["decode_kv_bytes"] == wb["decode_kv_bytes"] == 2 * wi["decode_kv_bytes"]
    assert w8["ctx_flops"] == wb["ctx_flops"] == 0
