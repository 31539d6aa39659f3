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


def test_roofline_follows_the_kernel_that_takes_the_most_time():
    """The reported roofline belongs to the kernel class with the largest measured time: the
    context kernel on a prefill-heavy step, the decode kernels (together) on a decode step."""
    pk_ = dict(hbm=6000.0, bf16=2000.0, bf16_sustained=1800.0, src="test")
    work = dict(decode_kv_bytes=6e8, decode_bytes=6.1e8, ctx_flops=2e12, append_bytes=1e8, tokens=100)
    prefill_heavy = {"append_rope": 0.05, "plan": 0.01, "context_attn": 1.3, "decode_splitkv": 0.4}
    r = bench.roofline_of(work, prefill_heavy, pk_, "none")
    assert r["kernel"] == "context_attn" and r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 2e12 / 1.3e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 2000.0) < 1e-12
    assert abs(r["frac_nominal"] - r["achieved"] / bench.NOMINAL_BF16_TFLOPS) < 1e-12
    decode_heavy = {"append_rope": 0.05, "context_attn": 0.1, "decode_splitkv": 0.3, "decode_tc": 0.2}
    r = bench.roofline_of(work, decode_heavy, pk_, "none")
    assert r["kernel"] == "decode_splitkv+decode_tc" and r["bound"] == "hbm"
    assert abs(r["achieved"] - 6.1e8 / 0.5e-3 / 1e9) < 1e-9
    k = bench.kernel_rates(work, decode_heavy, pk_)
    assert "GB/s" not in k["decode_splitkv"]  # two decode kernels share the bytes
    assert abs(k["context_attn"]["frac_bf16_nominal"] - 2e12 / 0.1e-3 / 1e12 / bench.NOMINAL_BF16_TFLOPS) < 1e-12
