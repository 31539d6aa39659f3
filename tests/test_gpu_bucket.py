"""Padding buckets: one CUDA graph, captured once per bucket, replayed over different batches.

The pages motivate fixed-shape buckets by the graph hit rate ("TensorRT-LLM 1.0 源码学习笔记",
section 五 5.2, CUDA graph: a graph is only replayed when the batch shape repeats) and allocate
the graph's metadata once ("TensorRT-LLM 源码完全拆解(一)", "AttentionMetadata 的字段与它的含义",
create_cuda_graph_metadata).  Here a step over a bucket takes every launch shape from the bucket,
so each replay reads whatever batch the fixed device arrays hold.  Every replayed batch is
checked against the fp64 oracle: the pool write image bit for bit, the attention rows within the
parity tolerance, and no device error bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from helpers import BF16_TOL, FP8_DEQ_TOL, bits, max_err, oracle_run
from paged_kv_cache_rope_gb300 import workloads as W

DEV = "cuda"
HQ, HKV, D, B = 32, 8, 128, 64
NB = 400


def _batch(ctx, gen, seed, kv_dtype="bf16", draft=False, Hq=HQ, Hkv=HKV, num_blocks=NB):
    return W.make_batch(name="bucket", ctx=ctx, gen=gen, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        tokens_per_block=B, kv_dtype=kv_dtype, seed=seed, num_blocks=num_blocks,
                        draft_tree=draft)


def _check(step, b, scale=None):
    """Loads nothing: compares the step's pool and output rows for batch ``b`` (whose pool the
    step's pool started from) with the oracle."""
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0, f"device error word {int(step.d_error.item()):#x}"
    bo = b if scale is None else dataclasses.replace(b, kv_scale=scale[0], inv_scale=scale[1])
    ref = oracle_run(bo)
    assert ref.status == 0
    got_pool = bits(step.pool.data).reshape(-1)
    assert np.array_equal(got_pool, ref.pool.reshape(-1)), "pool write image differs from the oracle"
    T = b.num_tokens
    assert np.array_equal(bits(step.q_out[:T]), ref.q_out), "rotated q differs from the oracle"
    got = step.out[:T].float().cpu().numpy().astype(np.float64).reshape(T, b.num_q_heads, D)
    tol = BF16_TOL if b.kv_dtype == "bf16" else FP8_DEQ_TOL
    err = max_err(got, ref.out)
    assert err <= tol, f"max abs error {err}"
    return err


def _run(step, b, replay=True, scale=None):
    step.pool.data.copy_(b.pool.to(DEV))  # this batch's cached history, outside the graph
    step.load(b.request_types, b.new_len, b.past, b.block_table, b.q.to(DEV), b.k.to(DEV), b.v.to(DEV),
              position_offsets=b.position_offsets, packed_mask=b.packed_mask)
    step.d_error.zero_()
    if replay:
        step.replay()
    else:
        step()
    return _check(step, b, scale)


def _fixed_scale(batches, kv_dtype):
    """8-bit pools: a captured graph holds the pool's scales, so every batch uses one pair."""
    amax = max(float(b.pool_bf16.float().nan_to_num(0.0).abs().max()) for b in batches)
    amax = max([amax] + [float(t.float().abs().max()) for b in batches for t in (b.k, b.v)])
    s = float(np.float32(amax / (127.0 if kv_dtype == "int8" else 448.0)))
    return s, float(np.float32(1.0 / s))


def _encode(pool_bf16, kv_dtype, inv_scale):
    """The history re-encoded with one scale: e4m3 by torch's cast after a clamp, int8 by
    round-half-even and a clamp; unused slots keep the poison code."""
    x = pool_bf16.float().nan_to_num(0.0) * inv_scale
    unused = pool_bf16.view(torch.int16) == W.BF16_NAN
    if kv_dtype == "int8":
        codes = x.round().clamp(-128.0, 127.0).to(torch.int8)
        codes[unused] = W.INT8_POISON
    else:
        codes = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        codes[unused] = W.E4M3_NAN
    return codes


@pytest.mark.gpu
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_one_graph_serves_batches_of_different_mixes(kv_dtype):
    """Captured once on the first batch, replayed on: the same mix with other lengths, only
    generation requests, only context requests (chunked, with cached prefixes), and one long
    context request beside one generation request."""
    bucket = pk.Bucket(context_slots=3, generation_slots=12, max_tokens=1200, max_context_tokens=1100,
                       max_kv_len=2048, max_gen_tokens=1, max_blocks_per_seq=32)
    rng = np.random.default_rng(11)
    batches = [
        _batch([(300, 0), (500, 128)], rng.integers(100, 2048, 5).tolist(), 1, kv_dtype),
        _batch([(200, 64), (100, 0)], rng.integers(1, 2048, 7).tolist(), 2, kv_dtype),
        _batch([], rng.integers(1000, 2048, 12).tolist(), 3, kv_dtype),
        _batch([(100, 0), (400, 64), (37, 1500)], [], 4, kv_dtype),
        _batch([(1000, 1000)], [2048], 5, kv_dtype),
    ]
    scale = _fixed_scale(batches, kv_dtype) if kv_dtype != "bf16" else None
    if scale is not None:  # re-encode every pool with the one scale the graph holds
        for i, b in enumerate(batches):
            batches[i] = dataclasses.replace(b, pool=_encode(b.pool_bf16, kv_dtype, scale[1]),
                                             kv_scale=scale[0], inv_scale=scale[1])
    b0 = batches[0]
    pool = pk.KVPool(b0.pool.to(DEV).clone(), b0.kv_scale, b0.inv_scale)
    table = pk.paged_rope_table_build(1e4, D, bucket.max_kv_len, DEV)
    step = pk.PagedAttentionBucketStep(pool, bucket, HQ, D, table)
    step.load(b0.request_types, b0.new_len, b0.past, b0.block_table, b0.q.to(DEV), b0.k.to(DEV), b0.v.to(DEV))
    step.capture()
    for b in batches:
        _run(step, b, replay=True, scale=scale)


@pytest.mark.gpu
def test_draft_token_bucket_replays_trees_of_different_sizes():
    """Generation slots of up to 8 draft tokens (tensor-core generation kernel), replayed over
    requests of 1 to 8 tokens with random candidate trees, beside a context request."""
    Hq, Hkv = 64, 8
    bucket = pk.Bucket(context_slots=1, generation_slots=6, max_tokens=400, max_context_tokens=300,
                       max_kv_len=1600, max_gen_tokens=8, max_blocks_per_seq=25)
    mk = lambda ctx, gen, seed: _batch(ctx, gen, seed, draft=True, Hq=Hq, Hkv=Hkv)
    batches = [
        mk([(200, 0)], [(8, 900), (8, 1200), (3, 40), (1, 700)], 21),
        mk([], [(8, 1500), (5, 1000), (8, 7), (2, 300), (6, 1590), (1, 1)], 22),
        mk([(300, 1200)], [(4, 100)], 23),
    ]
    b0 = batches[0]
    pool = pk.KVPool(b0.pool.to(DEV).clone())
    table = pk.paged_rope_table_build(1e4, D, bucket.max_kv_len, DEV)
    step = pk.PagedAttentionBucketStep(pool, bucket, Hq, D, table, draft=True)
    step.load(b0.request_types, b0.new_len, b0.past, b0.block_table, b0.q.to(DEV), b0.k.to(DEV), b0.v.to(DEV),
              position_offsets=b0.position_offsets, packed_mask=b0.packed_mask)
    step.capture()
    for b in batches:
        _run(step, b, replay=True)


@pytest.mark.gpu
def test_random_batches_fill_their_bucket_without_overflow():
    """Direct (uncaptured) bucket calls on random batches drawn inside one bucket: the device
    plan's counts never exceed the capacities the host sized the grids and the workspace for
    (that would set PKV_DEVERR_BUCKET), and every result matches the oracle."""
    bucket = pk.Bucket(context_slots=2, generation_slots=10, max_tokens=700, max_context_tokens=600,
                       max_kv_len=1500, max_gen_tokens=1, max_blocks_per_seq=24)
    rng = np.random.default_rng(31)
    pool = None
    for t in range(6):
        nc, ng = int(rng.integers(0, 3)), int(rng.integers(0, 11))
        if nc + ng == 0:
            ng = 1
        ctx = []
        left = 600
        for _ in range(nc):
            if left < 1:
                break
            n = int(rng.integers(1, min(left, 1500) + 1))
            left -= n
            ctx.append((n, int(rng.integers(0, 1500 - n + 1))))
        gen = rng.integers(1, 1501, ng).tolist()
        b = _batch(ctx, gen, 40 + t)
        if pool is None:
            pool = pk.KVPool(b.pool.to(DEV).clone())
            table = pk.paged_rope_table_build(1e4, D, bucket.max_kv_len, DEV)
            step = pk.PagedAttentionBucketStep(pool, bucket, HQ, D, table)
        _run(step, b, replay=False)


@pytest.mark.gpu
def test_batch_over_the_bucket_sets_bucket_error_and_next_batch_is_fine():
    """A batch whose device lengths break the bucket (past + new beyond max_kv_len) is rejected
    on the device: PKV_DEVERR_BUCKET, nothing after the append runs, the context stays usable."""
    bucket = pk.Bucket(context_slots=1, generation_slots=4, max_tokens=300, max_context_tokens=200,
                       max_kv_len=1024, max_gen_tokens=1, max_blocks_per_seq=16)
    b = _batch([(150, 0)], [500, 900, 1024], 51)
    pool = pk.KVPool(b.pool.to(DEV).clone())
    table = pk.paged_rope_table_build(1e4, D, bucket.max_kv_len, DEV)
    step = pk.PagedAttentionBucketStep(pool, bucket, HQ, D, table)
    step.load(b.request_types, b.new_len, b.past, b.block_table, b.q.to(DEV), b.k.to(DEV), b.v.to(DEV))
    step.capture()
    step.meta.d_past_kv_lengths[2] = 1500  # a generation slot now reaches past the bucket
    step.d_error.zero_()
    step.out.fill_(float("nan"))
    step.replay()
    torch.cuda.synchronize()
    assert int(step.d_error.item()) & pk.PKV_DEVERR_BUCKET
    assert torch.isnan(step.out.float()).all(), "a rejected batch must not write the output"
    _run(step, b, replay=True)


@pytest.mark.gpu
def test_device_lengths_that_disagree_with_the_host_plan_run_nothing():
    """Without a bucket the grids come from the host copies of the lengths: device copies that
    disagree are a plan mismatch, the plan's counts are zero and no attention kernel writes."""
    b = _batch([(150, 0)], [500, 900], 61)
    pool = pk.KVPool(b.pool.to(DEV).clone())
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, DEV)
    table = pk.paged_rope_table_build(1e4, D, b.max_pos, DEV)
    step = pk.PagedAttentionStep(pool, meta, HQ, D, table)
    step(b.q.to(DEV), b.k.to(DEV), b.v.to(DEV))
    torch.cuda.synchronize()
    assert int(step.d_error.item()) == 0
    meta.d_past_kv_lengths[1] = 100  # the host still says 499
    step.out.fill_(float("nan"))
    pk.paged_attention_forward(pool, meta, HQ, step.q_out, step.out, step.softmax_scale, step.workspace,
                               step.d_error)
    torch.cuda.synchronize()
    assert int(step.d_error.item()) & pk.PKV_DEVERR_PLAN_MISMATCH
    assert torch.isnan(step.out.float()).all()
