"""RoPE + append kernel vs the oracle's write image: bit-exact pool bytes (every byte, poisoned
unused slots included) and bit-exact rotated queries, through the C-ABI."""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import bits, gpu_run, oracle_run

pytestmark = pytest.mark.gpu

CASES = [
    # name, ctx [(n, past)], gen [L], Hq, Hkv, D, B
    ("tiny_d64_b16", [(37, 0)], [54], 4, 2, 64, 16),
    ("mixed_d128_b32", [(100, 0), (33, 64)], [1, 2, 31, 32, 33, 500], 16, 4, 128, 32),
    ("mha_b64", [(70, 5)], [129, 64, 65], 8, 8, 128, 64),
    ("gqa16_b128", [(300, 130)], [255, 256, 257], 32, 2, 128, 128),
    ("decode_only_d64", [], [1, 5, 17, 100, 1000], 16, 8, 64, 16),
]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_append_bit_exact(case, kv_dtype):
    name, ctx, gen, Hq, Hkv, D, B = case
    b = W.make_batch(name=name, ctx=ctx, gen=gen, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                     tokens_per_block=B, kv_dtype=kv_dtype, seed=zlib.crc32(name.encode()) % 1000)
    g = gpu_run(b, attention=False)
    o = oracle_run(b)
    assert g.error == 0 and o.status == 0
    assert np.array_equal(bits(g.q_out), o.q_out)
    assert np.array_equal(bits(g.pool).reshape(-1), o.pool.reshape(-1))


def test_append_in_place_and_fused_qkv_views():
    b = W.make_batch(name="fused", ctx=[(50, 10)], gen=[40, 7], num_q_heads=8, num_kv_heads=2,
                     head_dim=128, tokens_per_block=32, seed=3)
    T, Hq, Hkv, D = b.num_tokens, 8, 2, 128
    qkv = torch.cat([b.q, b.k, b.v], dim=1).cuda()  # one [T, (Hq + 2 Hkv) D] tensor
    q = qkv[:, :Hq * D]
    k = qkv[:, Hq * D:(Hq + Hkv) * D]
    v = qkv[:, (Hq + Hkv) * D:]
    pool = pk.KVPool(b.pool.cuda().clone())
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, "cuda")
    table = pk.paged_rope_table_build(b.rope_base, D, b.max_pos)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pk.paged_kv_append_rope(pool, meta, Hq, q, k, v, q, table, err)  # rotate q in place
    torch.cuda.synchronize()
    o = oracle_run(b)
    assert err.item() == 0
    assert np.array_equal(bits(q.contiguous()), o.q_out)
    assert np.array_equal(bits(pool.data).reshape(-1), o.pool.reshape(-1))


def test_append_flags_bad_page_and_skips_write():
    b = W.make_batch(name="bad", ctx=[], gen=[20, 40], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=4)
    tbl = b.block_table.copy()
    tbl[1, 2] = b.num_blocks + 100  # generation request 1 appends position 39 -> block 2
    b = dataclasses.replace(b, block_table=tbl)
    g = gpu_run(b, attention=False)
    assert g.error & pk.PKV_DEVERR_BAD_PAGE
    o = oracle_run(b)  # the oracle skips the same write
    assert np.array_equal(bits(g.q_out), o.q_out)
    assert np.array_equal(bits(g.pool).reshape(-1), o.pool.reshape(-1))
