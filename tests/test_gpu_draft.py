"""Generation requests of several draft tokens (page adg.csdn.net/69730cc6, section 1.4: generation
lengths, position offsets, packed mask; the Medusa candidate tree on page "TensorRT-LLM 源码完全
拆解(一)") through the C-ABI against the fp64 oracle: draft tokens rotated for past + offset and
stored at past + i (bit-exact pool and q_out), attention under chain (causal) or tree masks.
Narrow requests run on the split-KV decode kernel, whose score-tile columns are (token, query
head) pairs of one KV head; wider ones on the tcgen05 generation kernel (rows = those
pairs; 8-bit pools at head_dim 128 have their codes converted to f16 in shared memory) or, for
groups that do not divide 128 and 8-bit pools at head_dim 64, on the wide mma.sync kernel."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import BF16_TOL, FP8_DEQ_TOL, bits, gpu_out_f64, gpu_run, max_err, oracle_run

pytestmark = pytest.mark.gpu

CASES = [
    # name, ctx, gen (draft tokens, cached) or KV length, Hq, Hkv, D, B, tree
    ("chain_gqa4_d128", [], [(4, 300), (7, 1000), 50, (16, 2000)], 32, 8, 128, 64, False),
    ("tree_gqa4_d64_2words", [], [(5, 700), (13, 33), (40, 1500), (64, 3000)], 8, 2, 64, 16, True),
    ("tree_mha_d128_16tok", [], [(16, 900), (3, 17), 5000], 8, 8, 128, 32, True),
    ("chain_gqa16", [], [(2, 64), (3, 4100), 700], 32, 2, 128, 128, False),
    ("group32_single", [], [900, 33, 4097], 64, 2, 128, 64, False),
    ("mixed_ctx_tree", [(200, 64), (31, 0)], [(6, 500), 1200, (9, 2500)], 16, 4, 128, 32, True),
    # tensor-core generation kernel: one head per row (g = 1), several 128-row groups per request
    ("tree_mha_d64_64tok", [], [(64, 300), (20, 5000), 70], 4, 4, 64, 16, True),
    ("tree_gqa8_row_groups", [], [(20, 700), (64, 2000), (16, 4100)], 16, 2, 128, 32, True),
    # 16-token pages: eight pages per 128-key tile (one TMA box per producer lane)
    ("tree_gqa4_d128_b16", [], [(6, 900), (12, 2600), 40], 16, 4, 128, 16, True),
    # a group that does not divide 128 keeps the mma.sync wide kernel on every pool
    ("tree_gqa6_mma_wide", [], [(5, 300), (9, 1000), 77], 12, 2, 128, 32, True),
]


def _batch(case, kv_dtype):
    name, ctx, gen, Hq, Hkv, D, B, tree = case
    return W.make_batch(name=name, ctx=ctx, gen=gen, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        tokens_per_block=B, kv_dtype=kv_dtype, seed=len(name) * 7 + 3, draft_tree=tree)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_draft_tokens_match_oracle(case, kv_dtype):
    b = _batch(case, kv_dtype)
    g = gpu_run(b)
    assert g.error == 0
    o = oracle_run(b)
    assert o.status == 0
    assert np.array_equal(bits(g.pool).reshape(-1), o.pool.reshape(-1))  # write image, bit-exact
    assert np.array_equal(bits(g.q_out), o.q_out)
    tol = BF16_TOL if kv_dtype == "bf16" else FP8_DEQ_TOL
    assert max_err(gpu_out_f64(g, b), o.out) <= tol


def test_draft_request_alone_and_in_a_batch():
    """A draft request's rows match the oracle both when it runs alone and inside a batch, where
    other requests' splits and column groups share the launch (nothing leaks between them)."""
    b = _batch(CASES[2], "bf16")
    g_all = gpu_run(b)
    rows = slice(0, int(b.new_len[0]))  # the 16-token request
    alone = dataclasses.replace(b, request_types=b.request_types[:1], new_len=b.new_len[:1], past=b.past[:1],
                                block_table=b.block_table[:1], q=b.q[rows], k=b.k[rows], v=b.v[rows],
                                position_offsets=b.position_offsets[rows], packed_mask=b.packed_mask[rows])
    g1 = gpu_run(alone)
    assert g1.error == 0
    o = oracle_run(alone)
    assert max_err(gpu_out_f64(g1, alone), o.out) <= BF16_TOL
    assert max_err(gpu_out_f64(g_all, b)[rows], o.out) <= BF16_TOL


def test_draft_bad_offset_sets_error_and_skips_the_token():
    b = _batch(CASES[1], "bf16")
    off = b.position_offsets.copy()
    off[3] = int(b.new_len[0])  # first request has 5 tokens: offset 5 is out of range
    b2 = dataclasses.replace(b, position_offsets=off)
    g = gpu_run(b2, attention=False)
    assert g.error & pk.PKV_DEVERR_BAD_OFFSET
    import oracle
    cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos)
    pool_np = bits(b.pool).copy()
    ctx = []
    st, q_out = oracle.append_rope_ex(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=False, inv_scale=b.inv_scale, q_bits=bits(b.q), k_bits=bits(b.k),
        v_bits=bits(b.v), cs=cs, pool=pool_np, pos_offset=np.concatenate(ctx + [off]).astype(np.int32))
    assert st == -2
    assert np.array_equal(bits(g.pool).reshape(-1), pool_np.reshape(-1))
    good = np.ones(b.num_tokens, bool)
    good[3] = False
    assert np.array_equal(bits(g.q_out)[good], q_out[good])


def test_draft_deterministic_and_overlap_agrees():
    b = _batch(CASES[5], "bf16")
    g1, g2 = gpu_run(b), gpu_run(b)
    assert torch.equal(g1.out, g2.out)
    with pk.KernelEvents(8):
        g3 = gpu_run(b)  # every kernel on one stream
    assert torch.equal(g1.out, g3.out)
