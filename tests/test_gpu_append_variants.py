"""Append variants through paged_kv_append_rope_ex vs the oracle: rotate-half / interleaved
RoPE and partial rotary dims are bit-exact (same fixed fp32 recipe); with a QK RMSNorm the
kernel's fp32 sum of squares against the oracle's fp64 one allows one unit in the last place of
the stored format.  Attention over the variant-written pool is checked end to end."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import BF16_TOL, FP8_DEQ_TOL, bits, max_err

pytestmark = pytest.mark.gpu


def _ordered(u16: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values (for ulp distances)."""
    i = u16.astype(np.int32)
    return np.where(i & 0x8000, 0x8000 - i, i)


def _run(b, **kw):
    dev = "cuda"
    rot = kw.get("rotary_dim", 0) or b.head_dim
    pool = pk.KVPool(b.pool.to(dev).clone(), b.kv_scale, b.inv_scale)
    meta = pk.BatchMeta(b.request_types, b.new_len, b.past, b.block_table, dev)
    table = pk.paged_rope_table_build(b.rope_base, rot, b.max_pos, dev)
    q_out = torch.empty(b.num_tokens, b.num_q_heads * b.head_dim, dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gkw = dict(kw)
    for name in ("q_norm_w", "k_norm_w"):
        w = gkw.pop(name, None)
        gkw[name.replace("_w", "_weight")] = None if w is None else torch.from_numpy(w).to(dev)
    gkw.pop("norm_eps", None)
    if "style" in gkw:
        gkw["rope_style"] = gkw.pop("style")
    pk.paged_kv_append_rope_ex(pool, meta, b.num_q_heads, b.q.to(dev), b.k.to(dev), b.v.to(dev), q_out, table,
                               err, norm_eps=kw.get("norm_eps", 1e-6), **gkw)
    torch.cuda.synchronize()
    assert err.item() == 0
    cs = oracle.rope_table(b.rope_base, rot, b.max_pos)
    opool = bits(b.pool).copy()
    st, oq = oracle.append_rope_ex(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", inv_scale=b.inv_scale, q_bits=bits(b.q),
        k_bits=bits(b.k), v_bits=bits(b.v), cs=cs, pool=opool, **kw)
    assert st == 0
    return pool, meta, q_out, opool, oq


def _batch(name, kv_dtype, D=128):
    return W.make_batch(name=name, ctx=[(45, 16), (130, 0)], gen=[300, 17], num_q_heads=8, num_kv_heads=2,
                        head_dim=D, tokens_per_block=32, kv_dtype=kv_dtype, seed=zlib.crc32(name.encode()) % 997)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("style,rot,D", [(0, 0, 128), (1, 0, 128), (0, 64, 128), (1, 32, 128), (1, 0, 64),
                                         (0, 48, 64)])
def test_rope_variants_bit_exact(style, rot, D, kv_dtype):
    b = _batch(f"var{style}{rot}{D}", kv_dtype, D)
    pool, _, q_out, opool, oq = _run(b, style=style, rotary_dim=rot)
    assert np.array_equal(bits(q_out), oq)
    assert np.array_equal(bits(pool.data).reshape(-1), opool.reshape(-1))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("style", [0, 1])
def test_qk_rmsnorm_within_one_ulp_and_attention(style, kv_dtype):
    b = _batch(f"norm{style}", kv_dtype)
    rng = np.random.default_rng(3)
    qw = rng.uniform(0.5, 1.5, b.head_dim).astype(np.float32)
    kw = rng.uniform(0.5, 1.5, b.head_dim).astype(np.float32)
    pool, meta, q_out, opool, oq = _run(b, style=style, q_norm_w=qw, k_norm_w=kw, norm_eps=1e-6)
    assert np.max(np.abs(_ordered(bits(q_out)) - _ordered(oq))) <= 1
    g5 = bits(pool.data).reshape(b.num_blocks, 2, -1)
    o5 = opool.reshape(b.num_blocks, 2, -1)
    assert np.array_equal(g5[:, 1], o5[:, 1])  # V untouched by the norm: exact
    if kv_dtype == "bf16":
        assert np.max(np.abs(_ordered(g5[:, 0]) - _ordered(o5[:, 0]))) <= 1
    else:  # one E4M3 step at most (codes of one sign are ordered like their values)
        gk, ok_ = g5[:, 0].astype(np.int32), o5[:, 0].astype(np.int32)
        same = (gk & 0x80) == (ok_ & 0x80)
        assert np.all(np.abs(gk - ok_)[same] <= 1) and np.all((gk | ok_)[~same] & 0x7F <= 1)
    if kv_dtype == "bf16":  # end to end: attention over the variant-written pool
        out = torch.empty_like(q_out)
        ws = torch.empty(pk.paged_attention_workspace_size(pool, meta, b.num_q_heads), dtype=torch.uint8,
                         device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pk.paged_attention_forward(pool, meta, b.num_q_heads, q_out, out, b.softmax_scale, ws, err)
        torch.cuda.synchronize()
        st, ref = oracle.attention(
            new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
            num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
            num_blocks=b.num_blocks, kv_fp8=False, kv_scale=1.0, pool=opool,
            q=oracle.f32_from_bf16(oq).astype(np.float64), softmax_scale=b.softmax_scale)
        got = out.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
        assert max_err(got, ref) <= BF16_TOL
