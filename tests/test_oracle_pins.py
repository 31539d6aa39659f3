"""Pins for the fp64 CPU oracle: each test ties it to something other than itself.

  * number formats  -> torch's own bf16 / float8_e4m3fn casts (library routines) and the
                       closed values of the OCP E4M3 definition;
  * RoPE            -> closed forms (identity at position 0, unit vectors land on (cos, sin) at
                       (j, j + D/2), D = 2 is complex multiplication, norm preservation, relative
                       position property) and an error bound against the exact fp64 rotation;
  * write image     -> addresses recomputed through torch's 5-D view of the pool, untouched
                       bytes, page-permutation invariance, torch's casts for the stored codes;
  * attention       -> torch scaled_dot_product_attention in fp64 on K/V gathered by torch
                       indexing with an explicit causal mask, plus single key, equal keys,
                       dominant key, causality, chunking and the temperature worked example
                       printed on the pages (tests/golden/temperature_softmax.txt).
All run on the CPU (no GPU marker).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_rope_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------------------------

def test_bf16_rne_matches_torch_cast():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # keep finite values; add exact ties (low half == 0x8000) with both parities
    ties = (rng.integers(0, 2**16, size=20_000, dtype=np.uint32) << 16) | 0x8000
    bits = np.concatenate([bits, ties.astype(np.uint32)])
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ours = oracle.bf16_from_f32(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    finite = np.isfinite(oracle.f32_from_bf16(ref))
    assert np.array_equal(ours[finite], ref[finite])
    # overflow on rounding: torch gives inf, so must we
    assert np.array_equal(ours[~finite], ref[~finite])


def test_bf16_nan_stays_nan():
    out = oracle.bf16_from_f32(np.array([np.nan, -np.nan], dtype=np.float32))
    assert np.all(np.isnan(oracle.f32_from_bf16(out)))


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(ours[~nan], ref[~nan])
    # closed values from the format definition
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0**-9 and ours[0x08] == 2.0**-6 and ours[0x38] == 1.0


def test_e4m3_encode_matches_torch_in_range_and_ties():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.normal(0, 1, 100_000), rng.uniform(-448, 448, 100_000),
                        rng.normal(0, 1e-2, 20_000)]).astype(np.float32)
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact ties between neighbours
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 448.0, -448.0])])
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_nan():
    x = np.float32([449.0, 464.0, 479.9, 1e6, np.inf, -449.0, -1e30, -np.inf])
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 5 + [0xFE] * 3
    assert oracle.e4m3_encode(np.float32([np.nan]))[0] == 0x7F


def test_int8_encode_matches_torch_round_and_clamp():
    """torch.round rounds halves to even, then clamp to [-128, 127] -- an independent route."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 30, 200_000), rng.uniform(-200, 200, 100_000)]).astype(np.float32)
    ties = np.arange(-140, 140, dtype=np.float32) + np.float32(0.5)  # every exact half in range
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 127.0, -128.0, 127.49, -128.49, 1e9, -np.inf, np.inf])])
    ours = oracle.int8_encode(x)
    ref = torch.from_numpy(x.copy()).double().round().clamp(-128, 127).to(torch.int8).numpy()
    assert np.array_equal(ours, ref)
    assert oracle.int8_encode(np.float32([np.nan]))[0] == 0
    assert oracle.int8_encode(np.float32([0.5, 1.5, 2.5, -2.5, 126.5])).tolist() == [0, 2, 2, -2, 126]


# ----------------------------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------------------------

def test_rope_table_values():
    D, base = 64, 1e4
    cs = oracle.rope_table(base, D, 300).astype(np.float64)
    assert np.all(cs[0, :, 0] == 1.0) and np.all(cs[0, :, 1] == 0.0)
    p = np.arange(300)
    # theta_0 = 1: column 0 is (cos p, sin p); theta_{D/4} = base^-1/2 = 0.01
    for j, theta in ((0, 1.0), (D // 4, 0.01)):
        for col, fn in ((0, np.cos), (1, np.sin)):
            exact = fn(p * theta)
            ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
            assert np.all(np.abs(cs[:, j, col] - exact) <= ulp)


def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(3)
    cs = oracle.rope_table(1e4, 128, 1)
    x = oracle.f32_from_bf16(oracle.bf16_from_f32(rng.normal(size=128)))
    assert np.array_equal(oracle.rope32(x, cs[0]), x)


@pytest.mark.parametrize("D", [64, 128])
def test_rope_unit_vectors_land_on_rotate_half_pairs(D):
    """GPT-NeoX rotate-half: e_j (j < D/2) goes to cos at j and sin at j + D/2;
    e_{j+D/2} goes to -sin at j and cos at j + D/2."""
    base, p = 1e4, 37
    cs = oracle.rope_table(base, D, p + 1)
    for j in (0, 5, D // 2 - 1):
        c, s = cs[p, j]
        e = np.zeros(D, np.float32)
        e[j] = 1.0
        y = oracle.rope32(e, cs[p])
        expect = np.zeros(D, np.float32)
        expect[j], expect[j + D // 2] = c, s
        assert np.array_equal(y, expect)
        e = np.zeros(D, np.float32)
        e[j + D // 2] = 1.0
        y = oracle.rope32(e, cs[p])
        expect = np.zeros(D, np.float32)
        expect[j], expect[j + D // 2] = -s, c
        assert np.array_equal(y, expect)


def test_rope_d2_is_complex_multiplication():
    rng = np.random.default_rng(4)
    cs = oracle.rope_table(1e4, 2, 100)
    for p in (1, 17, 99):
        x = rng.normal(size=2)
        z = complex(x[0], x[1]) * np.exp(1j * p * 1.0)  # theta_0 = 1
        y = oracle.rope64(x, 1e4, p)
        assert abs(y[0] - z.real) < 1e-12 and abs(y[1] - z.imag) < 1e-12
        y32 = oracle.rope32(x.astype(np.float32), cs[p])
        assert abs(y32[0] - z.real) < 1e-6 and abs(y32[1] - z.imag) < 1e-6


def test_rope64_norms_and_relative_position():
    rng = np.random.default_rng(5)
    D, base = 128, 1e4
    q, k = rng.normal(size=D), rng.normal(size=D)
    for p in (0, 3, 1000):
        y = oracle.rope64(q, base, p)
        pn_in = q[: D // 2] ** 2 + q[D // 2:] ** 2
        pn_out = y[: D // 2] ** 2 + y[D // 2:] ** 2
        assert np.max(np.abs(pn_in - pn_out)) < 1e-12
    dots = [oracle.rope64(q, base, p) @ oracle.rope64(k, base, s) for p, s in ((10, 3), (507, 500), (7, 0))]
    assert max(dots) - min(dots) < 1e-10


def test_rope32_within_one_bf16_ulp_of_exact():
    rng = np.random.default_rng(6)
    D, base = 128, 5e5
    cs = oracle.rope_table(base, D, 131072)
    for p in rng.integers(0, 131072, 200):
        x = oracle.f32_from_bf16(oracle.bf16_from_f32(rng.normal(size=D)))
        got = oracle.f32_from_bf16(oracle.bf16_from_f32(oracle.rope32(x, cs[p]))).astype(np.float64)
        exact = oracle.rope64(x.astype(np.float64), base, int(p))
        bound = 2.0**-8 * np.abs(exact) + 2e-6 * np.max(np.abs(x))
        assert np.all(np.abs(got - exact) <= bound)


# ----------------------------------------------------------------------------------------------
# write image (O1)
# ----------------------------------------------------------------------------------------------

def _np_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def _run_append(b: W.Batch, pool_np: np.ndarray):
    cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos)
    return oracle.append_rope(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", inv_scale=b.inv_scale,
        q_bits=_np_bits(b.q), k_bits=_np_bits(b.k), v_bits=_np_bits(b.v), cs=cs, pool=pool_np,
        kv_int8=b.kv_dtype == "int8")


def _small_mixed(kv_dtype="bf16", seed=11):
    return W.make_batch(name="pin", ctx=[(21, 0), (9, 32)], gen=[1, 17, 40], num_q_heads=4,
                        num_kv_heads=2, head_dim=64, tokens_per_block=16, kv_dtype=kv_dtype,
                        seed=seed)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_write_image_addresses_and_untouched_bytes(kv_dtype):
    b = _small_mixed(kv_dtype)
    before = _np_bits(b.pool).copy()
    after = before.copy()
    st, q_out = _run_append(b, after)
    assert st == 0
    cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos)
    D, Hkv, Hq = b.head_dim, b.num_kv_heads, b.num_q_heads
    view5 = after.reshape(b.num_blocks, 2, b.tokens_per_block, Hkv, D)
    touched = np.zeros(view5.shape[:3], bool)
    kb, vb, qb = _np_bits(b.k), _np_bits(b.v), _np_bits(b.q)
    row = 0
    for r in range(b.num_requests):
        for i in range(int(b.new_len[r])):
            p = int(b.past[r]) + i
            blk, slot = int(b.block_table[r, p // b.tokens_per_block]), p % b.tokens_per_block
            touched[blk, :, slot] = True
            for h in range(Hkv):
                krot = oracle.rope32(oracle.f32_from_bf16(kb[row, h * D:(h + 1) * D]), cs[p])
                vval = oracle.f32_from_bf16(vb[row, h * D:(h + 1) * D])
                if kv_dtype == "bf16":
                    kref = torch.from_numpy(krot).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                    vref = vb[row, h * D:(h + 1) * D]
                elif kv_dtype == "fp8":
                    enc = lambda a: torch.from_numpy((a * np.float32(b.inv_scale)).astype(np.float32)).to(
                        torch.float8_e4m3fn).view(torch.uint8).numpy()
                    kref, vref = enc(krot), enc(vval)
                else:
                    enc = lambda a: torch.from_numpy((a * np.float32(b.inv_scale)).astype(np.float32)).round().clamp(
                        -128, 127).to(torch.int8).numpy()
                    kref, vref = enc(krot), enc(vval)
                assert np.array_equal(view5[blk, 0, slot, h], kref)
                assert np.array_equal(view5[blk, 1, slot, h], vref)
            for h in range(Hq):
                qrot = oracle.rope32(oracle.f32_from_bf16(qb[row, h * D:(h + 1) * D]), cs[p])
                qref = torch.from_numpy(qrot).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(q_out[row, h * D:(h + 1) * D], qref)
            row += 1
    b5 = before.reshape(view5.shape)
    assert np.array_equal(view5[~touched], b5[~touched])


def test_write_image_page_permutation_invariance():
    b = _small_mixed()
    a1 = _np_bits(b.pool).copy()
    _, q1 = _run_append(b, a1)
    perm = np.random.default_rng(9).permutation(b.num_blocks)
    inv = np.argsort(perm)
    pool2 = b.pool[torch.from_numpy(perm)].contiguous()  # new page n holds old page perm[n]
    tbl2 = np.where(b.block_table >= 0, inv[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    import dataclasses
    b2 = dataclasses.replace(b, pool=pool2, block_table=tbl2)
    a2 = _np_bits(pool2).copy()
    _, q2 = _run_append(b2, a2)
    assert np.array_equal(q1, q2)
    assert np.array_equal(a2.reshape(b.num_blocks, -1), a1.reshape(b.num_blocks, -1)[perm])


def test_write_image_rejects_bad_page():
    b = _small_mixed()
    tbl = b.block_table.copy()
    tbl[3, 1] = b.num_blocks + 5  # generation request 17: its new token lands in block 1
    import dataclasses
    b2 = dataclasses.replace(b, block_table=tbl)
    pool = _np_bits(b.pool).copy()
    st, _ = _run_append(b2, pool)
    assert st == -1


# ----------------------------------------------------------------------------------------------
# attention (O2)
# ----------------------------------------------------------------------------------------------

def _oracle_attention(b: W.Batch, pool_np, q64, rows=None, kv_fp8=None, kv_scale=None):
    return oracle.attention(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=(b.kv_dtype == "fp8") if kv_fp8 is None else kv_fp8,
        kv_scale=b.kv_scale if kv_scale is None else kv_scale, pool=pool_np, q=q64,
        softmax_scale=b.softmax_scale, rows=rows, kv_int8=b.kv_dtype == "int8" and kv_fp8 is None)


def _after_append(b):
    pool = _np_bits(b.pool).copy()
    st, q_out = _run_append(b, pool)
    assert st == 0
    q64 = oracle.f32_from_bf16(q_out).astype(np.float64).reshape(b.num_tokens, b.num_q_heads, b.head_dim)
    return pool, q64


def _sdpa_reference(b: W.Batch, pool_np, q64):
    """Independent route: gather each request's K/V with torch indexing on the 5-D pool view,
    expand GQA by repeat, run torch SDPA in fp64 with an explicit bottom-right causal mask."""
    D, Hkv, Hq, B = b.head_dim, b.num_kv_heads, b.num_q_heads, b.tokens_per_block
    if b.kv_dtype == "fp8":
        vals = torch.from_numpy(oracle.e4m3_decode(pool_np)) * b.kv_scale
    elif b.kv_dtype == "int8":
        vals = torch.from_numpy(pool_np.astype(np.float64)) * b.kv_scale
    else:
        vals = torch.from_numpy(oracle.f32_from_bf16(pool_np).astype(np.float64))
    pool5 = vals.reshape(b.num_blocks, 2, B, Hkv, D)
    outs, row = [], 0
    for r in range(b.num_requests):
        n, P = int(b.new_len[r]), int(b.past[r])
        L = P + n
        t = torch.arange(L)
        blk = torch.from_numpy(b.block_table[r]).long()[t // B]
        K = pool5[blk, 0, t % B]  # [L, Hkv, D]
        V = pool5[blk, 1, t % B]
        K = K.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)  # [Hq, L, D]
        V = V.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
        Q = torch.from_numpy(q64[row:row + n]).permute(1, 0, 2)  # [Hq, n, D]
        mask = t[None, :] <= (P + torch.arange(n))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                             scale=b.softmax_scale)
        outs.append(o.permute(1, 0, 2).numpy())
        row += n
    return np.concatenate(outs, axis=0)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("seed", [11, 12])
def test_attention_matches_sdpa_bruteforce(kv_dtype, seed):
    b = _small_mixed(kv_dtype, seed)
    pool, q64 = _after_append(b)
    st, out = _oracle_attention(b, pool, q64)
    assert st == 0
    ref = _sdpa_reference(b, pool, q64)
    assert np.max(np.abs(out - ref)) < 1e-12


def test_attention_gqa_groups_and_workload1():
    b = W.workload(1)
    pool, q64 = _after_append(b)
    st, out = _oracle_attention(b, pool, q64)
    assert st == 0
    assert np.max(np.abs(out - _sdpa_reference(b, pool, q64))) < 1e-12


def test_attention_single_cached_key_returns_v_row():
    b = W.make_batch(name="one", ctx=[], gen=[1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=3)
    pool, q64 = _after_append(b)
    st, out = _oracle_attention(b, pool, q64)
    assert st == 0
    v = _np_bits(b.v).reshape(2, 2, 64)
    for r in range(2):
        for h in range(4):
            assert np.array_equal(out[r, h], oracle.f32_from_bf16(v[r, h // 2]).astype(np.float64))


def test_attention_equal_keys_gives_mean_of_v_and_dominant_key():
    b = W.make_batch(name="eq", ctx=[], gen=[40], num_q_heads=2, num_kv_heads=1, head_dim=64,
                     tokens_per_block=16, seed=4)
    pool, q64 = _after_append(b)
    P5 = pool.reshape(b.num_blocks, 2, 16, 1, 64)
    blocks = b.block_table[0, :3]
    key = P5[blocks[0], 0, 0, 0].copy()
    for t in range(40):
        P5[blocks[t // 16], 0, t % 16, 0] = key
    st, out = _oracle_attention(b, pool, q64)
    Vs = np.stack([oracle.f32_from_bf16(P5[blocks[t // 16], 1, t % 16, 0]) for t in range(40)])
    assert np.max(np.abs(out[0] - Vs.astype(np.float64).mean(0))) < 1e-12
    # dominant key: scores of key 7 exceed all others by >= 50 -> output is V_7
    q = np.zeros((1, 2, 64))
    q[0, :, 0] = 1.0
    for t in range(40):
        P5[blocks[t // 16], 0, t % 16, 0] = 0
    P5[blocks[0], 0, 7, 0, 0] = oracle.bf16_from_f32(np.float32(50.0 * 8.0))  # scale 1/8
    st, out = _oracle_attention(b, pool, q)
    assert np.max(np.abs(out[0] - Vs[7])) < 1e-12


def test_attention_is_causal():
    b = W.make_batch(name="causal", ctx=[(30, 5)], gen=[], num_q_heads=2, num_kv_heads=1,
                     head_dim=64, tokens_per_block=16, seed=5)
    pool, q64 = _after_append(b)
    st, out1 = _oracle_attention(b, pool, q64)
    P5 = pool.reshape(b.num_blocks, 2, 16, 1, 64)
    cut = 5 + 17  # perturb every K/V at positions > cut
    for t in range(cut + 1, 35):
        P5[b.block_table[0, t // 16], :, t % 16] ^= np.uint16(0x1234)
    st, out2 = _oracle_attention(b, pool, q64)
    assert np.array_equal(out1[:18], out2[:18])       # rows 0..17 see positions <= 22
    assert not np.array_equal(out1[18:], out2[18:])


def test_attention_page_permutation_invariance():
    b = _small_mixed()
    pool, q64 = _after_append(b)
    _, out1 = _oracle_attention(b, pool, q64)
    perm = np.random.default_rng(10).permutation(b.num_blocks)
    inv = np.argsort(perm)
    pool2 = np.ascontiguousarray(pool.reshape(b.num_blocks, -1)[perm])
    tbl2 = np.where(b.block_table >= 0, inv[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    import dataclasses
    _, out2 = _oracle_attention(dataclasses.replace(b, block_table=tbl2), pool2, q64)
    assert np.array_equal(out1, out2)


def test_chunked_prefill_equals_single_prefill_and_generation_row():
    """One 40-token prompt as a single prefill vs as chunks 16 + 16 + 8 over three steps
    (each chunk a multiple of the block size except the last); and a generation step for
    token 40 vs the last row of a 41-token prefill."""
    import dataclasses
    full = W.make_batch(name="full", ctx=[(41, 0)], gen=[], num_q_heads=4, num_kv_heads=2,
                        head_dim=64, tokens_per_block=16, seed=6)
    pool_f, q_f = _after_append(full)
    _, out_f = _oracle_attention(full, pool_f, q_f)
    pool = _np_bits(full.pool).copy()
    row0 = 0
    for n in (16, 16, 8, 1):
        sl = slice(row0, row0 + n)
        typ = W.REQ_CONTEXT if n > 1 else W.REQ_GENERATION
        step = dataclasses.replace(full, request_types=np.int32([typ]), new_len=np.int32([n]),
                                   past=np.int32([row0]), q=full.q[sl], k=full.k[sl], v=full.v[sl])
        st, q_out = _run_append(step, pool)
        assert st == 0
        q64 = oracle.f32_from_bf16(q_out).astype(np.float64).reshape(n, 4, 64)
        _, out = _oracle_attention(step, pool, q64)
        assert np.array_equal(out, out_f[row0:row0 + n])
        row0 += n
    assert np.array_equal(pool, pool_f)


def test_temperature_example_from_the_pages():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "temperature_softmax.txt"))
            if l.strip() and not l.startswith("#")]
    for r in rows:
        T, logits, printed, asserted = float(r[0]), list(map(float, r[1:4])), list(map(float, r[4:7])), r[7] == "1"
        # attention with q = e_0, key t = (logit_t / scale) e_0 and V = identity rows gives
        # softmax(logits) exactly as its output vector
        D = 4
        scale = 1.0 / math.sqrt(D)
        b = W.make_batch(name="temp", ctx=[], gen=[3], num_q_heads=1, num_kv_heads=1, head_dim=D,
                         tokens_per_block=16, seed=7)
        pool = np.zeros((b.num_blocks, 2, 16, 1, D), np.uint16)
        blk = b.block_table[0, 0]
        for t in range(3):
            pool[blk, 0, t, 0, 0] = oracle.bf16_from_f32(np.float32(logits[t] / scale))
            pool[blk, 1, t, 0, t] = oracle.bf16_from_f32(np.float32(1.0))
        q = np.zeros((1, 1, D))
        q[0, 0, 0] = 1.0
        st, out = _oracle_attention(b, pool, q)
        probs = out[0, 0, :3]
        exact = np.exp(np.array(logits) - max(logits))
        exact /= exact.sum()
        assert np.max(np.abs(probs - exact)) < 1e-12
        if asserted:
            assert [round(float(p), 2) for p in probs] == printed


# ----------------------------------------------------------------------------------------------
# append variants: RoPE styles, partial rotary, QK RMSNorm
# ----------------------------------------------------------------------------------------------

def _variant_append(b, pool_np, **kw):
    rot = kw.get("rotary_dim", 0) or b.head_dim
    cs = oracle.rope_table(b.rope_base, rot, b.max_pos)
    return oracle.append_rope_ex(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", inv_scale=b.inv_scale,
        q_bits=_np_bits(b.q), k_bits=_np_bits(b.k), v_bits=_np_bits(b.v), cs=cs, pool=pool_np, **kw)


def test_variant_defaults_equal_plain_append():
    b = _small_mixed()
    p1, p2 = _np_bits(b.pool).copy(), _np_bits(b.pool).copy()
    _, q1 = _run_append(b, p1)
    _, q2 = _variant_append(b, p2)
    assert np.array_equal(q1, q2) and np.array_equal(p1, p2)


def test_gptj_interleaved_unit_vectors():
    """Interleaved pairs: e_{2j} -> cos at 2j, sin at 2j+1; e_{2j+1} -> -sin at 2j, cos at 2j+1."""
    D, p = 64, 23
    b = W.make_batch(name="gptj", ctx=[], gen=[p + 1], num_q_heads=1, num_kv_heads=1, head_dim=D,
                     tokens_per_block=16, seed=2)
    cs = oracle.rope_table(b.rope_base, D, p + 1)
    for j in (0, 7, D // 2 - 1):
        for which, expect in ((2 * j, (cs[p, j, 0], cs[p, j, 1])), (2 * j + 1, (-cs[p, j, 1], cs[p, j, 0]))):
            e = np.zeros((1, D), np.float32)
            e[0, which] = 1.0
            import dataclasses
            bb = dataclasses.replace(b, q=torch.from_numpy(e).to(torch.bfloat16))
            _, q_out = _variant_append(bb, _np_bits(b.pool).copy(), style=1)
            got = oracle.f32_from_bf16(q_out[0])
            ref = np.zeros(D, np.float32)
            ref[2 * j], ref[2 * j + 1] = expect
            assert np.array_equal(got, oracle.f32_from_bf16(oracle.bf16_from_f32(ref)))


@pytest.mark.parametrize("style", [0, 1])
def test_partial_rotary_passes_the_tail_through(style):
    b = _small_mixed()
    rot = 32
    pool = _np_bits(b.pool).copy()
    _, q_out = _variant_append(b, pool, style=style, rotary_dim=rot)
    qb = _np_bits(b.q)
    D = b.head_dim
    q3 = q_out.reshape(b.num_tokens, b.num_q_heads, D)
    q_in = qb.reshape(b.num_tokens, b.num_q_heads, D)
    assert np.array_equal(q3[:, :, rot:], q_in[:, :, rot:])  # untouched dims, bit for bit
    # the rotated part equals a standalone rotation of the first rot dims as a head of size rot
    cs = oracle.rope_table(b.rope_base, rot, b.max_pos)
    row = 0
    for r in range(b.num_requests):
        for i in range(int(b.new_len[r])):
            pos = int(b.past[r]) + i
            for h in range(b.num_q_heads):
                x = oracle.f32_from_bf16(q_in[row, h, :rot])
                if style == 0:
                    ref = oracle.rope32(x, cs[pos])
                else:  # interleaved = rotate-half applied to the de-interleaved vector
                    perm = np.concatenate([np.arange(0, rot, 2), np.arange(1, rot, 2)])
                    y = oracle.rope32(x[perm], cs[pos])
                    ref = np.empty_like(y)
                    ref[perm] = y
                assert np.array_equal(q3[row, h, :rot], oracle.bf16_from_f32(ref))
            row += 1


def test_qk_rmsnorm_matches_formula_and_scale_invariance():
    b = W.make_batch(name="norm", ctx=[(9, 0)], gen=[], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=8)  # past 0: position i, no rotation at row 0
    rng = np.random.default_rng(8)
    qw, kw = rng.uniform(0.5, 1.5, 64).astype(np.float32), rng.uniform(0.5, 1.5, 64).astype(np.float32)
    pool = _np_bits(b.pool).copy()
    _, q_out = _variant_append(b, pool, q_norm_w=qw, k_norm_w=kw, norm_eps=1e-6)
    x = torch.from_numpy(oracle.f32_from_bf16(_np_bits(b.q)[0]).astype(np.float64)).reshape(4, 64)
    ref = x / torch.sqrt((x * x).mean(-1, keepdim=True) + 1e-6) * torch.from_numpy(qw).double()
    got = oracle.f32_from_bf16(q_out[0]).reshape(4, 64).astype(np.float64)
    ulp = np.spacing(np.abs(ref.numpy()).astype(np.float32)).astype(np.float64) * 2**16  # 1 bf16 ulp
    assert np.all(np.abs(got - ref.numpy()) <= ulp)
    # RMSNorm is invariant to scaling the input by a power of two (exact in every format here)
    import dataclasses
    b4 = dataclasses.replace(b, q=(b.q.float() * 4).to(torch.bfloat16), k=(b.k.float() * 4).to(torch.bfloat16),
                             v=(b.v.float() * 4).to(torch.bfloat16))
    pool4 = _np_bits(b.pool).copy()
    _, q_out4 = _variant_append(b4, pool4, q_norm_w=qw, k_norm_w=kw, norm_eps=0.0)
    pool1 = _np_bits(b.pool).copy()
    _, q_out1 = _variant_append(b, pool1, q_norm_w=qw, k_norm_w=kw, norm_eps=0.0)
    assert np.array_equal(q_out4, q_out1)
    view4 = pool4.reshape(b.num_blocks, 2, 16, 2, 64)
    view1 = pool1.reshape(b.num_blocks, 2, 16, 2, 64)
    assert np.array_equal(view4[:, 0], view1[:, 0])        # K normalised: identical
    assert not np.array_equal(view4[:, 1], view1[:, 1])    # V is never normalised (stays 4x)


# ----------------------------------------------------------------------------------------------
# draft tokens: generation requests of several tokens with position offsets and packed masks
# (page adg.csdn.net/69730cc6, section 1.4: generation lengths, position offsets, packed mask)
# ----------------------------------------------------------------------------------------------

def _draft_offsets_all_rows(b: W.Batch) -> np.ndarray:
    """Per packed row: index i for context rows, the batch's offset for generation rows."""
    ctx = [np.arange(int(n), dtype=np.int32) for n in b.new_len[:b.num_contexts]]
    gen = [b.position_offsets] if b.position_offsets is not None else [
        np.concatenate([np.arange(int(n), dtype=np.int32) for n in b.new_len[b.num_contexts:]])]
    return np.concatenate(ctx + gen).astype(np.int32)


def _draft_append(b: W.Batch, pool_np, pos_offset=None, spare_pos=0):
    cs = oracle.rope_table(b.rope_base, b.head_dim, b.max_pos + spare_pos)
    return oracle.append_rope_ex(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", inv_scale=b.inv_scale,
        q_bits=_np_bits(b.q), k_bits=_np_bits(b.k), v_bits=_np_bits(b.v), cs=cs, pool=pool_np,
        pos_offset=_draft_offsets_all_rows(b) if pos_offset is None else pos_offset)


def _draft_attention(b: W.Batch, pool_np, q64, gen_mask):
    return oracle.attention(
        new_len=b.new_len, past=b.past, block_table=b.block_table, num_q_heads=b.num_q_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, tokens_per_block=b.tokens_per_block,
        num_blocks=b.num_blocks, kv_fp8=b.kv_dtype == "fp8", kv_scale=b.kv_scale, pool=pool_np,
        q=q64, softmax_scale=b.softmax_scale, num_contexts=b.num_contexts, gen_mask=gen_mask)


def _draft_batch(kv_dtype="bf16", seed=31, tree=True):
    return W.make_batch(name="draft", ctx=[(19, 5)], gen=[23, (6, 40), (37, 3), (1, 17)],
                        num_q_heads=4, num_kv_heads=2, head_dim=64, tokens_per_block=16,
                        kv_dtype=kv_dtype, seed=seed, draft_tree=tree)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("seed", [31, 32])
def test_draft_tree_attention_matches_sdpa_with_unpacked_mask(kv_dtype, seed):
    """Brute force: the visible-key set of every row rebuilt with numpy's own little-endian bit
    unpacking of the packed words (cached keys always, new key j when its bit is set or j is the
    row itself; context rows causal), then torch SDPA in fp64 over gathered K/V."""
    b = _draft_batch(kv_dtype, seed)
    pool = _np_bits(b.pool).copy()
    st, q_out = _draft_append(b, pool)
    assert st == 0
    T, Hq, D, Hkv, B = b.num_tokens, b.num_q_heads, b.head_dim, b.num_kv_heads, b.tokens_per_block
    q64 = oracle.f32_from_bf16(q_out).astype(np.float64).reshape(T, Hq, D)
    st, out = _draft_attention(b, pool, q64, b.packed_mask)
    assert st == 0
    bits = np.unpackbits(b.packed_mask.astype("<u4").view(np.uint8), axis=1, bitorder="little").astype(bool)
    if kv_dtype == "fp8":
        vals = torch.from_numpy(oracle.e4m3_decode(pool)) * b.kv_scale
    else:
        vals = torch.from_numpy(oracle.f32_from_bf16(pool).astype(np.float64))
    pool5 = vals.reshape(b.num_blocks, 2, B, Hkv, D)
    row, grow = 0, 0
    for r in range(b.num_requests):
        n, P = int(b.new_len[r]), int(b.past[r])
        t = torch.arange(P + n)
        blk = torch.from_numpy(b.block_table[r]).long()[t // B]
        K = pool5[blk, 0, t % B].repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
        V = pool5[blk, 1, t % B].repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
        Q = torch.from_numpy(q64[row:row + n]).permute(1, 0, 2)
        if r < b.num_contexts:
            mask = t[None, :] <= (P + torch.arange(n))[:, None]
        else:
            mask = torch.zeros(n, P + n, dtype=torch.bool)
            mask[:, :P] = True
            mask[:, P:] = torch.from_numpy(bits[grow:grow + n, :n].copy())
            mask[torch.arange(n), P + torch.arange(n)] = True
            grow += n
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=b.softmax_scale)
        assert np.max(np.abs(out[row:row + n] - ref.permute(1, 0, 2).numpy())) < 1e-12
        row += n


def test_draft_chain_mask_equals_causal_across_words():
    """A chain written out as explicit bits (j <= i, 40 tokens: two words per row) must give
    exactly the plain causal result: pins the word (j // 32) and bit (j % 32) addressing."""
    b = _draft_batch(tree=False)
    pool = _np_bits(b.pool).copy()
    st, q_out = _draft_append(b, pool)
    assert st == 0
    q64 = oracle.f32_from_bf16(q_out).astype(np.float64).reshape(b.num_tokens, b.num_q_heads, b.head_dim)
    _, causal = _draft_attention(b, pool, q64, None)
    gen_n = [int(n) for n in b.new_len[b.num_contexts:]]
    mask = np.zeros((sum(gen_n), 2), dtype=np.uint32)
    row = 0
    for n in gen_n:
        for i in range(n):
            for j in range(i + 1):
                mask[row + i, j // 32] |= np.uint32(1 << (j % 32))
        row += n
    st, explicit = _draft_attention(b, pool, q64, mask)
    assert st == 0 and np.array_equal(causal, explicit)
    # and a chain's rows equal the rows of the same tokens sent as a chunked context request
    r = b.num_contexts + 2  # the 37-token request
    import dataclasses
    rows = slice(int(b.new_len[:r].sum()), int(b.new_len[:r + 1].sum()))
    as_ctx = dataclasses.replace(b, request_types=np.int32([W.REQ_CONTEXT]), new_len=b.new_len[r:r + 1],
                                 past=b.past[r:r + 1], block_table=b.block_table[r:r + 1],
                                 q=b.q[rows], k=b.k[rows], v=b.v[rows], position_offsets=None,
                                 packed_mask=None)
    pool2 = _np_bits(b.pool).copy()
    st, q2 = _run_append(as_ctx, pool2)
    q2 = oracle.f32_from_bf16(q2).astype(np.float64).reshape(-1, b.num_q_heads, b.head_dim)
    _, out2 = _oracle_attention(as_ctx, pool2, q2)
    assert np.array_equal(out2, causal[rows])


def test_draft_self_only_mask_equals_one_token_requests():
    """Candidates that are all alternatives for the next position (offset 0, no bits set: each
    sees the cache and itself) equal one-token generation requests, one per candidate, whose
    single new token lands at slot `past` -- bit for bit."""
    import dataclasses
    n, P = 5, 37
    b = W.make_batch(name="siblings", ctx=[], gen=[(n, P)], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=8)
    b = dataclasses.replace(b, position_offsets=np.zeros(n, np.int32), packed_mask=np.zeros((n, 1), np.uint32))
    pool = _np_bits(b.pool).copy()
    st, q_out = _draft_append(b, pool)
    assert st == 0
    q64 = oracle.f32_from_bf16(q_out).astype(np.float64).reshape(n, 4, 64)
    st, out = _draft_attention(b, pool, q64, b.packed_mask)
    assert st == 0
    for i in range(n):
        one = dataclasses.replace(b, new_len=np.int32([1]), past=np.int32([P]), q=b.q[i:i + 1], k=b.k[i:i + 1],
                                  v=b.v[i:i + 1], position_offsets=None, packed_mask=None)
        pool1 = _np_bits(b.pool).copy()
        st, q1 = _run_append(one, pool1)
        assert st == 0 and np.array_equal(q1[0], q_out[i])
        _, o1 = _oracle_attention(one, pool1, oracle.f32_from_bf16(q1).astype(np.float64).reshape(1, 4, 64))
        assert np.array_equal(o1[0], out[i])


def test_draft_position_offsets_rotate_like_a_token_at_that_position():
    """Token i with offset o is rotated exactly as a lone token at position past + o, but is
    stored at slot past + i."""
    import dataclasses
    n, P, offs = 6, 50, [0, 1, 1, 2, 2, 3]
    b = W.make_batch(name="offsets", ctx=[], gen=[(n, P)], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=9)
    b = dataclasses.replace(b, position_offsets=np.int32(offs))
    pool = _np_bits(b.pool).copy()
    st, q_out = _draft_append(b, pool)
    assert st == 0
    view = pool.reshape(b.num_blocks, 2, 16, 2, 64)
    for i, o in enumerate(offs):
        one = dataclasses.replace(b, new_len=np.int32([1]), past=np.int32([P + o]), q=b.q[i:i + 1],
                                  k=b.k[i:i + 1], v=b.v[i:i + 1], position_offsets=None)
        pool1 = _np_bits(b.pool).copy()
        st, q1 = _run_append(one, pool1)
        assert st == 0 and np.array_equal(q1[0], q_out[i])
        v1 = pool1.reshape(view.shape)
        s_one, s_draft = P + o, P + i
        k_one = v1[b.block_table[0, s_one // 16], :, s_one % 16]
        k_draft = view[b.block_table[0, s_draft // 16], :, s_draft % 16]
        assert np.array_equal(k_one, k_draft)  # K (rotated at P + o) and V, at slot P + i


def test_draft_position_offset_out_of_range_is_rejected():
    import dataclasses
    b = W.make_batch(name="badoff", ctx=[], gen=[(4, 20)], num_q_heads=4, num_kv_heads=2, head_dim=64,
                     tokens_per_block=16, seed=10)
    for bad in (4, -1):
        b2 = dataclasses.replace(b, position_offsets=np.int32([0, 1, bad, 2]))
        pool = _np_bits(b.pool).copy()
        st, _ = _draft_append(b2, pool, spare_pos=16)  # the table itself would cover past + 4
        assert st == -2
        view, before = pool.reshape(b.num_blocks, 2, 16, 2, 64), _np_bits(b.pool).reshape(b.num_blocks, 2, 16, 2, 64)
        s = 22  # the skipped token's slot keeps its poison
        blk = b.block_table[0, s // 16]
        assert np.array_equal(view[blk, :, s % 16], before[blk, :, s % 16])
