"""Attention kernels (split-KV decode + LSE combine, tcgen05 context) vs the fp64 oracle through
the C-ABI, on small batches that still span several tiles, pages and splits with ragged tails:
max abs error <= 1e-2 for bf16 pools; FP8 pools <= 4e-2 against the unquantised values and
<= 1e-2 against the dequantised pool.  Also: deterministic reruns, page-permutation invariance,
NaN-poisoned unused slots (every batch here is poisoned), error words."""
import dataclasses
import zlib

import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import workloads as W

from helpers import BF16_TOL, FP8_DEQ_TOL, FP8_TOL, bits, gpu_out_f64, gpu_run, max_err, oracle_run

pytestmark = pytest.mark.gpu


def _batch(name, ctx, gen, Hq, Hkv, D, B, kv_dtype="bf16"):
    return W.make_batch(name=name, ctx=ctx, gen=gen, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        tokens_per_block=B, kv_dtype=kv_dtype, seed=zlib.crc32(name.encode()) % 1000)


DECODE = [
    # name, gen KV lengths, Hq, Hkv, D, B
    ("mha_d128_b64", [1, 2, 15, 16, 17, 63, 64, 65, 511, 777, 2049], 8, 8, 128, 64),
    ("gqa8_d128_b32", [1, 33, 128, 300, 1500, 4097], 64, 8, 128, 32),
    ("gqa4_d64_b16", [3, 16, 250, 999], 16, 4, 64, 16),
    ("gqa16_d128_b128", [5, 129, 1000], 32, 2, 128, 128),
    ("gqa2_d64_b64", [70, 2000], 4, 2, 64, 64),
    ("gqa3_d128_b16", [40, 600], 6, 2, 128, 16),
    # one long request of a small batch: 64-key splits, 130 of them (the widest combine, 16
    # warps over the splits)
    ("gqa2_d128_130_splits", [8300, 40], 4, 2, 128, 64),
]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_matches_oracle(case, kv_dtype):
    name, gen, Hq, Hkv, D, B = case
    b = _batch(name, [], gen, Hq, Hkv, D, B, kv_dtype)
    g = gpu_run(b)
    assert g.error == 0
    got = gpu_out_f64(g, b)
    o = oracle_run(b)
    assert o.status == 0
    if kv_dtype == "bf16":
        assert max_err(got, o.out) <= BF16_TOL
    else:
        # kernel arithmetic: against the oracle on the same (dequantised) 8-bit pool
        assert max_err(got, o.out) <= FP8_DEQ_TOL
        # quantisation: against the unquantised values the kernel may add at most the kernel
        # tolerance to the error the 8-bit codes themselves cause (measured exactly by the oracle)
        unq = oracle_run(b, unquantised=True).out
        inherent = max_err(o.out, unq, label="unquantised")
        assert max_err(got, unq, label="unquantised") <= inherent + FP8_DEQ_TOL


CONTEXT = [
    # name, ctx [(n, past)], gen, Hq, Hkv, D, B
    ("ctx_one_token", [(1, 0)], [], 4, 2, 128, 64),
    ("ctx_37_d64_b16", [(37, 0)], [], 4, 2, 64, 16),
    ("ctx_128_exact", [(128, 0)], [], 8, 8, 128, 64),
    ("ctx_129_tail", [(129, 0)], [], 8, 2, 128, 32),
    ("ctx_chunked", [(300, 192), (77, 64)], [], 16, 4, 128, 64),
    ("ctx_unaligned_past", [(200, 37)], [], 8, 4, 128, 16),
    ("ctx_b128", [(260, 128)], [], 8, 1, 128, 128),
    ("ctx_d64_gqa16", [(150, 20)], [], 32, 2, 64, 32),
    ("mixed", [(37, 0), (130, 70)], [54, 1, 300], 8, 2, 128, 16),
]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
@pytest.mark.parametrize("case", CONTEXT, ids=[c[0] for c in CONTEXT])
def test_context_matches_oracle(case, kv_dtype):
    name, ctx, gen, Hq, Hkv, D, B = case
    b = _batch(name, ctx, gen, Hq, Hkv, D, B, kv_dtype)
    g = gpu_run(b)
    assert g.error == 0
    o = oracle_run(b)
    assert o.status == 0
    got = gpu_out_f64(g, b)
    if kv_dtype == "bf16":
        assert max_err(got, o.out) <= BF16_TOL
    else:  # 8-bit pool: context pages are staged as exact bf16 code values first
        assert max_err(got, o.out) <= FP8_DEQ_TOL
        unq = oracle_run(b, unquantised=True).out
        assert max_err(got, unq, label="unquantised") <= max_err(o.out, unq, label="unquantised") + FP8_DEQ_TOL


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [128, 64])
def test_context_many_units_per_cta(D, kv_dtype):
    """More (unit, query head) items than SMs: every persistent context CTA claims several items
    of different shapes in turn (full and partial 256-row units, long and short cached prefixes,
    one-row requests), carrying its rings, TMEM and the output staging tile from one item to the
    next.  Every row of every head is checked against the oracle."""
    rng = np.random.default_rng(77 + D)
    ctx = []
    for i in range(40):
        n = int(rng.choice([1, 5, 128, 129, 256, 300, 511, 600]))
        ctx.append((n, int(rng.integers(0, 700))))
    b = _batch(f"many_units_d{D}", ctx, [], 8, 2, D, 32, kv_dtype)
    units = sum((n + 255) // 256 for n, _ in ctx)
    assert units * 8 > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    g = gpu_run(b)
    assert g.error == 0
    o = oracle_run(b)
    assert o.status == 0
    assert max_err(gpu_out_f64(g, b), o.out) <= (BF16_TOL if kv_dtype == "bf16" else FP8_DEQ_TOL)
    g2 = gpu_run(b)  # the queue order differs from run to run; the results do not
    assert torch.equal(g.out, g2.out)


def test_deterministic_and_page_permutation_invariant():
    b = _batch("perm", [(200, 100)], [900, 45, 3000], 16, 4, 128, 32)
    g1, g2 = gpu_run(b), gpu_run(b)
    assert torch.equal(g1.out, g2.out)
    perm = np.random.default_rng(5).permutation(b.num_blocks)
    inv = np.argsort(perm)
    tbl = np.where(b.block_table >= 0, inv[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    b2 = dataclasses.replace(b, pool=b.pool[torch.from_numpy(perm)].contiguous(), block_table=tbl)
    g3 = gpu_run(b2)
    assert torch.equal(g1.out, g3.out)
    # pools hold NaN poison in unused slots: compare bit patterns
    assert torch.equal(g1.pool[torch.from_numpy(perm).cuda()].view(torch.int16), g3.pool.view(torch.int16))


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_overlapped_and_serial_schedules_agree(kv_dtype):
    """A mixed batch runs its generation kernels on the library's auxiliary stream beside the
    context kernel; with per-kernel timing events set, everything runs on the caller's stream.
    Each output row is written by one kernel either way, so the two must agree bit for bit."""
    b = _batch("overlap_" + kv_dtype, [(300, 64), (40, 0)], [900, 45, 3000, 1], 16, 4, 128, 32, kv_dtype)
    overlapped = gpu_run(b)
    with pk.KernelEvents(8):
        serial = gpu_run(b)
    assert overlapped.error == 0 and serial.error == 0
    assert torch.equal(overlapped.out, serial.out)
    o = oracle_run(b)
    tol = BF16_TOL if kv_dtype == "bf16" else FP8_DEQ_TOL
    assert max_err(gpu_out_f64(overlapped, b), o.out) <= tol


def test_decode_bad_page_sets_error_word():
    b = _batch("badread", [], [100, 300], 8, 2, 128, 32)
    tbl = b.block_table.copy()
    tbl[1, 3] = -5  # a cached (not appended) page of request 1
    g = gpu_run(dataclasses.replace(b, block_table=tbl))
    assert g.error & pk.PKV_DEVERR_BAD_PAGE


def test_context_bad_page_sets_error_word():
    b = _batch("badctx", [(200, 128)], [], 8, 2, 128, 64)
    tbl = b.block_table.copy()
    tbl[0, 1] = b.num_blocks  # cached page
    g = gpu_run(dataclasses.replace(b, block_table=tbl))
    assert g.error & pk.PKV_DEVERR_BAD_PAGE


def test_launch_counts():
    b = _batch("launches", [(100, 0)], [5000, 20], 8, 2, 128, 64)
    g = gpu_run(b)
    assert g.launches == 5  # append, plan, context, decode, combine
    g8 = gpu_run(_batch("launches8", [(100, 0)], [5000, 20], 8, 2, 128, 64, "fp8"))
    assert g8.launches == 6  # append, plan, stage_q8, context, decode, combine


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8", "int8"])
def test_prefix_shared_pages(kv_dtype):
    """Prefix reuse: several requests' block tables point at the same physical pages for a
    common cached prefix (read-only); each request's own new tokens land in pages of its own."""
    b = _batch("shared_" + kv_dtype, [(70, 96)], [200, 150, 97], 8, 2, 128, 32, kv_dtype)
    tbl = b.block_table.copy()
    donor = b.num_requests - 1  # the 97-token decode: its first 3 pages hold 96 cached tokens
    for r in range(b.num_requests - 1):
        tbl[r, :3] = tbl[donor, :3]
    b2 = dataclasses.replace(b, block_table=tbl)
    g = gpu_run(b2)
    assert g.error == 0
    o = oracle_run(b2)
    assert o.status == 0
    tol = BF16_TOL if kv_dtype == "bf16" else FP8_DEQ_TOL
    assert max_err(gpu_out_f64(g, b2), o.out) <= tol
    assert np.array_equal(bits(g.pool).reshape(-1), o.pool.reshape(-1))
