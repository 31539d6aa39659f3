"""CPU-only checks of the C-ABI library: it builds for sm_103a, loads, exports every symbol the
header declares, rejects bad arguments on the host, and its RoPE table matches the oracle's
bit for bit (the table is the one input the kernels and the oracle must share exactly)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import build as pkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pkbuild.build()
    return pk.lib()


def test_header_declarations_are_exported(L):
    header = open(os.path.join(ROOT, "include", "paged_kv.h")).read()
    declared = set(re.findall(r"^[A-Za-z_][\w \t*]*?\b(paged_\w+)\s*\(", header, re.M))
    assert declared == set(pk.EXPORTS), declared ^ set(pk.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(0, -8, -1):
        s = pk.status_string(code)
        assert s and s != "unknown status"


def test_rope_table_matches_oracle_bitwise(L):
    for base, D, max_pos in ((1e4, 64, 300), (1e4, 128, 5000), (5e5, 128, 131072)):
        ours = np.empty((max_pos, D // 2, 2), dtype=np.float32)
        assert L.paged_rope_table_build(C.c_double(base), D, max_pos, ours.ctypes.data) == 0
        ref = oracle.rope_table(base, D, max_pos)
        assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))
    assert L.paged_rope_table_bytes(128, 10) == 10 * 128 * 4


def _descs(D=128, B=64, dtype=pk.PKV_BF16, types=(0, 1), lens=(5, 1), past=(0, 9), nb=8, mb=4):
    pool = pk.PkvPool(0x1000, dtype, nb, B, 8, D, 1.0, 1.0)
    t = np.array(types, np.int32)
    n = np.array(lens, np.int32)
    p = np.array(past, np.int32)
    keep = (t, n, p)
    batch = pk.PkvBatch(len(n), int((t == 0).sum()), int(n.sum()), mb, t.ctypes.data, n.ctypes.data,
                        p.ctypes.data, 0x2000, 0x3000, 0x4000)
    return pool, batch, keep


def _fwd(L, pool, batch, Hq=32, q=0x10000, out=0x20000, ws=0x30000, ws_bytes=1 << 20):
    return L.paged_attention_forward(C.byref(pool), C.byref(batch), Hq, q, Hq * pool.head_dim, out,
                                     C.c_float(0.088), ws, ws_bytes, 0x5000, None)


@pytest.mark.parametrize("mutate,code", [
    (dict(D=96), -2),
    (dict(B=24), -2),
    (dict(dtype=7), -2),
    (dict(types=(1, 0), lens=(1, 5), past=(9, 0)), -3),   # generation before context
    (dict(lens=(5, 65), mb=8), -3),                        # generation beyond 64 draft tokens
    (dict(past=(0, 300)), -4),                             # exceeds 4 blocks x 64
])
def test_host_rejects_bad_batches(L, mutate, code):
    pool, batch, keep = _descs(**mutate)
    assert _fwd(L, pool, batch) == code


def test_host_rejects_bad_heads_alignment_workspace(L):
    pool, batch, keep = _descs()
    assert _fwd(L, pool, batch, Hq=12) == -2          # 12 % 8 != 0
    assert L.paged_attention_workspace_size(C.byref(pool), C.byref(batch), 256) > 0  # any group size plans
    assert _fwd(L, pool, batch, q=0x10004) == -5      # misaligned q
    assert _fwd(L, pool, batch, ws=0) == -6           # no workspace
    assert _fwd(L, pool, batch, ws_bytes=16) == -6    # too small
    need = L.paged_attention_workspace_size(C.byref(pool), C.byref(batch), 32)
    assert need > 0 and need % 256 == 0
    empty = pk.PkvBatch(0, 0, 0, 1, None, None, None, None, None, None)
    assert _fwd(L, pool, empty) == 0                  # empty batch is a no-op
    fp8, batch2, keep2 = _descs(dtype=pk.PKV_FP8_E4M3)
    fp8.kv_scale_quant_orig = float("nan")
    assert _fwd(L, fp8, batch2) == -1


def test_append_rejects_capacity_of_rope_table(L):
    pool, batch, keep = _descs()
    code = L.paged_kv_append_rope(C.byref(pool), C.byref(batch), 32, 0x10000, 32 * 128, 0x20000, 8 * 128,
                                  0x30000, 8 * 128, 0x10000, 32 * 128, 0x40000, 8, 0x5000, None)
    assert code == -4   # past 9 + 1 > max_pos 8


def test_host_checks_draft_mask_words(L):
    pool, batch, keep = _descs(lens=(5, 40), mb=4)
    batch.d_packed_mask = 0x6000
    batch.mask_words = 0
    assert _fwd(L, pool, batch) == -1                 # a mask needs words
    batch.mask_words = 1
    assert _fwd(L, pool, batch) == -1                 # 40 draft tokens need two words per row
    assert L.paged_attention_workspace_size(C.byref(pool), C.byref(batch), 32) == 0
    batch.mask_words = 2
    assert L.paged_attention_workspace_size(C.byref(pool), C.byref(batch), 32) > 0


def _bucket_descs(C_slots=2, G_slots=6, T=600, mb=16, B=64, dtype=pk.PKV_BF16):
    pool = pk.PkvPool(0x1000, dtype, 256, B, 8, 128, 1.0, 1.0)
    batch = pk.PkvBatch(C_slots + G_slots, C_slots, T, mb, None, None, None, 0x2000, 0x3000, 0x4000)
    return pool, batch


def test_bucket_host_checks(L):
    """Bucket calls read no host lengths (NULL host arrays are fine); the host checks the slot
    layout and the bucket's limits against the block table, the RoPE table and the draft cap."""
    pool, batch = _bucket_descs()
    ok = pk.PkvBucket(512, 1000, 1)
    assert L.paged_attention_bucket_workspace_size(C.byref(pool), C.byref(batch), C.byref(ok), 32) > 0

    def fwd(bk, Hq=32):
        return L.paged_attention_forward_bucket(C.byref(pool), C.byref(batch), C.byref(bk), Hq, 0x10000, Hq * 128,
                                                0x20000, C.c_float(0.088), 0x30000, 1 << 30, 0x5000, None)
    assert fwd(pk.PkvBucket(512, 16 * 64 + 1, 1)) == -4   # past + new beyond the block table
    assert fwd(pk.PkvBucket(601, 1000, 1)) == -1          # more context rows than rows
    assert fwd(pk.PkvBucket(512, 1000, 65)) == -3         # beyond 64 draft tokens
    assert fwd(pk.PkvBucket(512, 1000, 0)) == -3          # generation slots need >= 1 token
    assert fwd(ok, Hq=12) == -2
    small = L.paged_attention_bucket_workspace_size(C.byref(pool), C.byref(batch), C.byref(ok), 32)
    assert L.paged_attention_forward_bucket(C.byref(pool), C.byref(batch), C.byref(ok), 32, 0x10000, 32 * 128,
                                            0x20000, C.c_float(0.088), 0x30000, small - 256, 0x5000, None) == -6
    code = L.paged_kv_append_rope_bucket(C.byref(pool), C.byref(batch), C.byref(ok), 32, 0x10000, 32 * 128,
                                         0x20000, 8 * 128, 0x30000, 8 * 128, 0x10000, 32 * 128, 0x40000, 999,
                                         None, 0x5000, None)
    assert code == -4                                     # the RoPE table must cover max_kv_len
