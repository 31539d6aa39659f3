"""Host side of padding buckets (CPU): PagedAttentionBucketStep.load places a batch into the
bucket's fixed slots (context requests into the first context slots, generation requests into
the first generation slots, every other slot empty with no new tokens) and refuses batches that
do not fit; the workspace size depends on the bucket only."""
import numpy as np
import pytest
import torch

import paged_kv_cache_rope_gb300 as pk
from paged_kv_cache_rope_gb300 import build as pkbuild

HQ, HKV, D, B = 8, 2, 64, 16


@pytest.fixture(scope="module")
def step():
    pkbuild.build()
    pool = pk.KVPool(torch.zeros(64, 2, B, HKV, D, dtype=torch.bfloat16))
    bucket = pk.Bucket(context_slots=2, generation_slots=3, max_tokens=100, max_context_tokens=80,
                       max_kv_len=256, max_gen_tokens=4, max_blocks_per_seq=16)
    table = torch.zeros(256, D // 2, 2, dtype=torch.float32)
    return pk.PagedAttentionBucketStep(pool, bucket, HQ, D, table, draft=True)


def _rows(T, H):
    return torch.arange(T * H * D, dtype=torch.float32).reshape(T, H * D).to(torch.bfloat16)


def test_load_places_requests_in_slots(step):
    types, n, past = [0, 1, 1], [30, 2, 1], [5, 100, 7]
    tbl = np.arange(3 * 8, dtype=np.int32).reshape(3, 8)
    T = sum(n)
    q, k, v = _rows(T, HQ), _rows(T, HKV), _rows(T, HKV)
    offs = np.array([0, 1, 0], np.int32)
    mask = np.array([[1], [3], [1]], np.uint32)
    step.load(types, n, past, tbl, q, k, v, position_offsets=offs, packed_mask=mask)
    assert step.num_tokens == T
    assert step.meta.d_context_lengths.tolist() == [30, 0, 2, 1, 0]
    assert step.meta.d_past_kv_lengths.tolist() == [5, 0, 100, 7, 0]
    t = step.meta.d_block_offsets
    assert t[0, :8].tolist() == tbl[0].tolist() and (t[0, 8:] == -1).all()
    assert (t[1] == -1).all() and (t[4] == -1).all()
    assert t[2, :8].tolist() == tbl[1].tolist() and t[3, :8].tolist() == tbl[2].tolist()
    assert torch.equal(step.q[:T], q) and torch.equal(step.k[:T], k) and torch.equal(step.v[:T], v)
    assert step.meta.d_position_offsets[:3].tolist() == [0, 1, 0]
    assert step.meta.d_packed_mask[:3, 0].tolist() == [1, 3, 1]


@pytest.mark.parametrize("types,n,past,why", [
    ([0, 0, 0], [10, 10, 10], [0, 0, 0], "slots"),                # 3 contexts, 2 context slots
    ([1, 1, 1, 1], [1, 1, 1, 1], [0, 0, 0, 0], "slots"),          # 4 generations, 3 slots
    ([0, 1], [81, 1], [0, 0], "rows"),                            # context rows over 80
    ([0, 1], [60, 1], [0, 256], "limits"),                        # past + new over 256
    ([0, 1], [60, 5], [0, 0], "limits"),                          # 5 draft tokens over 4
    ([1, 0], [1, 10], [0, 0], "first"),                           # a context after a generation
])
def test_load_refuses_batches_over_the_bucket(step, types, n, past, why):
    T = sum(n)
    tbl = np.zeros((len(n), 4), np.int32)
    with pytest.raises(pk.PagedKVError):
        step.load(types, n, past, tbl, _rows(T, HQ), _rows(T, HKV), _rows(T, HKV))


def test_bucket_workspace_depends_on_the_bucket_only(step):
    a = pk.paged_attention_bucket_workspace_size(step.pool, step.meta, HQ)
    step.meta.d_past_kv_lengths.fill_(200)  # device contents are never read on the host
    assert pk.paged_attention_bucket_workspace_size(step.pool, step.meta, HQ) == a > 0
