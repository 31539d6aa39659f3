"""Python binding of libpaged_kv.so, the GB300 (sm_103a) paged-KV RoPE + attention library.

Argument marshalling only: every step of the hot path runs in the library's CUDA kernels.
PyTorch provides device memory and streams.  The entry points keep the C names:

    paged_rope_table_build(base, head_dim, max_pos, device)        -> fp32 table on the device
    paged_kv_append_rope(pool, batch, num_q_heads, q, k, v, q_out, rope_table, d_error)
    paged_attention_workspace_size(pool, batch, num_q_heads)       -> bytes
    paged_attention_forward(pool, batch, num_q_heads, q_rot, out, softmax_scale, workspace, d_error)

``pool`` is a :class:`KVPool` (the [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]
tensor plus its dtype and FP8 scales) and ``batch`` a :class:`BatchMeta` (host and device
copies of the per-request metadata).  A missing or unloadable library raises immediately; there
is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import dataclasses
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_kv.so")

PKV_OK = 0
PKV_BF16 = 0
PKV_FP8_E4M3 = 1
PKV_INT8 = 2
PKV_REQ_CONTEXT = 0
PKV_REQ_GENERATION = 1
PKV_DEVERR_BAD_PAGE = 1
PKV_DEVERR_TIMEOUT = 2
PKV_DEVERR_PLAN_MISMATCH = 4
PKV_DEVERR_BAD_OFFSET = 8
PKV_DEVERR_BUCKET = 16
PKV_MAX_GEN_TOKENS = 64

# the C ABI's exported symbols (include/paged_kv.h)
EXPORTS = (
    "paged_rope_table_bytes",
    "paged_rope_table_build",
    "paged_kv_append_rope",
    "paged_kv_append_rope_ex",
    "paged_attention_workspace_size",
    "paged_attention_forward",
    "paged_attention_forward_noalloc",
    "paged_attention_bucket_workspace_size",
    "paged_kv_append_rope_bucket",
    "paged_attention_forward_bucket",
    "paged_kv_last_launch_count",
    "paged_kv_last_launch_name",
    "paged_kv_set_kernel_events",
    "paged_kv_status_string",
)


class PkvPool(C.Structure):
    _fields_ = [("pool", C.c_void_p), ("dtype", C.c_int32), ("num_blocks", C.c_int32),
                ("tokens_per_block", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("kv_scale_quant_orig", C.c_float),
                ("kv_scale_orig_quant", C.c_float)]


class PkvBatch(C.Structure):
    _fields_ = [("num_requests", C.c_int32), ("num_contexts", C.c_int32),
                ("num_tokens", C.c_int32), ("max_blocks_per_seq", C.c_int32),
                ("h_request_types", C.c_void_p), ("h_context_lengths", C.c_void_p),
                ("h_past_kv_lengths", C.c_void_p), ("d_context_lengths", C.c_void_p),
                ("d_past_kv_lengths", C.c_void_p), ("d_block_offsets", C.c_void_p),
                ("d_position_offsets", C.c_void_p), ("d_packed_mask", C.c_void_p),
                ("mask_words", C.c_int32)]


class PkvBucket(C.Structure):
    _fields_ = [("max_context_tokens", C.c_int32), ("max_kv_len", C.c_int32), ("max_gen_tokens", C.c_int32)]


class PagedKVError(RuntimeError):
    pass


_lib = None


def lib() -> C.CDLL:
    """Load libpaged_kv.so (built in-tree by ``paged_kv_cache_rope_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise PagedKVError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_rope_gb300.build` (CUDA 13, sm_103a)")
        L = C.CDLL(LIB_PATH)
        P, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        L.paged_rope_table_bytes.argtypes = [i32, i32]
        L.paged_rope_table_bytes.restype = sz
        L.paged_rope_table_build.argtypes = [C.c_double, i32, i32, P]
        L.paged_rope_table_build.restype = C.c_int
        L.paged_kv_append_rope.argtypes = [P, P, i32, P, i64, P, i64, P, i64, P, i64, P, i32, P, P]
        L.paged_kv_append_rope.restype = C.c_int
        L.paged_kv_append_rope_ex.argtypes = [P, P, i32, P, i64, P, i64, P, i64, P, i64, P, i32, P, P, P]
        L.paged_kv_append_rope_ex.restype = C.c_int
        L.paged_attention_workspace_size.argtypes = [P, P, i32]
        L.paged_attention_workspace_size.restype = sz
        L.paged_attention_forward.argtypes = [P, P, i32, P, i64, P, C.c_float, P, sz, P, P]
        L.paged_attention_forward.restype = C.c_int
        L.paged_attention_forward_noalloc.argtypes = [P, P, i32, P, i64, P, C.c_float, P, P]
        L.paged_attention_forward_noalloc.restype = C.c_int
        L.paged_attention_bucket_workspace_size.argtypes = [P, P, P, i32]
        L.paged_attention_bucket_workspace_size.restype = sz
        L.paged_kv_append_rope_bucket.argtypes = [P, P, P, i32, P, i64, P, i64, P, i64, P, i64, P, i32, P, P, P]
        L.paged_kv_append_rope_bucket.restype = C.c_int
        L.paged_attention_forward_bucket.argtypes = [P, P, P, i32, P, i64, P, C.c_float, P, sz, P, P]
        L.paged_attention_forward_bucket.restype = C.c_int
        L.paged_kv_last_launch_count.argtypes = []
        L.paged_kv_last_launch_count.restype = i32
        L.paged_kv_last_launch_name.argtypes = [i32]
        L.paged_kv_last_launch_name.restype = C.c_char_p
        L.paged_kv_set_kernel_events.argtypes = [P, i32]
        L.paged_kv_set_kernel_events.restype = C.c_int
        L.paged_kv_status_string.argtypes = [C.c_int]
        L.paged_kv_status_string.restype = C.c_char_p
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().paged_kv_status_string(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != PKV_OK:
        raise PagedKVError(f"{what}: {status_string(code)} ({code})")


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


@dataclasses.dataclass
class KVPool:
    """One layer's paged KV pool [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]:
    bf16; uint8 / float8_e4m3fn holding E4M3 codes; or int8 codes -- the 8-bit kinds with one
    per-pool scale."""
    data: torch.Tensor
    kv_scale_quant_orig: float = 1.0
    kv_scale_orig_quant: float = 1.0

    def __post_init__(self):
        assert self.data.dim() == 5 and self.data.shape[1] == 2, "pool must be [NB, 2, B, Hkv, D]"
        assert self.data.is_contiguous()
        assert self.data.dtype in (torch.bfloat16, torch.uint8, torch.float8_e4m3fn, torch.int8)

    @property
    def dtype(self) -> int:
        if self.data.dtype == torch.bfloat16:
            return PKV_BF16
        return PKV_INT8 if self.data.dtype == torch.int8 else PKV_FP8_E4M3

    @property
    def fp8(self) -> bool:
        return self.dtype == PKV_FP8_E4M3

    def c(self) -> PkvPool:
        NB, _, B, Hkv, D = self.data.shape
        return PkvPool(self.data.data_ptr(), self.dtype, NB, B, Hkv, D,
                       float(self.kv_scale_quant_orig), float(self.kv_scale_orig_quant))


class BatchMeta:
    """Host and device copies of one inflight batch's metadata (context requests first)."""

    def __init__(self, request_types, context_lengths, past_kv_lengths, block_offsets, device,
                 position_offsets=None, packed_mask=None):
        """``position_offsets`` (int32 [generation rows]) and ``packed_mask`` (uint32
        [generation rows, words]) describe draft tokens of generation requests that bring
        several new tokens; both optional."""
        self.h_request_types = np.ascontiguousarray(request_types, dtype=np.int32)
        self.h_context_lengths = np.ascontiguousarray(context_lengths, dtype=np.int32)
        self.h_past_kv_lengths = np.ascontiguousarray(past_kv_lengths, dtype=np.int32)
        tbl = np.ascontiguousarray(block_offsets, dtype=np.int32)
        if tbl.ndim == 1:
            tbl = tbl.reshape(len(self.h_context_lengths), -1)
        self.h_block_offsets = tbl
        self.d_context_lengths = torch.from_numpy(self.h_context_lengths.copy()).to(device)
        self.d_past_kv_lengths = torch.from_numpy(self.h_past_kv_lengths.copy()).to(device)
        self.d_block_offsets = torch.from_numpy(tbl.copy()).to(device)
        self.d_position_offsets = self.d_packed_mask = None
        self.mask_words = 0
        if position_offsets is not None:
            off = np.ascontiguousarray(position_offsets, dtype=np.int32).reshape(-1)
            self.d_position_offsets = torch.from_numpy(off.copy()).to(device)
        if packed_mask is not None:
            m = np.ascontiguousarray(packed_mask, dtype=np.uint32)
            self.mask_words = int(m.shape[1])
            self.d_packed_mask = torch.from_numpy(m.view(np.int32).copy()).to(device)

    @property
    def num_requests(self) -> int:
        return int(self.h_context_lengths.shape[0])

    @property
    def num_contexts(self) -> int:
        return int((self.h_request_types == PKV_REQ_CONTEXT).sum())

    @property
    def num_tokens(self) -> int:
        return int(self.h_context_lengths.sum())

    def c(self) -> PkvBatch:
        R = self.num_requests
        return PkvBatch(R, self.num_contexts, self.num_tokens, int(self.h_block_offsets.shape[1]),
                        self.h_request_types.ctypes.data, self.h_context_lengths.ctypes.data,
                        self.h_past_kv_lengths.ctypes.data, self.d_context_lengths.data_ptr(),
                        self.d_past_kv_lengths.data_ptr(), self.d_block_offsets.data_ptr(),
                        None if self.d_position_offsets is None else self.d_position_offsets.data_ptr(),
                        None if self.d_packed_mask is None else self.d_packed_mask.data_ptr(),
                        self.mask_words)


# --- entry points --------------------------------------------------------------------------

def paged_rope_table_build(base: float, head_dim: int, max_pos: int, device="cuda") -> torch.Tensor:
    """GPT-NeoX (cos, sin) table [max_pos, head_dim // 2, 2] fp32, built on the host by the
    library and uploaded once."""
    host = np.empty((max_pos, head_dim // 2, 2), dtype=np.float32)
    _check(lib().paged_rope_table_build(float(base), int(head_dim), int(max_pos), host.ctypes.data),
           "paged_rope_table_build")
    return torch.from_numpy(host).to(device)


def paged_kv_append_rope(pool: KVPool, batch: BatchMeta, num_q_heads: int, q: torch.Tensor,
                         k: torch.Tensor, v: torch.Tensor, q_out: torch.Tensor,
                         rope_table: torch.Tensor, d_error: torch.Tensor, stream=None) -> None:
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out)):
        assert t.dtype == torch.bfloat16 and t.dim() == 2 and t.stride(1) == 1, name
    assert rope_table.dtype == torch.float32 and rope_table.is_contiguous()
    pc, bc = pool.c(), batch.c()
    code = lib().paged_kv_append_rope(
        C.byref(pc), C.byref(bc), int(num_q_heads), _ptr(q), q.stride(0), _ptr(k), k.stride(0),
        _ptr(v), v.stride(0), _ptr(q_out), q_out.stride(0), _ptr(rope_table),
        int(rope_table.shape[0]), _ptr(d_error), _stream_ptr(stream))
    _check(code, "paged_kv_append_rope")


PKV_ROPE_NEOX = 0
PKV_ROPE_GPTJ = 1


class PkvAppendOpts(C.Structure):
    _fields_ = [("rope_style", C.c_int32), ("rotary_dim", C.c_int32), ("q_norm_weight", C.c_void_p),
                ("k_norm_weight", C.c_void_p), ("norm_eps", C.c_float)]


def paged_kv_append_rope_ex(pool: KVPool, batch: BatchMeta, num_q_heads: int, q: torch.Tensor,
                            k: torch.Tensor, v: torch.Tensor, q_out: torch.Tensor,
                            rope_table: torch.Tensor, d_error: torch.Tensor, *, rope_style: int = 0,
                            rotary_dim: int = 0, q_norm_weight: torch.Tensor | None = None,
                            k_norm_weight: torch.Tensor | None = None, norm_eps: float = 1e-6,
                            stream=None) -> None:
    """Append with RoPE variants (rotate-half / interleaved, partial rotary) and optional
    RMSNorm of q / k heads; ``rope_table`` must have rotary_dim / 2 pairs per position."""
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out)):
        assert t.dtype == torch.bfloat16 and t.dim() == 2 and t.stride(1) == 1, name
    for w in (q_norm_weight, k_norm_weight):
        assert w is None or (w.dtype == torch.float32 and w.is_contiguous())
    opts = PkvAppendOpts(int(rope_style), int(rotary_dim), _ptr(q_norm_weight), _ptr(k_norm_weight),
                         float(norm_eps))
    pc, bc = pool.c(), batch.c()
    code = lib().paged_kv_append_rope_ex(
        C.byref(pc), C.byref(bc), int(num_q_heads), _ptr(q), q.stride(0), _ptr(k), k.stride(0),
        _ptr(v), v.stride(0), _ptr(q_out), q_out.stride(0), _ptr(rope_table),
        int(rope_table.shape[0]), C.byref(opts), _ptr(d_error), _stream_ptr(stream))
    _check(code, "paged_kv_append_rope_ex")


def paged_attention_workspace_size(pool: KVPool, batch: BatchMeta, num_q_heads: int) -> int:
    pc, bc = pool.c(), batch.c()
    return int(lib().paged_attention_workspace_size(C.byref(pc), C.byref(bc), int(num_q_heads)))


def paged_attention_forward(pool: KVPool, batch: BatchMeta, num_q_heads: int, q_rot: torch.Tensor,
                            out: torch.Tensor, softmax_scale: float, workspace: torch.Tensor,
                            d_error: torch.Tensor, stream=None) -> None:
    assert q_rot.dtype == torch.bfloat16 and q_rot.stride(1) == 1
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    pc, bc = pool.c(), batch.c()
    code = lib().paged_attention_forward(
        C.byref(pc), C.byref(bc), int(num_q_heads), _ptr(q_rot), q_rot.stride(0), _ptr(out),
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(d_error), _stream_ptr(stream))
    _check(code, "paged_attention_forward")


NOALLOC_SCRATCH_BYTES = 64 << 20


def paged_attention_forward_noalloc(pool: KVPool, batch: BatchMeta, num_q_heads: int,
                                    q_rot: torch.Tensor, out: torch.Tensor, softmax_scale: float,
                                    d_error: torch.Tensor, stream=None) -> None:
    """paged_attention_forward on the library's own static scratch buffer, for callers that
    cannot allocate a workspace (see include/paged_kv.h).  Batches needing more than
    NOALLOC_SCRATCH_BYTES of scratch raise; concurrent calls on different streams race."""
    assert q_rot.dtype == torch.bfloat16 and q_rot.stride(1) == 1
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    pc, bc = pool.c(), batch.c()
    code = lib().paged_attention_forward_noalloc(
        C.byref(pc), C.byref(bc), int(num_q_heads), _ptr(q_rot), q_rot.stride(0), _ptr(out),
        float(softmax_scale), _ptr(d_error), _stream_ptr(stream))
    _check(code, "paged_attention_forward_noalloc")


def last_launch_count() -> int:
    return int(lib().paged_kv_last_launch_count())


def last_launch_names() -> list[str]:
    out = []
    for i in range(last_launch_count()):
        n = lib().paged_kv_last_launch_name(i)
        out.append(n.decode() if n else "?")
    return out


class KernelEvents:
    """Caller-owned cudaEvent_t handles the library records around each of its kernels
    (``paged_kv_set_kernel_events``); used by the benchmark to time kernels on their stream."""

    def __init__(self, max_kernels: int):
        self.max_kernels = max_kernels
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_kernels)]
        for e in self.events:  # force creation of the underlying CUDA events
            e.record()
        self._arr = (C.c_void_p * (2 * max_kernels))(*[int(e.cuda_event) for e in self.events])

    def __enter__(self):
        _check(lib().paged_kv_set_kernel_events(self._arr, self.max_kernels), "paged_kv_set_kernel_events")
        return self

    def __exit__(self, *exc):
        lib().paged_kv_set_kernel_events(None, 0)

    def elapsed_ms(self, i: int) -> float:
        return self.events[2 * i].elapsed_time(self.events[2 * i + 1])


class PagedAttentionStep:
    """One layer step (append + attention) over a resident pool, with every buffer allocated
    once up front so repeated calls allocate nothing."""

    def __init__(self, pool: KVPool, batch: BatchMeta, num_q_heads: int, head_dim: int,
                 rope_table: torch.Tensor, softmax_scale: float | None = None):
        dev = pool.data.device
        self.pool, self.batch, self.Hq, self.D = pool, batch, int(num_q_heads), int(head_dim)
        self.rope_table = rope_table
        self.softmax_scale = softmax_scale if softmax_scale is not None else head_dim ** -0.5
        T = batch.num_tokens
        self.q_out = torch.empty(T, self.Hq * self.D, dtype=torch.bfloat16, device=dev)
        self.out = torch.empty(T, self.Hq * self.D, dtype=torch.bfloat16, device=dev)
        ws = paged_attention_workspace_size(pool, batch, num_q_heads)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.d_error = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches = 0

    def __call__(self, q, k, v, stream=None) -> torch.Tensor:
        paged_kv_append_rope(self.pool, self.batch, self.Hq, q, k, v, self.q_out,
                             self.rope_table, self.d_error, stream)
        n = last_launch_count()
        paged_attention_forward(self.pool, self.batch, self.Hq, self.q_out, self.out,
                                self.softmax_scale, self.workspace, self.d_error, stream)
        self.launches = n + last_launch_count()
        return self.out


# --- padding buckets (one CUDA-graph capture per bucket) -------------------------------------

@dataclasses.dataclass(frozen=True)
class Bucket:
    """A padding bucket: the largest batch one captured step serves.  ``context_slots`` request
    slots take context requests and ``generation_slots`` slots generation requests (a slot with
    no new tokens is empty); at most ``max_tokens`` packed rows, ``max_context_tokens`` of them in
    context slots; past + new <= ``max_kv_len`` for every request; at most ``max_gen_tokens`` new
    tokens per generation request; block tables of ``max_blocks_per_seq`` entries."""
    context_slots: int
    generation_slots: int
    max_tokens: int
    max_context_tokens: int
    max_kv_len: int
    max_gen_tokens: int
    max_blocks_per_seq: int

    @property
    def slots(self) -> int:
        return self.context_slots + self.generation_slots

    def c(self) -> PkvBucket:
        return PkvBucket(self.max_context_tokens, self.max_kv_len, self.max_gen_tokens)


class BucketMeta:
    """Device arrays of one bucket's batch (fixed addresses; rewritten in place per step)."""

    def __init__(self, bucket: Bucket, device, draft: bool = False):
        R, mb = bucket.slots, bucket.max_blocks_per_seq
        gen_rows = min(bucket.max_tokens, bucket.generation_slots * bucket.max_gen_tokens)
        self.bucket = bucket
        self.d_context_lengths = torch.zeros(R, dtype=torch.int32, device=device)
        self.d_past_kv_lengths = torch.zeros(R, dtype=torch.int32, device=device)
        self.d_block_offsets = torch.full((R, mb), -1, dtype=torch.int32, device=device)
        self.mask_words = max(1, -(-bucket.max_gen_tokens // 32)) if draft else 0
        self.d_position_offsets = torch.zeros(max(gen_rows, 1), dtype=torch.int32, device=device) if draft else None
        self.d_packed_mask = (torch.zeros(max(gen_rows, 1), self.mask_words, dtype=torch.int32, device=device)
                              if draft else None)

    def c(self) -> PkvBatch:
        b = self.bucket
        return PkvBatch(b.slots, b.context_slots, b.max_tokens, b.max_blocks_per_seq, None, None, None,
                        self.d_context_lengths.data_ptr(), self.d_past_kv_lengths.data_ptr(),
                        self.d_block_offsets.data_ptr(),
                        None if self.d_position_offsets is None else self.d_position_offsets.data_ptr(),
                        None if self.d_packed_mask is None else self.d_packed_mask.data_ptr(), self.mask_words)


def paged_attention_bucket_workspace_size(pool: KVPool, meta: BucketMeta, num_q_heads: int) -> int:
    pc, bc, kc = pool.c(), meta.c(), meta.bucket.c()
    return int(lib().paged_attention_bucket_workspace_size(C.byref(pc), C.byref(bc), C.byref(kc), int(num_q_heads)))


def paged_kv_append_rope_bucket(pool: KVPool, meta: BucketMeta, num_q_heads: int, q: torch.Tensor,
                                k: torch.Tensor, v: torch.Tensor, q_out: torch.Tensor, rope_table: torch.Tensor,
                                d_error: torch.Tensor, stream=None) -> None:
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out)):
        assert t.dtype == torch.bfloat16 and t.dim() == 2 and t.stride(1) == 1, name
        assert t.shape[0] >= meta.bucket.max_tokens, name
    assert rope_table.dtype == torch.float32 and rope_table.is_contiguous()
    pc, bc, kc = pool.c(), meta.c(), meta.bucket.c()
    code = lib().paged_kv_append_rope_bucket(
        C.byref(pc), C.byref(bc), C.byref(kc), int(num_q_heads), _ptr(q), q.stride(0), _ptr(k), k.stride(0),
        _ptr(v), v.stride(0), _ptr(q_out), q_out.stride(0), _ptr(rope_table), int(rope_table.shape[0]), None,
        _ptr(d_error), _stream_ptr(stream))
    _check(code, "paged_kv_append_rope_bucket")


def paged_attention_forward_bucket(pool: KVPool, meta: BucketMeta, num_q_heads: int, q_rot: torch.Tensor,
                                   out: torch.Tensor, softmax_scale: float, workspace: torch.Tensor,
                                   d_error: torch.Tensor, stream=None) -> None:
    assert q_rot.dtype == torch.bfloat16 and q_rot.stride(1) == 1
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    pc, bc, kc = pool.c(), meta.c(), meta.bucket.c()
    code = lib().paged_attention_forward_bucket(
        C.byref(pc), C.byref(bc), C.byref(kc), int(num_q_heads), _ptr(q_rot), q_rot.stride(0), _ptr(out),
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(d_error),
        _stream_ptr(stream))
    _check(code, "paged_attention_forward_bucket")


class PagedAttentionBucketStep:
    """One layer step (append + attention) over a padding bucket, with every buffer -- metadata
    included -- allocated once, so that the step can be captured into a CUDA graph once and
    replayed for every batch of the bucket.

    ``load(...)`` writes a batch into the fixed buffers (lengths, block table, draft-token arrays
    and the q / k / v rows; outside any capture), ``__call__`` enqueues the step, ``capture()``
    records it into a graph and ``replay()`` runs that graph.  Rows ``[0, num_tokens)`` of
    ``out`` hold the loaded batch's result."""

    def __init__(self, pool: KVPool, bucket: Bucket, num_q_heads: int, head_dim: int, rope_table: torch.Tensor,
                 softmax_scale: float | None = None, draft: bool = False):
        dev = pool.data.device
        self.pool, self.bucket, self.Hq, self.D = pool, bucket, int(num_q_heads), int(head_dim)
        self.Hkv = int(pool.data.shape[3])
        self.rope_table = rope_table
        self.softmax_scale = softmax_scale if softmax_scale is not None else head_dim ** -0.5
        self.meta = BucketMeta(bucket, dev, draft)
        T = bucket.max_tokens
        self.q = torch.zeros(T, self.Hq * self.D, dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros(T, self.Hkv * self.D, dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros(T, self.Hkv * self.D, dtype=torch.bfloat16, device=dev)
        self.q_out = torch.zeros(T, self.Hq * self.D, dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros(T, self.Hq * self.D, dtype=torch.bfloat16, device=dev)
        ws = paged_attention_bucket_workspace_size(pool, self.meta, num_q_heads)
        if ws == 0:
            raise PagedKVError("paged_attention_bucket_workspace_size: invalid bucket")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.d_error = torch.zeros(1, dtype=torch.int32, device=dev)
        self.num_tokens = 0
        self.graph = None

    def load(self, request_types, context_lengths, past_kv_lengths, block_offsets, q, k, v,
             position_offsets=None, packed_mask=None, stream=None) -> None:
        """Writes one batch (context requests first, as always) into the bucket's slots: its
        context requests into the first context slots, its generation requests into the first
        generation slots, every other slot empty.  Checks on the host that it fits."""
        bk = self.bucket
        types = np.asarray(request_types, dtype=np.int32)
        n = np.asarray(context_lengths, dtype=np.int32)
        past = np.asarray(past_kv_lengths, dtype=np.int32)
        tbl = np.asarray(block_offsets, dtype=np.int32).reshape(len(n), -1)
        nc = int((types == PKV_REQ_CONTEXT).sum())
        ng = len(n) - nc
        if not (types[:nc] == PKV_REQ_CONTEXT).all():
            raise PagedKVError("context requests must come first")
        if nc > bk.context_slots or ng > bk.generation_slots:
            raise PagedKVError("more requests than the bucket's slots")
        T = int(n.sum())
        if T > bk.max_tokens or int(n[:nc].sum()) > bk.max_context_tokens:
            raise PagedKVError("more rows than the bucket holds")
        if len(n) and (int((past + n).max()) > bk.max_kv_len or (ng and int(n[nc:].max()) > bk.max_gen_tokens)):
            raise PagedKVError("a request exceeds the bucket's limits")
        if tbl.shape[1] > bk.max_blocks_per_seq:
            raise PagedKVError("block table wider than the bucket's")
        R = bk.slots
        sl_n = np.zeros(R, np.int32)
        sl_p = np.zeros(R, np.int32)
        sl_t = np.full((R, bk.max_blocks_per_seq), -1, np.int32)
        slots = list(range(nc)) + list(range(bk.context_slots, bk.context_slots + ng))
        sl_n[slots], sl_p[slots] = n, past
        sl_t[slots, :tbl.shape[1]] = tbl
        on_gpu = self.q.device.type == "cuda"
        s = stream if stream is not None else (torch.cuda.current_stream() if on_gpu else None)
        with torch.cuda.stream(s) if on_gpu else contextlib.nullcontext():
            self.meta.d_context_lengths.copy_(torch.from_numpy(sl_n), non_blocking=False)
            self.meta.d_past_kv_lengths.copy_(torch.from_numpy(sl_p), non_blocking=False)
            self.meta.d_block_offsets.copy_(torch.from_numpy(sl_t), non_blocking=False)
            if self.meta.d_position_offsets is not None:
                self.meta.d_position_offsets.zero_()
                self.meta.d_packed_mask.zero_()
                if position_offsets is not None:
                    off = torch.from_numpy(np.ascontiguousarray(position_offsets, dtype=np.int32))
                    self.meta.d_position_offsets[:off.numel()].copy_(off)
                if packed_mask is not None:
                    m = np.ascontiguousarray(packed_mask, dtype=np.uint32)
                    mt = torch.from_numpy(m.view(np.int32))
                    self.meta.d_packed_mask[:mt.shape[0], :mt.shape[1]].copy_(mt)
            for dst, src in ((self.q, q), (self.k, k), (self.v, v)):
                dst[:T].copy_(src[:T])
        self.num_tokens = T

    def __call__(self, stream=None) -> torch.Tensor:
        paged_kv_append_rope_bucket(self.pool, self.meta, self.Hq, self.q, self.k, self.v, self.q_out,
                                    self.rope_table, self.d_error, stream)
        paged_attention_forward_bucket(self.pool, self.meta, self.Hq, self.q_out, self.out, self.softmax_scale,
                                       self.workspace, self.d_error, stream)
        return self.out

    def capture(self) -> None:
        """Records the step into a CUDA graph (after one uncaptured warm-up call)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self()
        self.graph = g

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out
