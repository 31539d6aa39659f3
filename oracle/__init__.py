"""fp64 CPU oracle for the paged-KV RoPE + attention hot path (ctypes front end).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg are the only callers.  Nothing in ``paged_kv_cache_rope_gb300`` imports this package, and
this package imports nothing from it: the two sides share only the seeded input generators.

Functions (all on host numpy arrays):
  bf16_from_f32 / f32_from_bf16     IEEE round-to-nearest-even bf16
  e4m3_encode / e4m3_decode         OCP FP8 E4M3, RNE with saturation to +-448
  int8_encode                       INT8 codes: nearest integer, ties to even, saturating
  rope_table                        fp32 (cos, sin) table computed in fp64
  rope32 / rope64                   GPT-NeoX rotate-half rotation (fp32 recipe / exact fp64)
  append_rope                       O1 write image: q_out rows and pool bytes after the append
  append_rope_ex                    O1 with RoPE variants, QK-norm and draft-token position offsets
  attention                         O2 fp64 causal GQA attention read through the block table
                                    (optionally with packed masks for draft-token requests)
Each C function cites its page and section in oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        # a mutated build of oracle.c can be swapped in by the planted-mistake tests
        path = os.environ.get("PKV_ORACLE_LIB") or _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, f32, f64 = C.c_int32, C.c_int64, C.c_float, C.c_double
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_bf16_to_f32.restype = f32
        L.orc_f32_to_bf16.argtypes = [f32]
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_e4m3_to_f64.argtypes = [C.c_uint8]
        L.orc_e4m3_to_f64.restype = f64
        L.orc_f32_to_e4m3.argtypes = [f32]
        L.orc_f32_to_e4m3.restype = C.c_uint8
        L.orc_rope_table.argtypes = [f64, i32, i32, P]
        L.orc_rope_table.restype = None
        L.orc_rope32.argtypes = [P, i32, P, P]
        L.orc_rope32.restype = None
        L.orc_rope64.argtypes = [P, i32, f64, i64, P]
        L.orc_rope64.restype = None
        L.orc_append_rope.argtypes = [i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                      P, i64, P, i64, P, i64, P, i32, P, i64, P]
        L.orc_append_rope.restype = C.c_int
        L.orc_append_rope_ex.argtypes = [i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                         P, i64, P, i64, P, i64, P, i32, i32, i32, P, P, f64,
                                         P, i64, P]
        L.orc_append_rope_ex.restype = C.c_int
        L.orc_attention.argtypes = [i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, f64, P,
                                    P, f64, P, i64, P]
        L.orc_attention.restype = C.c_int
        L.orc_append_rope_spec.argtypes = [i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                           P, i64, P, i64, P, i64, P, i32, i32, i32, P, P, f64,
                                           P, P, i64, P]
        L.orc_append_rope_spec.restype = C.c_int
        L.orc_attention_spec.argtypes = [i32, P, P, P, i32, i32, i32, i32, i32, i32, i32, f64, P,
                                         P, f64, P, i64, i32, P, i32, P]
        L.orc_attention_spec.restype = C.c_int
        L.orc_f32_to_bf16_array.argtypes = [P, i64, P]
        L.orc_f32_to_bf16_array.restype = None
        L.orc_f32_to_e4m3_array.argtypes = [P, i64, P]
        L.orc_f32_to_e4m3_array.restype = None
        L.orc_f32_to_int8_array.argtypes = [P, i64, P]
        L.orc_f32_to_int8_array.restype = None
        L.orc_e4m3_to_f64_array.argtypes = [P, i64, P]
        L.orc_e4m3_to_f64_array.restype = None
        L.orc_num_threads.argtypes = []
        L.orc_num_threads.restype = C.c_int
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return int(lib().orc_num_threads())


# --- scalar formats --------------------------------------------------------------------------

def bf16_from_f32(x) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), round to nearest even."""
    shape = np.shape(x)
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(x), int(x.size), _ptr(out))
    return out.reshape(shape)


def f32_from_bf16(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def e4m3_decode(codes) -> np.ndarray:
    shape = np.shape(codes)
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8)).reshape(-1)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_to_f64_array(_ptr(c), int(c.size), _ptr(out))
    return out.reshape(shape)


def e4m3_encode(x) -> np.ndarray:
    shape = np.shape(x)
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_f32_to_e4m3_array(_ptr(x), int(x.size), _ptr(out))
    return out.reshape(shape)


def int8_encode(x) -> np.ndarray:
    """fp32 values -> int8 codes: nearest integer, ties to even, saturated to [-128, 127]."""
    shape = np.shape(x)
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    out = np.empty(x.shape, dtype=np.int8)
    lib().orc_f32_to_int8_array(_ptr(x), int(x.size), _ptr(out))
    return out.reshape(shape)


def _kind(kv_fp8, kv_int8) -> int:
    """Pool element type for the C side: 0 bf16, 1 FP8 E4M3, 2 INT8."""
    return 2 if kv_int8 else int(bool(kv_fp8))


# --- RoPE -------------------------------------------------------------------------------------

def rope_table(base: float, head_dim: int, max_pos: int) -> np.ndarray:
    """[max_pos, head_dim // 2, 2] float32 (cos, sin) table."""
    cs = np.empty((max_pos, head_dim // 2, 2), dtype=np.float32)
    lib().orc_rope_table(float(base), int(head_dim), int(max_pos), _ptr(cs))
    return cs


def rope32(x: np.ndarray, cs_row: np.ndarray) -> np.ndarray:
    """fp32 rotation of one head vector by one table row (fp32 result, not rounded)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    cs_row = np.ascontiguousarray(cs_row, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_rope32(_ptr(x), int(x.shape[0]), _ptr(cs_row), _ptr(y))
    return y


def rope64(x: np.ndarray, base: float, pos: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().orc_rope64(_ptr(x), int(x.shape[0]), float(base), int(pos), _ptr(y))
    return y


# --- the two hot-path operations --------------------------------------------------------------

def append_rope(*, new_len, past, block_table, num_q_heads, num_kv_heads, head_dim,
                tokens_per_block, num_blocks, kv_fp8, inv_scale, q_bits, k_bits, v_bits, cs,
                pool, q_out=None, kv_int8=False):
    """O1 write image.  Updates ``pool`` (uint16 bf16 bits or uint8 e4m3 codes, any shape,
    C-contiguous) in place and returns (status, q_out bits [T, Hq*D])."""
    new_len = np.ascontiguousarray(new_len, dtype=np.int32)
    past = np.ascontiguousarray(past, dtype=np.int32)
    tbl = np.ascontiguousarray(block_table, dtype=np.int32)
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    cs = np.ascontiguousarray(cs, dtype=np.float32)
    T = int(new_len.sum())
    if q_out is None:
        q_out = np.zeros((T, num_q_heads * head_dim), dtype=np.uint16)
    assert pool.flags["C_CONTIGUOUS"]
    st = lib().orc_append_rope(
        int(new_len.shape[0]), _ptr(new_len), _ptr(past), _ptr(tbl), int(tbl.shape[1]),
        int(num_q_heads), int(num_kv_heads), int(head_dim), int(tokens_per_block),
        int(num_blocks), _kind(kv_fp8, kv_int8), float(inv_scale),
        _ptr(q_bits), int(q_bits.shape[1]) if T else 0, _ptr(k_bits), int(k_bits.shape[1]) if T else 0,
        _ptr(v_bits), int(v_bits.shape[1]) if T else 0, _ptr(cs), int(cs.shape[0]),
        _ptr(q_out), int(q_out.shape[1]), _ptr(pool))
    return int(st), q_out


def append_rope_ex(*, new_len, past, block_table, num_q_heads, num_kv_heads, head_dim,
                   tokens_per_block, num_blocks, kv_fp8, inv_scale, q_bits, k_bits, v_bits, cs,
                   pool, style=0, rotary_dim=0, q_norm_w=None, k_norm_w=None, norm_eps=1e-6,
                   pos_offset=None, q_out=None, kv_int8=False):
    """O1 with the variants: style 0 rotate-half / 1 interleaved, rotary_dim (0 = head_dim),
    optional RMSNorm weights for q and k heads.  ``cs`` has rotary_dim / 2 pairs per row.
    ``pos_offset`` (int32 [T], one per packed row) rotates row (r, i) for position
    past_r + pos_offset[row] instead of past_r + i; the slot stays past_r + i."""
    new_len = np.ascontiguousarray(new_len, dtype=np.int32)
    past = np.ascontiguousarray(past, dtype=np.int32)
    tbl = np.ascontiguousarray(block_table, dtype=np.int32)
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    cs = np.ascontiguousarray(cs, dtype=np.float32)
    T = int(new_len.sum())
    if q_out is None:
        q_out = np.zeros((T, num_q_heads * head_dim), dtype=np.uint16)
    qw = None if q_norm_w is None else np.ascontiguousarray(q_norm_w, dtype=np.float32)
    kw = None if k_norm_w is None else np.ascontiguousarray(k_norm_w, dtype=np.float32)
    common = (int(new_len.shape[0]), _ptr(new_len), _ptr(past), _ptr(tbl), int(tbl.shape[1]),
              int(num_q_heads), int(num_kv_heads), int(head_dim), int(tokens_per_block),
              int(num_blocks), _kind(kv_fp8, kv_int8), float(inv_scale),
              _ptr(q_bits), int(q_bits.shape[1]) if T else 0, _ptr(k_bits), int(k_bits.shape[1]) if T else 0,
              _ptr(v_bits), int(v_bits.shape[1]) if T else 0, _ptr(cs), int(cs.shape[0]), int(style),
              int(rotary_dim), None if qw is None else _ptr(qw), None if kw is None else _ptr(kw),
              float(norm_eps))
    if pos_offset is None:
        st = lib().orc_append_rope_ex(*common, _ptr(q_out), int(q_out.shape[1]), _ptr(pool))
    else:
        off = np.ascontiguousarray(pos_offset, dtype=np.int32)
        assert off.shape == (T,)
        st = lib().orc_append_rope_spec(*common, _ptr(off), _ptr(q_out), int(q_out.shape[1]), _ptr(pool))
    return int(st), q_out


def attention(*, new_len, past, block_table, num_q_heads, num_kv_heads, head_dim,
              tokens_per_block, num_blocks, kv_fp8, kv_scale, pool, q, softmax_scale,
              rows=None, num_contexts=None, gen_mask=None, kv_int8=False):
    """O2 fp64 attention.  ``q`` is float64 [T, Hq, D] (or [T, Hq*D]); returns
    (status, out float64 [T, Hq, D]); rows not in ``rows`` (when given) are NaN.
    ``gen_mask`` (uint32 [generation rows, words], with ``num_contexts``) gives each token of a
    generation request the new tokens of its request it may see (bit j of word j // 32; the
    token itself is always seen); without it every request is causal."""
    new_len = np.ascontiguousarray(new_len, dtype=np.int32)
    past = np.ascontiguousarray(past, dtype=np.int32)
    tbl = np.ascontiguousarray(block_table, dtype=np.int32)
    T = int(new_len.sum())
    q = np.ascontiguousarray(q, dtype=np.float64).reshape(T, num_q_heads, head_dim)
    out = np.full((T, num_q_heads, head_dim), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rows_p, n = _ptr(rows), int(rows.shape[0])
    else:
        rows_p, n = None, T
    common = (int(new_len.shape[0]), _ptr(new_len), _ptr(past), _ptr(tbl), int(tbl.shape[1]),
              int(num_q_heads), int(num_kv_heads), int(head_dim), int(tokens_per_block),
              int(num_blocks), _kind(kv_fp8, kv_int8), float(kv_scale), _ptr(pool), _ptr(q),
              float(softmax_scale), rows_p, n)
    if gen_mask is None:
        st = lib().orc_attention(*common, _ptr(out))
    else:
        m = np.ascontiguousarray(gen_mask, dtype=np.uint32)
        C_ = int(num_contexts)
        assert m.ndim == 2 and m.shape[0] == T - int(new_len[:C_].sum())
        st = lib().orc_attention_spec(*common, C_, _ptr(m), int(m.shape[1]), _ptr(out))
    return int(st), out
