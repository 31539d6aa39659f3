"""Seeded synthetic inflight batches shaped like the pages' workloads.

This module only draws inputs: lengths, page placement, Q/K/V values and the cached history
already sitting in the pool.  It holds none of the method's arithmetic (no RoPE, no attention,
no FP8 encoding of its own; the FP8 history codes come from torch's own float8 cast).  Both the
CUDA library and the CPU oracle are fed from here.

Batch structure (page "TensorRT-LLM 源码完全拆解(一)", sections "AttentionMetadata 的字段与它的含义"
and "KVCacheManager 的三个对外接口"; page adg.csdn.net/69730cc6, section 1.3):
  * requests are packed with no padding, context requests first, generation requests after;
  * request r brings ``new_len[r]`` tokens (1 for generation, or several draft tokens to verify)
    on top of ``past[r]`` cached ones;
  * the pool is ``[num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]`` (K at index 0,
    V at index 1) and ``block_table[r, j]`` is the physical page of logical block j.

Recipe: lengths as stated per workload; page placement is a seeded random permutation of all
pool pages (pages never referenced stay unused); q, k, v and the cached K/V history are i.i.d.
N(0, 1) rounded to bf16; the history is treated as already rotated.  Pool slots holding no
cached token are poisoned with NaN (bf16 0x7FC0, e4m3 0x7F; int8, having no NaN, -128) when
``poison`` is set, else zero, and unused block-table entries are -1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
INT8_POISON = -128  # int8 has no NaN: unused slots hold the most negative code
REQ_CONTEXT = 0
REQ_GENERATION = 1


@dataclasses.dataclass
class Batch:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    tokens_per_block: int
    num_blocks: int
    kv_dtype: str                 # "bf16", "fp8" or "int8"
    rope_base: float
    request_types: np.ndarray     # int32 [R]
    new_len: np.ndarray           # int32 [R]
    past: np.ndarray              # int32 [R]
    block_table: np.ndarray       # int32 [R, max_blocks_per_seq]
    q: torch.Tensor               # bf16 [T, Hq*D]
    k: torch.Tensor               # bf16 [T, Hkv*D]
    v: torch.Tensor               # bf16 [T, Hkv*D]
    pool: torch.Tensor            # [NB, 2, B, Hkv, D], bf16, uint8 (e4m3 codes) or int8 codes
    pool_bf16: torch.Tensor | None  # 8-bit batches: the unquantised bf16 twin of ``pool``
    kv_scale: float               # dequantisation multiplier (amax / 448 or amax / 127), 1 for bf16
    inv_scale: float              # fp32(1 / kv_scale), the quantisation multiplier
    # draft-token trees (generation requests of several tokens), else None: per generation
    # row, the RoPE position offset (depth in the tree) and the packed mask row (bit j of word
    # j // 32: the row's token sees new token j of its request -- its ancestors and itself)
    position_offsets: np.ndarray | None = None  # int32 [T_gen]
    packed_mask: np.ndarray | None = None       # uint32 [T_gen, words]

    @property
    def num_requests(self) -> int:
        return int(self.new_len.shape[0])

    @property
    def num_contexts(self) -> int:
        return int((self.request_types == REQ_CONTEXT).sum())

    @property
    def num_tokens(self) -> int:
        return int(self.new_len.sum())

    @property
    def kv_lengths(self) -> np.ndarray:
        return (self.past + self.new_len).astype(np.int64)

    @property
    def num_ctx_tokens(self) -> int:
        return int(self.new_len[:self.num_contexts].sum())

    @property
    def max_pos(self) -> int:
        return int(self.kv_lengths.max()) if self.num_requests else 1

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def to(self, device) -> "Batch":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, q=f(self.q), k=f(self.k), v=f(self.v),
                                   pool=f(self.pool), pool_bf16=f(self.pool_bf16))


def make_batch(*, name: str, ctx: list[tuple[int, int]], gen: list, num_q_heads: int,
               num_kv_heads: int, head_dim: int, tokens_per_block: int, kv_dtype: str = "bf16",
               rope_base: float = 1e4, seed: int = 0, device: str = "cpu", poison: bool = True,
               extra_blocks: float = 0.1, min_spare_blocks: int = 4,
               num_blocks: int | None = None, draft_tree: bool = False) -> Batch:
    """``ctx``: (new tokens, cached tokens) per context request; ``gen``: per generation
    request either its KV length counting this step's one token (so ``past = L - 1``), or a
    pair (draft tokens, cached tokens) for a request verifying several tokens at once.
    ``draft_tree`` draws a seeded random candidate tree per generation request (token 0 the
    root, each later token a child of an earlier one) and fills ``position_offsets`` and
    ``packed_mask``; without it the draft tokens form a chain (plain causal order)."""
    assert kv_dtype in ("bf16", "fp8", "int8")
    B, Hkv, D = tokens_per_block, num_kv_heads, head_dim
    gen = [(1, L - 1) if np.ndim(L) == 0 else (int(L[0]), int(L[1])) for L in gen]
    new_len = np.array([n for n, _ in ctx] + [n for n, _ in gen], dtype=np.int32)
    past = np.array([p for _, p in ctx] + [p for _, p in gen], dtype=np.int32)
    types = np.array([REQ_CONTEXT] * len(ctx) + [REQ_GENERATION] * len(gen), dtype=np.int32)
    R = len(new_len)
    kv_len = past.astype(np.int64) + new_len
    pages = [-(-int(L) // B) for L in kv_len]
    used = int(sum(pages))
    if num_blocks is None:
        num_blocks = int(math.ceil(used * (1.0 + extra_blocks))) + min_spare_blocks
    assert num_blocks >= used
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max(pages) if pages else 1
    table = np.full((R, max_blocks), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        table[r, :pages[r]] = perm[off:off + pages[r]]
        off += pages[r]

    offsets = mask = None
    if draft_tree:
        words = max(1, -(-max([n for n, _ in gen] + [1]) // 32))
        offsets = np.zeros(sum(n for n, _ in gen), dtype=np.int32)
        mask = np.zeros((offsets.shape[0], words), dtype=np.uint32)
        trng = np.random.default_rng(seed + 7919)
        row = 0
        for n, _ in gen:
            parent = [-1] + [int(trng.integers(0, i)) for i in range(1, n)]
            for i in range(n):
                a, depth = i, 0
                while a >= 0:  # the token and its ancestors
                    mask[row + i, a // 32] |= np.uint32(1 << (a % 32))
                    a = parent[a]
                    depth += 1
                offsets[row + i] = depth - 1
            row += n

    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(seed)
    T = int(new_len.sum())
    Hq = num_q_heads

    def randn(*shape):
        return torch.randn(*shape, generator=gen_t, device=device, dtype=torch.float32)

    q = randn(T, Hq * D).to(torch.bfloat16)
    k = randn(T, Hkv * D).to(torch.bfloat16)
    v = randn(T, Hkv * D).to(torch.bfloat16)

    # cached history: positions 0 .. past-1 of every request, K and V, already rotated
    tok_blk, tok_slot = [], []
    for r in range(R):
        t = np.arange(int(past[r]), dtype=np.int64)
        tok_blk.append(table[r, t // B])
        tok_slot.append(t % B)
    tok_blk = torch.from_numpy(np.concatenate(tok_blk) if tok_blk else np.zeros(0, np.int64)).long()
    tok_slot = torch.from_numpy(np.concatenate(tok_slot) if tok_slot else np.zeros(0, np.int64)).long()
    n_hist = int(tok_blk.numel())
    hist = randn(n_hist, 2, Hkv, D).to(torch.bfloat16)
    tok_blk, tok_slot = tok_blk.to(device), tok_slot.to(device)

    bf16_pool = torch.empty(num_blocks, 2, B, Hkv, D, dtype=torch.bfloat16, device=device)
    if poison:
        bf16_pool.view(torch.int16).fill_(BF16_NAN)
    else:
        bf16_pool.zero_()
    bf16_pool[tok_blk, 0, tok_slot] = hist[:, 0]
    bf16_pool[tok_blk, 1, tok_slot] = hist[:, 1]

    if kv_dtype == "bf16":
        return Batch(name, Hq, Hkv, D, B, num_blocks, kv_dtype, rope_base, types, new_len,
                     past, table, q, k, v, bf16_pool, None, 1.0, 1.0, offsets, mask)

    # 8-bit pool: one per-tensor scale, amax over every K/V value drawn (history and new k/v)
    amax = max(float(hist.float().abs().max()) if n_hist else 0.0,
               float(k.float().abs().max()) if T else 0.0,
               float(v.float().abs().max()) if T else 0.0, 1e-30)
    kv_scale = float(np.float32(amax / (127.0 if kv_dtype == "int8" else 448.0)))
    inv_scale = float(np.float32(1.0 / kv_scale))
    if kv_dtype == "int8":  # history codes by torch's round-half-even and a clamp
        codes = (hist.float() * inv_scale).round().clamp(-128.0, 127.0).to(torch.int8)
        i8_pool = torch.empty(num_blocks, 2, B, Hkv, D, dtype=torch.int8, device=device)
        i8_pool.fill_(INT8_POISON if poison else 0)
        i8_pool[tok_blk, 0, tok_slot] = codes[:, 0]
        i8_pool[tok_blk, 1, tok_slot] = codes[:, 1]
        return Batch(name, Hq, Hkv, D, B, num_blocks, kv_dtype, rope_base, types, new_len, past,
                     table, q, k, v, i8_pool, bf16_pool, kv_scale, inv_scale, offsets, mask)
    codes = (hist.float() * inv_scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    fp8_pool = torch.empty(num_blocks, 2, B, Hkv, D, dtype=torch.uint8, device=device)
    fp8_pool.fill_(E4M3_NAN if poison else 0)
    fp8_pool[tok_blk, 0, tok_slot] = codes[:, 0]
    fp8_pool[tok_blk, 1, tok_slot] = codes[:, 1]
    return Batch(name, Hq, Hkv, D, B, num_blocks, kv_dtype, rope_base, types, new_len, past,
                 table, q, k, v, fp8_pool, bf16_pool, kv_scale, inv_scale, offsets, mask)


# --- the five workloads ------------------------------------------------------------------------

def _log_uniform_int(rng, lo, hi, n):
    return np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), n))).astype(np.int64)


WORKLOADS = {
    1: "tiny_mixed",
    2: "decode_llama7b_mha",
    3: "decode_llama70b_gqa",
    4: "inflight_mixed_chunked",
    5: "long_context_16k_prefill",
    6: "spec_decode_tree_gqa",
}


def workload(idx: int, *, kv_dtype: str = "bf16", device: str = "cpu", poison: bool = True,
             seed: int | None = None, max_gen: int | None = None) -> Batch:
    """The synthetic workloads (seed = workload index unless given): 1-5 shaped like the pages'
    configurations, 6 a draft-token verification batch.  ``max_gen`` keeps only the first
    generation requests (smaller captures for profiling)."""
    seed = idx if seed is None else seed
    rng = np.random.default_rng(1000 + idx)  # lengths depend on the workload only, values on seed

    def _mk(**kw):
        if max_gen is not None:
            kw["gen"] = list(kw["gen"])[:max_gen]
        return make_batch(**kw)

    if idx == 1:  # 1 context (37 new, 0 cached) + 1 decode (53 cached + 1 new); 16-page pool
        return _mk(name=WORKLOADS[1], ctx=[(37, 0)], gen=[54], num_q_heads=4,
                          num_kv_heads=2, head_dim=64, tokens_per_block=16, kv_dtype=kv_dtype,
                          rope_base=1e4, seed=seed, device=device, poison=poison, num_blocks=16)
    if idx == 2:  # 64 decodes, MHA 32/32, L ~ U[512, 4096], block 64
        gen = rng.integers(512, 4096, size=64, endpoint=True).tolist()
        return _mk(name=WORKLOADS[2], ctx=[], gen=gen, num_q_heads=32, num_kv_heads=32,
                          head_dim=128, tokens_per_block=64, kv_dtype=kv_dtype, seed=seed,
                          device=device, poison=poison)
    if idx == 3:  # 256 decodes, GQA 64/8, L log-uniform 128..8192, block 32
        gen = np.clip(_log_uniform_int(rng, 128, 8192, 256), 128, 8192).tolist()
        return _mk(name=WORKLOADS[3], ctx=[], gen=gen, num_q_heads=64, num_kv_heads=8,
                          head_dim=128, tokens_per_block=32, kv_dtype=kv_dtype, seed=seed,
                          device=device, poison=poison)
    if idx == 4:  # 4 chunked contexts (1024 new, 0..3072 cached, multiple of 64) + 128 decodes
        ctx = [(1024, int(64 * rng.integers(0, 48, endpoint=True))) for _ in range(4)]
        gen = rng.integers(256, 4096, size=128, endpoint=True).tolist()
        return _mk(name=WORKLOADS[4], ctx=ctx, gen=gen, num_q_heads=32, num_kv_heads=8,
                          head_dim=128, tokens_per_block=64, kv_dtype=kv_dtype, seed=seed,
                          device=device, poison=poison)
    if idx == 5:  # 16384-token prefill + 8 decodes with L ~ U[32768, 131072], RoPE base 5e5
        gen = rng.integers(32768, 131072, size=8, endpoint=True).tolist()
        return _mk(name=WORKLOADS[5], ctx=[(16384, 0)], gen=gen, num_q_heads=32,
                          num_kv_heads=8, head_dim=128, tokens_per_block=64, kv_dtype=kv_dtype,
                          rope_base=5e5, seed=seed, device=device, poison=poison)
    if idx == 6:  # 64 generation requests verifying 8-token draft trees, GQA 64/8, L ~ U[1024, 4096]
        past = rng.integers(1024 - 8, 4096 - 8, size=64, endpoint=True).tolist()
        return _mk(name=WORKLOADS[6], ctx=[], gen=[(8, int(p)) for p in past], num_q_heads=64,
                   num_kv_heads=8, head_dim=128, tokens_per_block=32, kv_dtype=kv_dtype, seed=seed,
                   device=device, poison=poison, draft_tree=True)
    raise ValueError(f"unknown workload {idx}")
