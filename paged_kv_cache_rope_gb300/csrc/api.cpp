// api.cpp -- C-ABI front end of libpaged_kv.so: argument validation, launch planning and
// dispatch.  Everything here runs on the host and only enqueues work on the caller's stream
// (and, for mixed batches, on an auxiliary stream forked from and joined back into it); no
// device memory is allocated and no stream is ever synchronised.
//
// Dispatch follows "TensorRT-LLM 1.0 源码学习笔记" 6.1 "两者分工": context requests (input length
// > 1, and chunked-context requests) go to the flash-attention style tensor-core kernel,
// generation requests (length 1) to the paged split-KV decode kernel.  Batch ordering (context
// requests first) follows adg.csdn.net/69730cc6 section 1.3; the workspace-size query mirrors
// the scratch-workspace check of section 5.1 of the same notes page.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "paged_kv.h"

namespace {

thread_local int32_t g_last_launches = 0;
thread_local const char* g_last_names[8] = {nullptr};
thread_local void* const* g_events = nullptr;
thread_local int32_t g_events_n = 0;

// Brackets one kernel launch of the current call with the caller's timing events (if set) and
// records its name.
struct LaunchScope {
  int idx;
  cudaStream_t s;
  LaunchScope(int i, const char* name, cudaStream_t st) : idx(i), s(st) {
    if (idx < 8) g_last_names[idx] = name;
    if (g_events && idx < g_events_n) cudaEventRecord(static_cast<cudaEvent_t>(g_events[2 * idx]), s);
  }
  ~LaunchScope() {
    if (g_events && idx < g_events_n) cudaEventRecord(static_cast<cudaEvent_t>(g_events[2 * idx + 1]), s);
  }
};

void reset_names() {
  for (auto& n : g_last_names) n = nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (sms[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 152;
  }
  return sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 4-D bf16 map (64-wide head-dim half, head-dim halves, heads, rows) with a 128-byte swizzle;
// box = one 64-wide half of `box_rows` rows of one head.
bool encode_rows_map(CUtensorMap* map, const void* base, int D, int heads, int64_t rows, int64_t row_bytes,
                     int box_rows, int box_heads = 1) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 8-bit pool rows of D one-byte codes: dims (D, heads, rows), box D x 1 head x box_rows, with
// the 128-byte swizzle (D = 128: one row per swizzle span).
bool encode_raw8_map(CUtensorMap* map, const void* base, int D, int heads, int64_t rows, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads) * D};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The launch plan.  Without a bucket every count is exact (from the host copies of the
// lengths); with a bucket (dyn) every count is a capacity for the bucket's largest batch and the
// device plan finds the actual counts.
struct HostPlan {
  int R = 0, C = 0, G = 0, T = 0, ctx_tokens = 0, max_gen_tokens = 0;
  int gen_rows = 0;                                  // rows of the generation requests
  int num_tiles = 0, num_splits = 0, kv_chunk = 0, max_splits = 0;
  int decode_nt = 1, num_items = 0, num_parts = 0;  // narrow decode n-tiles per CTA, CTAs per KV head, partial rows
  bool decode_merge = false;                         // every narrow request has at most 4 columns
  int num_witems = 0;                                // wide decode CTAs per KV head
  int num_titems = 0;                                // tensor-core generation CTAs per KV head
  int max_tc_cols = 0;                               // most (token, head) columns of such a request
  bool tc_wide = false;                              // wide requests take the tensor-core kernel
  bool staging = false;                              // 8-bit pool with context rows: stage their pages
  bool dyn = false;                                  // bucket mode
  int max_ctx_tokens = 0, max_kv_len = 0;            // bucket limits (dyn)
  pkv::PlanLayout lay{};
};

int validate_pool(const pkv_pool* pool) {
  if (!pool || !pool->pool) return PKV_ERR_INVALID_ARGUMENT;
  if (pool->dtype != PKV_BF16 && pool->dtype != PKV_FP8_E4M3 && pool->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
  if (pool->num_blocks <= 0 || pool->num_kv_heads <= 0) return PKV_ERR_INVALID_ARGUMENT;
  const int B = pool->tokens_per_block;
  if (B != 16 && B != 32 && B != 64 && B != 128) return PKV_ERR_UNSUPPORTED;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (!aligned16(pool->pool)) return PKV_ERR_ALIGNMENT;
  if (pool->dtype != PKV_BF16 &&
      !(std::isfinite(pool->kv_scale_quant_orig) && std::isfinite(pool->kv_scale_orig_quant) &&
        pool->kv_scale_quant_orig > 0.f && pool->kv_scale_orig_quant > 0.f))
    return PKV_ERR_INVALID_ARGUMENT;
  return PKV_OK;
}

// Checks the batch against the host copies and fills the counts shared by both entry points.
int validate_batch(const pkv_pool* pool, const pkv_batch* b, int32_t Hq, HostPlan* hp) {
  if (!b) return PKV_ERR_INVALID_ARGUMENT;
  if (Hq <= 0 || Hq % pool->num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int R = b->num_requests, C = b->num_contexts;
  if (R < 0 || C < 0 || C > R || b->num_tokens < 0) return PKV_ERR_INVALID_ARGUMENT;
  hp->R = R;
  hp->C = C;
  hp->G = R - C;
  hp->T = b->num_tokens;
  if (R == 0) return b->num_tokens == 0 ? PKV_OK : PKV_ERR_INVALID_ARGUMENT;
  if (b->max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARGUMENT;
  if (!b->h_request_types || !b->h_context_lengths || !b->h_past_kv_lengths || !b->d_context_lengths ||
      !b->d_past_kv_lengths || !b->d_block_offsets)
    return PKV_ERR_INVALID_ARGUMENT;
  const int64_t cap = static_cast<int64_t>(b->max_blocks_per_seq) * pool->tokens_per_block;
  int64_t T = 0, ctx_tokens = 0;
  int max_gen = 0;
  for (int r = 0; r < R; ++r) {
    const int type = b->h_request_types[r];
    const int n = b->h_context_lengths[r], past = b->h_past_kv_lengths[r];
    if (n < 1 || past < 0) return PKV_ERR_INVALID_ARGUMENT;
    if (r < C) {
      if (type != PKV_REQ_CONTEXT) return PKV_ERR_BATCH_ORDER;
      ctx_tokens += n;
    } else {
      if (type != PKV_REQ_GENERATION || n > PKV_MAX_GEN_TOKENS) return PKV_ERR_BATCH_ORDER;
      max_gen = std::max(max_gen, n);
    }
    if (static_cast<int64_t>(past) + n > cap) return PKV_ERR_CAPACITY;
    if (static_cast<int64_t>(past) + n > INT32_MAX / 2) return PKV_ERR_CAPACITY;
    T += n;
  }
  if (T != b->num_tokens) return PKV_ERR_INVALID_ARGUMENT;
  if (b->d_packed_mask && (b->mask_words <= 0 || 32LL * b->mask_words < max_gen)) return PKV_ERR_INVALID_ARGUMENT;
  hp->ctx_tokens = static_cast<int>(ctx_tokens);
  hp->max_gen_tokens = max_gen;
  return PKV_OK;
}

// Largest K+V byte count one decode CTA streams.  Measured on the 7B-like, 70B-like GQA and
// mixed batches with the flat (item, KV head) grid: bf16 pools are fastest at 1 MB (2048 keys
// of a 128-dim head; 512 KB and 2 MB were 1-5 % slower), 8-bit pools at 2 MB (8192 keys), whose
// per-CTA set-up (Q split into hi / lo codes, the warps' merge) is dearer per key.
#ifndef PKV_DECODE_SPLIT_KB
#define PKV_DECODE_SPLIT_KB 1024
#endif
#ifndef PKV_DECODE_SPLIT_KB_8BIT
#define PKV_DECODE_SPLIT_KB_8BIT 2048
#endif

// Decode split length (tokens, multiple of 16): about 4 CTAs per SM over the whole batch, each
// CTA streaming at most the pool kind's byte cap above.
int choose_kv_chunk(const pkv_pool* pool, int64_t total) {
  const int64_t target = static_cast<int64_t>(device_sm_count()) * 4;
  int64_t chunk = (total * pool->num_kv_heads + target - 1) / std::max<int64_t>(target, 1);
  chunk = (chunk + 15) / 16 * 16;
  const bool q8 = pool->dtype != PKV_BF16;
  const int64_t token_bytes = 2LL * pool->head_dim * (q8 ? 1 : 2);
  const int64_t cap_kb = q8 ? PKV_DECODE_SPLIT_KB_8BIT : PKV_DECODE_SPLIT_KB;
  const int64_t cap = std::max<int64_t>(64, (cap_kb * 1024LL / token_bytes) / 16 * 16);
  return static_cast<int>(std::min<int64_t>(cap, std::max<int64_t>(64, chunk)));
}

#ifndef PKV_TC_MIN_CHUNK
#define PKV_TC_MIN_CHUNK 2048
#endif

// Decode routing and split length, from the generation requests' total KV tokens and the
// widest narrow request.  Requests with at most kDecodeNarrowMaxCols (token, query head) columns
// take the narrow kernel (8 or 16 columns per CTA, the split's tiles shared out among the warps).
// Wider ones (draft tokens, large query groups) take the tensor-core kernel when a 128-row tile
// holds whole groups and the pool is bf16 or 8-bit at head_dim 128 (rows = pairs, 128 per CTA;
// splits of whole 128-key tiles), else the wide mma.sync kernel (64 columns per CTA, every warp
// over every tile), in as many column groups as needed.
void plan_decode_shape(const pkv_pool* pool, int32_t Hq, int64_t total, int max_narrow, bool any_wide, HostPlan* hp) {
  const int group = Hq / pool->num_kv_heads;
  hp->kv_chunk = choose_kv_chunk(pool, total);
  // the tensor-core generation kernel: bf16 pools, and 8-bit pools at head_dim 128 (their codes
  // are converted to f16 in shared memory)
  hp->tc_wide = any_wide && group <= 128 && 128 % group == 0 && (pool->dtype == PKV_BF16 || pool->head_dim == 128);
  if (hp->tc_wide) {
    // whole 128-key tiles per split, enough of them to amortise a CTA's set-up, and about two
    // waves of the (one-per-SM) tensor-core CTAs: a longer split costs nothing there while every
    // extra split adds partial rows and a combine pass (measured on 64 requests x 8 draft
    // tokens: no split at all ran the kernel as fast and saved the 17 us combine)
    const int64_t waves2 = 2LL * device_sm_count();
    const int64_t tc_chunk = (total * pool->num_kv_heads + waves2 - 1) / waves2;
    hp->kv_chunk = static_cast<int>(std::max<int64_t>(
        PKV_TC_MIN_CHUNK, (std::max<int64_t>(tc_chunk, hp->kv_chunk) + pkv::kTcChunkAlign - 1) / pkv::kTcChunkAlign *
                              pkv::kTcChunkAlign));
  }
  hp->decode_nt = max_narrow > 8 ? 2 : 1;
  hp->decode_merge = max_narrow <= 4;
}

// Workspace layout for the plan's counts and capacities (hp->lay.stage_pages set by the caller).
void plan_layout(const pkv_pool* pool, const pkv_batch* b, int32_t Hq, HostPlan* hp) {
  pkv::PlanLayout& L = hp->lay;
  L.counts = 0;
  L.cu_q = L.counts + pkv::kCntWords;
  L.tile_prefix = L.cu_q + hp->R + 1;
  L.split_prefix = L.tile_prefix + hp->C + 1;
  L.item_prefix = L.split_prefix + hp->G + 1;
  L.part_prefix = L.item_prefix + hp->G + 1;
  L.item_map = (L.part_prefix + hp->G + 1 + 1) & ~1LL;  // int2 entries: 8-byte aligned
  L.witem_map = L.item_map + 2LL * hp->num_items;
  L.titem_map = L.witem_map + 2LL * hp->num_witems;
  L.titem_order = L.titem_map + 2LL * hp->num_titems;
  L.item_order = L.titem_order + 2LL * hp->num_titems;
  L.row_map = (L.item_order + 2LL * hp->num_items + 3) & ~3LL;  // int4 entries: 16-byte aligned
  L.unit_info = L.row_map + 4LL * hp->gen_rows;                 // int4 entries: 16-byte aligned
  L.stage_prefix = L.unit_info + 4LL * hp->num_tiles;
  L.stage_tbl = L.stage_prefix + (hp->staging ? hp->C + 1 : 0);
  L.int_words = L.stage_tbl + (hp->staging ? static_cast<int64_t>(hp->C) * b->max_blocks_per_seq : 0);
  const int64_t int_bytes = (L.int_words * 4 + 255) / 256 * 256;
  const int64_t D = pool->head_dim;
  L.part_o = int_bytes;
  L.part_ml = L.part_o + (static_cast<int64_t>(hp->num_parts) * Hq * D * 4 + 255) / 256 * 256;
  L.stage_pool = L.part_ml + (static_cast<int64_t>(hp->num_parts) * Hq * 2 * 4 + 255) / 256 * 256;
  L.total_bytes = L.stage_pool + (L.stage_pages * 2 * pool->tokens_per_block * pool->num_kv_heads * D * 2 + 255) / 256 * 256;
}

// Exact plan from the host copies of the lengths.
void plan_attention(const pkv_pool* pool, const pkv_batch* b, int32_t Hq, HostPlan* hp) {
  hp->dyn = false;
  hp->staging = pool->dtype != PKV_BF16 && hp->C > 0;
  hp->gen_rows = hp->T - hp->ctx_tokens;
  hp->num_tiles = 0;
  for (int r = 0; r < hp->C; ++r)
    hp->num_tiles += (b->h_context_lengths[r] + pkv::kCtxRowsPerCta - 1) / pkv::kCtxRowsPerCta;
  const int group = Hq / pool->num_kv_heads;
  int max_narrow = 0;
  bool any_wide = false;
  int64_t total = 0;
  for (int r = hp->C; r < hp->R; ++r) {
    const int cols_r = b->h_context_lengths[r] * group;
    if (cols_r <= pkv::kDecodeNarrowMaxCols) max_narrow = std::max(max_narrow, cols_r);
    else any_wide = true;
    total += b->h_past_kv_lengths[r] + b->h_context_lengths[r];
  }
  plan_decode_shape(pool, Hq, total, max_narrow, any_wide, hp);
  const int cols = 8 * hp->decode_nt;
  hp->num_splits = hp->max_splits = hp->num_items = hp->num_witems = hp->num_titems = hp->num_parts = 0;
  hp->max_tc_cols = 0;
  for (int r = hp->C; r < hp->R; ++r) {
    const int n = b->h_context_lengths[r], cols_r = n * group;
    const int s = (b->h_past_kv_lengths[r] + n + hp->kv_chunk - 1) / hp->kv_chunk;
    hp->num_splits += s;
    if (cols_r <= pkv::kDecodeNarrowMaxCols) hp->num_items += s * ((cols_r + cols - 1) / cols);
    else if (hp->tc_wide) {
      hp->num_titems += s * ((cols_r + pkv::kCtxTileM - 1) / pkv::kCtxTileM);
      hp->max_tc_cols = std::max(hp->max_tc_cols, cols_r);
    } else {
      hp->num_witems += s * ((cols_r + pkv::kDecodeWideCols - 1) / pkv::kDecodeWideCols);
    }
    hp->num_parts += s * n;
    hp->max_splits = std::max(hp->max_splits, s);
  }
  hp->lay.stage_pages = 0;
  if (hp->staging)
    for (int r = 0; r < hp->C; ++r)
      hp->lay.stage_pages += (b->h_past_kv_lengths[r] + b->h_context_lengths[r] + pool->tokens_per_block - 1) /
                             pool->tokens_per_block;
  plan_layout(pool, b, Hq, hp);
}

// Checks a bucket call's slot layout and limits (no lengths are read on the host).
int validate_bucket(const pkv_pool* pool, const pkv_batch* b, const pkv_bucket* bk, int32_t Hq, HostPlan* hp) {
  if (!b || !bk) return PKV_ERR_INVALID_ARGUMENT;
  if (Hq <= 0 || Hq % pool->num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int R = b->num_requests, C = b->num_contexts, T = b->num_tokens;
  if (R < 0 || C < 0 || C > R || T < 0) return PKV_ERR_INVALID_ARGUMENT;
  hp->R = R;
  hp->C = C;
  hp->G = R - C;
  hp->T = T;
  if (R == 0 || T == 0) return PKV_OK;
  if (b->max_blocks_per_seq <= 0 || !b->d_context_lengths || !b->d_past_kv_lengths || !b->d_block_offsets)
    return PKV_ERR_INVALID_ARGUMENT;
  if (bk->max_kv_len < 1 || bk->max_context_tokens < 0 || bk->max_context_tokens > T) return PKV_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(bk->max_kv_len) > static_cast<int64_t>(b->max_blocks_per_seq) * pool->tokens_per_block ||
      bk->max_kv_len > INT32_MAX / 2)
    return PKV_ERR_CAPACITY;
  if (hp->G > 0 && (bk->max_gen_tokens < 1 || bk->max_gen_tokens > PKV_MAX_GEN_TOKENS)) return PKV_ERR_BATCH_ORDER;
  const int max_gen = hp->G > 0 ? bk->max_gen_tokens : 0;
  if (b->d_packed_mask && (b->mask_words <= 0 || 32LL * b->mask_words < max_gen)) return PKV_ERR_INVALID_ARGUMENT;
  hp->dyn = true;
  hp->max_ctx_tokens = C > 0 ? bk->max_context_tokens : 0;
  hp->max_kv_len = bk->max_kv_len;
  hp->max_gen_tokens = max_gen;
  return PKV_OK;
}

// Capacities for the largest batch a bucket admits.  Context units: sum_r ceil(n_r / 256) is at
// most floor(rows / 256) + (context slots).  Generation: at most min(T, G * max_gen) rows, each
// slot at most ceil(max_kv_len / kv_chunk) splits of one column group (narrow) or
// ceil(max_gen * g / columns per CTA) groups (wide / tensor-core).
void plan_attention_bucket(const pkv_pool* pool, const pkv_batch* b, int32_t Hq, HostPlan* hp) {
  const int group = Hq / pool->num_kv_heads;
  hp->staging = pool->dtype != PKV_BF16 && hp->max_ctx_tokens > 0;
  hp->num_tiles = hp->max_ctx_tokens > 0 ? hp->max_ctx_tokens / pkv::kCtxRowsPerCta + hp->C : 0;
  hp->ctx_tokens = hp->max_ctx_tokens;
  hp->gen_rows = static_cast<int>(std::min<int64_t>(hp->T, static_cast<int64_t>(hp->G) * hp->max_gen_tokens));
  int max_narrow = 0;
  for (int n = 1; n <= hp->max_gen_tokens; ++n)
    if (n * group <= pkv::kDecodeNarrowMaxCols) max_narrow = n * group;
  const bool any_wide = hp->G > 0 && hp->max_gen_tokens * group > pkv::kDecodeNarrowMaxCols;
  plan_decode_shape(pool, Hq, static_cast<int64_t>(hp->G) * hp->max_kv_len, max_narrow, any_wide, hp);
  const int s_max = hp->G > 0 ? (hp->max_kv_len + hp->kv_chunk - 1) / hp->kv_chunk : 0;
  const int wide_cols = hp->max_gen_tokens * group;
  hp->num_splits = hp->G * s_max;
  hp->max_splits = s_max;
  hp->num_items = (hp->G > 0 && group <= pkv::kDecodeNarrowMaxCols) ? hp->G * s_max : 0;
  hp->num_witems = (any_wide && !hp->tc_wide)
                       ? hp->G * s_max * ((wide_cols + pkv::kDecodeWideCols - 1) / pkv::kDecodeWideCols)
                       : 0;
  hp->num_titems = hp->tc_wide ? hp->G * s_max * ((wide_cols + pkv::kCtxTileM - 1) / pkv::kCtxTileM) : 0;
  hp->max_tc_cols = hp->tc_wide ? wide_cols : 0;
  hp->num_parts = s_max * hp->gen_rows;
  hp->lay.stage_pages =
      hp->staging ? static_cast<int64_t>(hp->C) * ((hp->max_kv_len + pool->tokens_per_block - 1) / pool->tokens_per_block)
                  : 0;
  plan_layout(pool, b, Hq, hp);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// A batch with both context and generation rows runs its generation kernels (HBM-bound) on an
// auxiliary stream of the device's highest priority, beside the context kernel (tensor-bound)
// on the caller's stream; the auxiliary stream is forked from and joined back into the
// caller's stream with events.  Whenever an SM frees up, pending generation CTAs are placed
// first, so the long context units fill the rest of the machine.  (Measured against the
// context kernel on the auxiliary stream, at default or high priority: this order gave the
// shortest mixed steps.)  One stream and event pair per device, created on first use and kept
// for the life of the process; `lock` is held from the fork's record to the join's wait so
// that calls from several host threads never interleave on the shared events.
struct AuxStream {
  std::mutex lock;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};

AuxStream* aux_stream_for_current_device(cudaStream_t caller) {
  static AuxStream aux[64];
  static std::mutex create_lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  AuxStream* a = &aux[dev];
  std::lock_guard<std::mutex> g(create_lock);
  if (!a->tried) {
    // creating a stream is not a stream operation, but stay clear of it while the caller's
    // stream is being captured: such a call keeps the single-stream order until the next
    // uncaptured call has created the pair
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
    a->tried = true;
    int lo = 0, hi = 0;
    cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (cudaStreamCreateWithPriority(&a->stream, cudaStreamNonBlocking, hi) != cudaSuccess ||
        cudaEventCreateWithFlags(&a->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&a->join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      a->stream = nullptr;
    }
  }
  return a->stream ? a : nullptr;
}

// Joins the auxiliary stream back into the caller's stream when the call returns, on error
// paths too, so that a capture never ends with forked work left over.
struct AuxJoin {
  AuxStream* aux;
  cudaStream_t caller;
  bool join() {
    if (!aux) return true;
    const bool ok = cudaEventRecord(aux->join, aux->stream) == cudaSuccess &&
                    cudaStreamWaitEvent(caller, aux->join, 0) == cudaSuccess;
    aux = nullptr;
    return ok;
  }
  ~AuxJoin() { join(); }
};

// The append's argument checks and launch, shared by the exact and the bucket entry points
// (hp.T is the rows' count or capacity; the lengths themselves are only read on the device).
int append_impl(const pkv_pool* pool, const pkv_batch* batch, const HostPlan& hp, int32_t num_q_heads, const void* q,
                int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v, int64_t v_row_stride,
                void* q_out, int64_t q_out_row_stride, const float* rope_table, int32_t max_pos,
                const pkv_append_opts* opts, int32_t* d_error, pkv_stream_t stream) {
  const int D = pool->head_dim, Hkv = pool->num_kv_heads;
  if (!q || !k || !v || !q_out || !rope_table || max_pos <= 0) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(rope_table))
    return PKV_ERR_ALIGNMENT;
  if ((q_row_stride & 7) || (k_row_stride & 7) || (v_row_stride & 7) || (q_out_row_stride & 7)) return PKV_ERR_ALIGNMENT;
  if (q_row_stride < static_cast<int64_t>(num_q_heads) * D || q_out_row_stride < static_cast<int64_t>(num_q_heads) * D ||
      k_row_stride < static_cast<int64_t>(Hkv) * D || v_row_stride < static_cast<int64_t>(Hkv) * D)
    return PKV_ERR_INVALID_ARGUMENT;
  if (q_out == q && q_out_row_stride != q_row_stride) return PKV_ERR_INVALID_ARGUMENT;
  if (hp.R > 12000) return PKV_ERR_UNSUPPORTED;  // in-CTA prefix scan keeps R + 1 ints in shared memory
  const int style = opts ? opts->rope_style : PKV_ROPE_NEOX;
  const int rot = (opts && opts->rotary_dim) ? opts->rotary_dim : D;
  if (style != PKV_ROPE_NEOX && style != PKV_ROPE_GPTJ) return PKV_ERR_UNSUPPORTED;
  if (rot < 16 || rot > D || (rot & 15)) return PKV_ERR_UNSUPPORTED;
  if (opts && ((opts->q_norm_weight && !aligned16(opts->q_norm_weight)) ||
               (opts->k_norm_weight && !aligned16(opts->k_norm_weight))))
    return PKV_ERR_ALIGNMENT;
  if (opts && !(opts->norm_eps >= 0.f && std::isfinite(opts->norm_eps))) return PKV_ERR_INVALID_ARGUMENT;

  pkv::AppendParams p{};
  p.R = hp.R;
  p.C = hp.C;
  p.T = hp.T;
  p.dyn = hp.dyn ? 1 : 0;
  p.Hq = num_q_heads;
  p.Hkv = Hkv;
  p.D = D;
  p.B = pool->tokens_per_block;
  p.NB = pool->num_blocks;
  p.max_blocks = batch->max_blocks_per_seq;
  p.q = static_cast<const uint16_t*>(q);
  p.q_stride = q_row_stride;
  p.k = static_cast<const uint16_t*>(k);
  p.k_stride = k_row_stride;
  p.v = static_cast<const uint16_t*>(v);
  p.v_stride = v_row_stride;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.q_out_stride = q_out_row_stride;
  p.rope = reinterpret_cast<const float2*>(rope_table);
  p.max_pos = max_pos;
  p.style = style;
  p.rot = rot;
  p.q_norm_w = opts ? opts->q_norm_weight : nullptr;
  p.k_norm_w = opts ? opts->k_norm_weight : nullptr;
  p.norm_eps = opts ? opts->norm_eps : 0.f;
  p.pool = pool->pool;
  p.inv_scale = pool->kv_scale_orig_quant;
  p.ctx_len = batch->d_context_lengths;
  p.past = batch->d_past_kv_lengths;
  p.tbl = batch->d_block_offsets;
  p.pos_off = batch->d_position_offsets;
  p.d_error = d_error;
  reset_names();
  cudaError_t e;
  {
    LaunchScope ls(0, "append_rope", reinterpret_cast<cudaStream_t>(stream));
    e = pkv::launch_append(p, pool->dtype, reinterpret_cast<cudaStream_t>(stream));
  }
  if (e == cudaSuccess) g_last_launches = 1;
  return cuda_status(e);
}

// Persistent context CTAs beside the generation kernels (pkv::context_cta_share) from the host
// lengths of an exact plan; 8-bit pools (their decode is bound by instruction issue, not by HBM)
// keep every SM, and bucket plans leave the choice to the plan kernel.
int context_ctas(const pkv_pool* pool, const pkv_batch* b, const HostPlan& hp, int Hq, int S) {
  if (hp.dyn || pool->dtype != PKV_BF16 || hp.G == 0 || S < 8) return S;
  double tile_pairs = 0.0, items = 0.0;  // per query head
  for (int r = 0; r < hp.C; ++r) {
    const int64_t n = b->h_context_lengths[r], c = b->h_past_kv_lengths[r];
    for (int64_t j = 0; pkv::kCtxRowsPerCta * j < n; ++j) {
      const int64_t first = pkv::kCtxRowsPerCta * j;
      const int64_t rows = std::min<int64_t>(pkv::kCtxRowsPerCta, n - first);
      tile_pairs += static_cast<double>((c + first + rows + pkv::kCtxTileN - 1) / pkv::kCtxTileN);
      items += 1.0;
    }
  }
  double gen_keys = 0.0;
  for (int r = hp.C; r < hp.R; ++r)
    gen_keys += static_cast<double>(b->h_past_kv_lengths[r]) + static_cast<double>(b->h_context_lengths[r]);
  return pkv::context_cta_share(static_cast<float>(tile_pairs), static_cast<float>(items), static_cast<float>(gen_keys), Hq,
                                pool->num_kv_heads, pool->head_dim, S);
}

// The attention's argument checks and launches, shared by the exact and the bucket entry
// points: every grid comes from the plan's counts (exact) or capacities (bucket); the kernels
// read the device plan's counts and skip what this batch does not use.
int forward_impl(const pkv_pool* pool, const pkv_batch* batch, const HostPlan& hp, int32_t num_q_heads,
                 const void* q_rot, int64_t q_row_stride, void* out, float softmax_scale, void* workspace,
                 size_t workspace_bytes, int32_t* d_error, pkv_stream_t stream) {
  const int D = pool->head_dim, Hkv = pool->num_kv_heads;
  if (!q_rot || !out) return PKV_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_rot) || !aligned16(out) || (q_row_stride & 7)) return PKV_ERR_ALIGNMENT;
  if (q_row_stride < static_cast<int64_t>(num_q_heads) * D) return PKV_ERR_INVALID_ARGUMENT;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return PKV_ERR_INVALID_ARGUMENT;
  const bool q8 = pool->dtype != PKV_BF16;  // 8-bit codes with one pool scale
  if (!workspace || workspace_bytes < static_cast<size_t>(hp.lay.total_bytes)) return PKV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* ws = static_cast<int32_t*>(workspace);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;

  // generation work on the auxiliary stream when a context kernel runs beside it; while the
  // caller has per-kernel timing events set, every kernel stays on `stream` so that each pair
  // of events brackets one kernel's own work
  const bool has_ctx = hp.num_tiles > 0;
  const bool has_gen = hp.num_items + hp.num_witems + hp.num_titems > 0;
  const bool concurrent = has_ctx && has_gen && !g_events;

  pkv::PlanParams pp{};
  pp.R = hp.R;
  pp.C = hp.C;
  pp.G = hp.G;
  pp.T = hp.T;
  pp.Hkv = Hkv;
  pp.B = pool->tokens_per_block;
  pp.Hq = num_q_heads;
  pp.group = num_q_heads / Hkv;
  pp.cols_per_cta = 8 * hp.decode_nt;
  pp.cap_items = hp.num_items;
  pp.cap_parts = hp.num_parts;
  pp.cap_witems = hp.num_witems;
  pp.cap_titems = hp.num_titems;
  pp.tc_wide = hp.tc_wide ? 1 : 0;
  pp.staging = hp.staging ? 1 : 0;
  pp.gen_rows = hp.gen_rows;
  pp.dyn = hp.dyn ? 1 : 0;
  pp.max_ctx_tokens = hp.max_ctx_tokens;
  pp.max_kv_len = hp.max_kv_len;
  pp.max_gen_tokens = hp.max_gen_tokens;
  pp.ctx_share = (concurrent && hp.dyn && pool->dtype == PKV_BF16) ? 1 : 0;
  pp.num_sms = device_sm_count();
  pp.D = D;
  pp.sort_items = pool->dtype != PKV_BF16 ? 1 : 0;
  pp.cap_stage_pages = static_cast<int32_t>(hp.lay.stage_pages);
  pp.cap_tiles = hp.num_tiles;
  pp.cap_splits = hp.num_splits;
  pp.kv_chunk = hp.kv_chunk;
  pp.ctx_len = batch->d_context_lengths;
  pp.past = batch->d_past_kv_lengths;
  pp.ws = ws;
  pp.lay = hp.lay;
  pp.d_error = d_error;
  int launches = 0;
  reset_names();
  cudaError_t e;
  {
    LaunchScope ls(launches, "plan", s);
    e = pkv::launch_plan(pp, s);
  }
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  ++launches;

  const int32_t* counts = ws + hp.lay.counts;
  AuxStream* aux = concurrent ? aux_stream_for_current_device(s) : nullptr;
  std::unique_lock<std::mutex> aux_hold;
  const cudaStream_t cs = s;  // context kernels
  cudaStream_t gs = s;        // generation kernels
  if (aux) {
    aux_hold = std::unique_lock<std::mutex>(aux->lock);
    if (cudaEventRecord(aux->fork, s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaStreamWaitEvent(aux->stream, aux->fork, 0) != cudaSuccess) return PKV_ERR_CUDA;
    gs = aux->stream;
  }
  AuxJoin aux_join{aux, s};

  if (has_ctx) {
    // 8-bit pools: stage the context requests' pages as bf16 first (exact values, own table)
    const void* ctx_pool = pool->pool;
    const int32_t* ctx_tbl = batch->d_block_offsets;
    int64_t ctx_blocks = pool->num_blocks;
    if (q8) {
      pkv::StageParams sp{};
      sp.C = hp.C;
      sp.kv_dtype = pool->dtype;
      sp.B = pool->tokens_per_block;
      sp.Hkv = Hkv;
      sp.D = D;
      sp.NB = pool->num_blocks;
      sp.max_blocks = batch->max_blocks_per_seq;
      sp.total_pages = static_cast<int32_t>(hp.lay.stage_pages);
      sp.ctx_len = batch->d_context_lengths;
      sp.past = batch->d_past_kv_lengths;
      sp.tbl = batch->d_block_offsets;
      sp.stage_prefix = ws + hp.lay.stage_prefix;
      sp.stage_tbl = ws + hp.lay.stage_tbl;
      sp.pool = static_cast<const uint8_t*>(pool->pool);
      sp.stage_pool = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + hp.lay.stage_pool);
      sp.d_error = d_error;
      sp.counts = counts;
      {
        LaunchScope ls(launches, "stage_q8", cs);
        e = pkv::launch_stage_q8(sp, cs);
      }
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      ++launches;
      ctx_pool = sp.stage_pool;
      ctx_tbl = sp.stage_tbl;
      ctx_blocks = hp.lay.stage_pages;
    }
    CUtensorMap qmap, kvmap;
    if (!encode_rows_map(&qmap, q_rot, D, num_q_heads, hp.T, q_row_stride * 2, pkv::kCtxTileM)) return PKV_ERR_CUDA;
    CUtensorMap omap;  // output rows [T, Hq * D] (packed), for the full tiles' TMA stores
    if (!encode_rows_map(&omap, out, D, num_q_heads, hp.T, static_cast<int64_t>(num_q_heads) * D * 2, pkv::kCtxTileM))
      return PKV_ERR_CUDA;
    const int64_t pool_rows = ctx_blocks * 2 * pool->tokens_per_block;
    if (!encode_rows_map(&kvmap, ctx_pool, D, Hkv, pool_rows, static_cast<int64_t>(Hkv) * D * 2,
                         std::min(pool->tokens_per_block, pkv::kCtxTileN)))
      return PKV_ERR_CUDA;
    pkv::ContextParams cp{};
    cp.C = hp.C;
    cp.T = hp.T;
    cp.Hq = num_q_heads;
    cp.Hkv = Hkv;
    cp.group = num_q_heads / Hkv;
    cp.D = D;
    cp.B = pool->tokens_per_block;
    cp.NB = static_cast<int32_t>(ctx_blocks);
    cp.max_blocks = batch->max_blocks_per_seq;
    cp.num_tiles = hp.num_tiles;
    cp.num_ctas = aux ? context_ctas(pool, batch, hp, num_q_heads, device_sm_count()) : device_sm_count();
    cp.counts = counts;
    cp.cursor = ws + hp.lay.counts + pkv::kCntCursor;
    cp.cu_q = ws + hp.lay.cu_q;
    cp.tile_prefix = ws + hp.lay.tile_prefix;
    cp.unit_info = reinterpret_cast<const int4*>(ws + hp.lay.unit_info);
    cp.ctx_len = batch->d_context_lengths;
    cp.past = batch->d_past_kv_lengths;
    cp.tbl = ctx_tbl;
    cp.pool = static_cast<const uint8_t*>(ctx_pool);
    cp.out = static_cast<uint16_t*>(out);
    cp.out_stride = static_cast<int64_t>(num_q_heads) * D;
    cp.scale_log2 = q8 ? scale_log2 * pool->kv_scale_quant_orig : scale_log2;
    cp.out_scale = q8 ? pool->kv_scale_quant_orig : 1.0f;
    cp.d_error = d_error;
    {
      LaunchScope ls(launches, "context_attn", cs);
      e = pkv::launch_context(cp, &qmap, &kvmap, &omap, cs);
    }
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    ++launches;
  }

  if (has_gen) {
    pkv::DecodeParams dp{};
    dp.C = hp.C;
    dp.G = hp.G;
    dp.Hq = num_q_heads;
    dp.Hkv = Hkv;
    dp.group = num_q_heads / Hkv;
    dp.D = D;
    dp.B = pool->tokens_per_block;
    dp.NB = pool->num_blocks;
    dp.max_blocks = batch->max_blocks_per_seq;
    dp.kv_chunk = hp.kv_chunk;
    dp.gen_rows = hp.gen_rows;
    dp.counts = counts;
    dp.total_items = hp.num_items;
    dp.total_witems = hp.num_witems;
    dp.total_parts = hp.num_parts;
    dp.nt = hp.decode_nt;
    dp.merge_hilo = hp.decode_merge ? 1 : 0;
    dp.pool = static_cast<const uint8_t*>(pool->pool);
    dp.kv_scale = q8 ? pool->kv_scale_quant_orig : 1.0f;
    dp.scale_log2 = scale_log2;
    dp.q = static_cast<const uint16_t*>(q_rot);
    dp.q_stride = q_row_stride;
    dp.out = static_cast<uint16_t*>(out);
    dp.past = batch->d_past_kv_lengths;
    dp.new_len = batch->d_context_lengths;
    dp.tbl = batch->d_block_offsets;
    dp.cu_q = ws + hp.lay.cu_q;
    dp.split_prefix = ws + hp.lay.split_prefix;
    // 8-bit pools: most KV tiles first (sorted by the plan); bf16: request order
    dp.item_map = reinterpret_cast<const int2*>(ws + (q8 ? hp.lay.item_order : hp.lay.item_map));
    dp.witem_map = reinterpret_cast<const int2*>(ws + hp.lay.witem_map);
    dp.row_map = reinterpret_cast<const int4*>(ws + hp.lay.row_map);
    dp.part_prefix = ws + hp.lay.part_prefix;
    dp.mask = batch->d_packed_mask;
    dp.mask_words = batch->d_packed_mask ? batch->mask_words : 0;
    dp.part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + hp.lay.part_o);
    dp.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + hp.lay.part_ml);
    dp.d_error = d_error;
    if (hp.num_items > 0) {
      {
        LaunchScope ls(launches, "decode_splitkv", gs);
        e = pkv::launch_decode(dp, pool->dtype, false, gs);
      }
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      ++launches;
    }
    if (hp.num_witems > 0) {
      {
        LaunchScope ls(launches, "decode_splitkv_wide", gs);
        e = pkv::launch_decode(dp, pool->dtype, true, gs);
      }
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      ++launches;
    }
    if (hp.num_titems > 0) {
      // wide generation requests on the tensor-core kernel: a Q box is g heads x 128/g tokens,
      // i.e. 128 (token, head) rows of one KV head
      const int group = num_q_heads / Hkv;
      // at most 64 rows per request (and g dividing 16): two threads per Q row, the Q tile
      // loaded as four boxes of 16 rows (g heads x 16 / g tokens)
      const bool half_rows = hp.max_tc_cols <= pkv::kCtxTileM / 2 && 16 % group == 0;
      CUtensorMap qmap_g, kvmap_g;
      if (!encode_rows_map(&qmap_g, q_rot, D, num_q_heads, hp.T, q_row_stride * 2,
                           (half_rows ? 16 : pkv::kCtxTileM) / group, group))
        return PKV_ERR_CUDA;
      const int64_t pool_rows_g = static_cast<int64_t>(pool->num_blocks) * 2 * pool->tokens_per_block;
      const int box_rows_g = std::min(pool->tokens_per_block, pkv::kCtxTileN);
      if (q8 ? !encode_raw8_map(&kvmap_g, pool->pool, D, Hkv, pool_rows_g, box_rows_g)
             : !encode_rows_map(&kvmap_g, pool->pool, D, Hkv, pool_rows_g, static_cast<int64_t>(Hkv) * D * 2, box_rows_g))
        return PKV_ERR_CUDA;
      pkv::ContextParams tp{};
      tp.C = hp.C;
      tp.T = hp.T;
      tp.Hq = num_q_heads;
      tp.Hkv = Hkv;
      tp.group = group;
      tp.D = D;
      tp.B = pool->tokens_per_block;
      tp.NB = pool->num_blocks;
      tp.max_blocks = batch->max_blocks_per_seq;
      tp.cu_q = ws + hp.lay.cu_q;
      tp.ctx_len = batch->d_context_lengths;
      tp.past = batch->d_past_kv_lengths;
      tp.tbl = batch->d_block_offsets;
      tp.pool = static_cast<const uint8_t*>(pool->pool);
      tp.out = static_cast<uint16_t*>(out);
      tp.out_stride = static_cast<int64_t>(num_q_heads) * D;
      tp.scale_log2 = q8 ? scale_log2 * pool->kv_scale_quant_orig : scale_log2;
      tp.out_scale = q8 ? pool->kv_scale_quant_orig : 1.0f;
      tp.kv_dtype = pool->dtype;
      tp.half_rows = half_rows ? 1 : 0;
      tp.d_error = d_error;
      tp.G = hp.G;
      tp.counts = counts;
      tp.num_ctas = device_sm_count();
      tp.gen_cursor = ws + hp.lay.counts + pkv::kCntGenCursor;
      tp.kv_chunk = hp.kv_chunk;
      tp.num_titems = hp.num_titems;
      tp.total_parts = hp.num_parts;
      tp.titem_map = reinterpret_cast<const int2*>(ws + hp.lay.titem_order);  // most KV tiles first
      tp.split_prefix = ws + hp.lay.split_prefix;
      tp.part_prefix = ws + hp.lay.part_prefix;
      tp.mask = batch->d_packed_mask;
      tp.mask_words = batch->d_packed_mask ? batch->mask_words : 0;
      tp.part_o = dp.part_o;
      tp.part_ml = dp.part_ml;
      {
        LaunchScope ls(launches, "decode_tc", gs);
        e = pkv::launch_gen_tc(tp, &qmap_g, &kvmap_g, gs);
      }
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      ++launches;
    }
    if (hp.max_splits > 1) {
      {
        LaunchScope ls(launches, "combine", gs);
        e = pkv::launch_combine(dp, hp.max_splits, gs);
      }
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      ++launches;
    }
  }
  if (!aux_join.join()) return PKV_ERR_CUDA;  // later work on the caller's stream sees every row
  g_last_launches = launches;
  return PKV_OK;
}

}  // namespace

extern "C" {

const char* paged_kv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported geometry or dtype";
    case PKV_ERR_BATCH_ORDER: return "batch order: context requests must come first, generation requests have one token";
    case PKV_ERR_CAPACITY: return "sequence exceeds block table or RoPE table capacity";
    case PKV_ERR_ALIGNMENT: return "pointer or row stride not 16-byte aligned";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA runtime or driver call failed";
    default: return "unknown status";
  }
}

int32_t paged_kv_last_launch_count(void) { return g_last_launches; }

const char* paged_kv_last_launch_name(int32_t i) {
  return (i >= 0 && i < g_last_launches && i < 8) ? g_last_names[i] : nullptr;
}

int paged_kv_set_kernel_events(void* const* events, int32_t max_kernels) {
  if (events && max_kernels <= 0) return PKV_ERR_INVALID_ARGUMENT;
  g_events = events;
  g_events_n = events ? max_kernels : 0;
  return PKV_OK;
}

size_t paged_rope_table_bytes(int32_t head_dim, int32_t max_pos) {
  if (head_dim <= 0 || max_pos <= 0) return 0;
  return static_cast<size_t>(max_pos) * static_cast<size_t>(head_dim) * sizeof(float);
}

int paged_rope_table_build(double base, int32_t head_dim, int32_t max_pos, float* h_table) {
  if (!h_table || head_dim <= 0 || (head_dim & 1) || max_pos <= 0 || !(base > 0.0)) return PKV_ERR_INVALID_ARGUMENT;
  const int half = head_dim / 2;
  std::vector<double> theta(half);
  for (int j = 0; j < half; ++j) theta[j] = std::pow(base, -(2.0 * static_cast<double>(j)) / static_cast<double>(head_dim));
  for (int64_t p = 0; p < max_pos; ++p) {
    float* row = h_table + p * head_dim;
    for (int j = 0; j < half; ++j) {
      const double a = static_cast<double>(p) * theta[j];
      row[2 * j] = static_cast<float>(std::cos(a));
      row[2 * j + 1] = static_cast<float>(std::sin(a));
    }
  }
  return PKV_OK;
}

int paged_kv_append_rope(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads, const void* q,
                         int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                         int64_t v_row_stride, void* q_out, int64_t q_out_row_stride, const float* rope_table,
                         int32_t max_pos, int32_t* d_error, pkv_stream_t stream) {
  return paged_kv_append_rope_ex(pool, batch, num_q_heads, q, q_row_stride, k, k_row_stride, v, v_row_stride,
                                 q_out, q_out_row_stride, rope_table, max_pos, nullptr, d_error, stream);
}

int paged_kv_append_rope_ex(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads, const void* q,
                            int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                            int64_t v_row_stride, void* q_out, int64_t q_out_row_stride, const float* rope_table,
                            int32_t max_pos, const pkv_append_opts* opts, int32_t* d_error, pkv_stream_t stream) {
  g_last_launches = 0;
  int st = validate_pool(pool);
  if (st) return st;
  HostPlan hp;
  st = validate_batch(pool, batch, num_q_heads, &hp);
  if (st) return st;
  if (hp.T == 0) return PKV_OK;
  for (int r = 0; r < hp.R; ++r)
    if (static_cast<int64_t>(batch->h_past_kv_lengths[r]) + batch->h_context_lengths[r] > max_pos) return PKV_ERR_CAPACITY;
  return append_impl(pool, batch, hp, num_q_heads, q, q_row_stride, k, k_row_stride, v, v_row_stride, q_out,
                     q_out_row_stride, rope_table, max_pos, opts, d_error, stream);
}

int paged_kv_append_rope_bucket(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                int32_t num_q_heads, const void* q, int64_t q_row_stride, const void* k,
                                int64_t k_row_stride, const void* v, int64_t v_row_stride, void* q_out,
                                int64_t q_out_row_stride, const float* rope_table, int32_t max_pos,
                                const pkv_append_opts* opts, int32_t* d_error, pkv_stream_t stream) {
  g_last_launches = 0;
  int st = validate_pool(pool);
  if (st) return st;
  HostPlan hp;
  st = validate_bucket(pool, batch, bucket, num_q_heads, &hp);
  if (st) return st;
  if (hp.T == 0 || hp.R == 0) return PKV_OK;
  if (max_pos < bucket->max_kv_len) return PKV_ERR_CAPACITY;  // every position of the bucket has a table row
  return append_impl(pool, batch, hp, num_q_heads, q, q_row_stride, k, k_row_stride, v, v_row_stride, q_out,
                     q_out_row_stride, rope_table, max_pos, opts, d_error, stream);
}

size_t paged_attention_workspace_size(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads) {
  if (validate_pool(pool)) return 0;
  HostPlan hp;
  if (validate_batch(pool, batch, num_q_heads, &hp)) return 0;
  plan_attention(pool, batch, num_q_heads, &hp);
  return static_cast<size_t>(hp.lay.total_bytes);
}

int paged_attention_forward(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads, const void* q_rot,
                            int64_t q_row_stride, void* out, float softmax_scale, void* workspace,
                            size_t workspace_bytes, int32_t* d_error, pkv_stream_t stream) {
  g_last_launches = 0;
  int st = validate_pool(pool);
  if (st) return st;
  HostPlan hp;
  st = validate_batch(pool, batch, num_q_heads, &hp);
  if (st) return st;
  if (hp.T == 0) return PKV_OK;
  plan_attention(pool, batch, num_q_heads, &hp);
  return forward_impl(pool, batch, hp, num_q_heads, q_rot, q_row_stride, out, softmax_scale, workspace,
                      workspace_bytes, d_error, stream);
}

size_t paged_attention_bucket_workspace_size(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                             int32_t num_q_heads) {
  if (validate_pool(pool)) return 0;
  HostPlan hp;
  if (validate_bucket(pool, batch, bucket, num_q_heads, &hp)) return 0;
  if (hp.R == 0 || hp.T == 0) return 256;
  plan_attention_bucket(pool, batch, num_q_heads, &hp);
  return static_cast<size_t>(hp.lay.total_bytes);
}

int paged_attention_forward_bucket(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                   int32_t num_q_heads, const void* q_rot, int64_t q_row_stride, void* out,
                                   float softmax_scale, void* workspace, size_t workspace_bytes, int32_t* d_error,
                                   pkv_stream_t stream) {
  g_last_launches = 0;
  int st = validate_pool(pool);
  if (st) return st;
  HostPlan hp;
  st = validate_bucket(pool, batch, bucket, num_q_heads, &hp);
  if (st) return st;
  if (hp.T == 0 || hp.R == 0) return PKV_OK;
  plan_attention_bucket(pool, batch, num_q_heads, &hp);
  return forward_impl(pool, batch, hp, num_q_heads, q_rot, q_row_stride, out, softmax_scale, workspace,
                      workspace_bytes, d_error, stream);
}

}  // extern "C"
