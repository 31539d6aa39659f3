// internal.h -- parameter blocks and launchers shared between the C-ABI front end (api.cpp)
// and the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "paged_kv.h"

namespace pkv {

constexpr int kCtxTileM = 128;   // query rows per context-attention tile (tcgen05 M)
constexpr int kCtxRowsPerCta = 256;  // a context CTA owns two query tiles
constexpr int kCtxTileN = 128;   // keys per context-attention KV tile
constexpr int kDecodeTile = 16;  // tokens per decode warp tile (mma.sync M)
// Generation requests whose score tile has at most this many (token, query head) columns run
// on the narrow decode kernel, wider ones (draft tokens, large query groups) on the wide one.
constexpr int kDecodeNarrowMaxCols = 16;
constexpr int kDecodeWideCols = 64;  // columns per wide-decode CTA (4 warps x 16)
constexpr int kTcChunkAlign = 128;   // split length multiple when generation rows use the tensor-core kernel

// Counts the plan kernel derives from the device lengths (int32 words at the front of the
// workspace).  Every later kernel of the call reads them: a CTA whose index is at or past its
// kernel's count exits at once.  Without a bucket the counts equal the host's (the grids are
// sized exactly); with a bucket the grids are sized for the bucket's largest batch and the counts
// say how much of each grid this step's batch uses.  A batch the plan rejects gets all-zero
// counts, so nothing runs after the plan.
enum PlanCount {
  kCntTokens = 0,      // packed rows of the batch (sum of context_lengths)
  kCntGenRow0 = 1,     // first packed row of the generation requests (= context rows)
  kCntGenRows = 2,     // packed rows of the generation requests
  kCntUnits = 3,       // context units (CTAs per query head of the context kernel)
  kCntItems = 4,       // narrow decode CTAs per KV head
  kCntWitems = 5,      // wide decode CTAs per KV head
  kCntTitems = 6,      // tensor-core generation CTAs per KV head
  kCntParts = 7,       // split-KV partial rows per query head
  kCntStagePages = 8,  // 8-bit pools: staged context pages
  kCntCursor = 9,      // work-queue cursor of the context kernel (written as zero by the plan)
  kCntWords = 16
};

// Device-side plan written by plan_kernel into the front of the workspace (int32 words).
struct PlanLayout {
  int64_t counts;        // [kCntWords] PlanCount values
  int64_t cu_q;          // [R + 1]  exclusive prefix of context_lengths
  int64_t tile_prefix;   // [C + 1]  prefix of ceil(n_r / kCtxRowsPerCta) over context requests
  int64_t split_prefix;  // [G + 1]  prefix of S_r = ceil(L_r / kv_chunk) over generation requests
  int64_t item_prefix;   // [G + 1]  prefix of S_r * column groups_r (decode CTAs per KV head)
  int64_t part_prefix;   // [G + 1]  prefix of S_r * n_r (partial-result rows per query head)
  int64_t item_map;      // [num_items] int2 (generation request, item index within it)
  int64_t witem_map;     // [num_witems] the same for the wide decode kernel's CTAs
  int64_t titem_map;     // [num_titems] the same for the tensor-core kernel's generation CTAs
  int64_t row_map;       // [generation rows] int4 (splits, partial row of split 0, rows between
                         // splits = the request's new tokens, token index), 16-byte aligned
  int64_t unit_info;     // [num context units] int4 (request, first q row, past + first row,
                         // rows left), most KV tiles first (longest-first launch order)
  int64_t stage_prefix;  // [C + 1]  8-bit pools: prefix of the context requests' page counts
  int64_t stage_tbl;     // [C * max_blocks] 8-bit pools: block table into the bf16 staging pool
  int64_t int_words;     // total int32 words of the plan
  int64_t part_o;        // byte offset of fp32 partial outputs [num_parts, Hq, D]
  int64_t part_ml;       // byte offset of fp32 (m, l) pairs   [num_parts, Hq, 2]
  int64_t stage_pool;    // byte offset of the bf16 staging pool [stage_pages, 2, B, Hkv, D]
  int64_t stage_pages;   // pages in the staging pool (0 unless FP8 pool with context requests)
  int64_t total_bytes;
};

struct AppendParams {
  int32_t R, T, Hq, Hkv, D, B, NB, max_blocks;
  int32_t C;    // context requests (slots 0 .. C-1)
  int32_t dyn;  // 1: bucket mode -- T is the rows' capacity, the batch may use fewer
  int32_t stages;          // set by the launcher: depth of the shared-memory token ring
  int32_t consumer_warps;  // set by the launcher: warps that process a token's tasks
  const uint16_t* q;
  int64_t q_stride;
  const uint16_t* k;
  int64_t k_stride;
  const uint16_t* v;
  int64_t v_stride;
  uint16_t* q_out;
  int64_t q_out_stride;
  const float2* rope;  // [max_pos, rot/2]
  int32_t max_pos;
  int32_t style, rot;  // rope style (0 rotate-half, 1 interleaved), rotated dims per head
  const float* q_norm_w;  // RMSNorm weights [D] or null
  const float* k_norm_w;
  float norm_eps;
  void* pool;
  float inv_scale;
  const int32_t* ctx_len;
  const int32_t* past;
  const int32_t* tbl;
  const int32_t* pos_off;  // draft-token rotation offsets [generation rows] or null
  int32_t* d_error;
};

// Without a bucket (dyn = 0) the cap_* fields are the exact counts the host planned from its
// copies of the lengths, and a device count that differs is a plan mismatch.  With a bucket
// (dyn = 1) they are capacities: the grids' sizes for the bucket's largest batch.
struct PlanParams {
  int32_t R, C, G, T, Hkv, B, cap_tiles, cap_splits, kv_chunk, cap_stage_pages;
  int32_t Hq, group;
  int32_t cols_per_cta;  // decode score-tile columns per CTA: (token, query head) pairs
  int32_t cap_items, cap_parts, cap_witems, cap_titems;
  int32_t tc_wide;   // wide requests run on the tensor-core kernel (bf16 pool, 128 % group == 0)
  int32_t staging;   // 8-bit pool with context requests: stage their pages
  int32_t gen_rows;  // generation rows: exact (dyn = 0) or capacity (dyn = 1)
  int32_t dyn;
  // bucket limits (dyn = 1): a batch over any of them is rejected (PKV_DEVERR_BUCKET)
  int32_t max_ctx_tokens, max_kv_len, max_gen_tokens;
  const int32_t* ctx_len;
  const int32_t* past;
  int32_t* ws;  // plan words
  PlanLayout lay;
  int32_t* d_error;
};

struct DecodeParams {
  int32_t C, G, Hq, Hkv, group, D, B, NB, max_blocks, kv_chunk, total_items, total_witems;
  int32_t gen_rows;         // generation rows the combine grid covers (count or capacity)
  int32_t total_parts;      // partial-result rows the workspace holds (per query head)
  const int32_t* counts;    // the plan's PlanCount words
  int32_t nt;               // n-tiles of 8 columns per decode CTA (1 or 2)
  const uint8_t* pool;
  float kv_scale;           // dequantisation multiplier (1 for bf16)
  float scale_log2;         // softmax_scale * log2(e)
  const uint16_t* q;        // rotated q rows (bf16)
  int64_t q_stride;
  uint16_t* out;            // [T, Hq*D] bf16
  const int32_t* past;
  const int32_t* new_len;   // context_lengths
  const int32_t* tbl;
  const int32_t* cu_q;
  const int32_t* split_prefix;
  const int2* item_map;
  const int2* witem_map;
  const int4* row_map;
  const int32_t* part_prefix;
  const uint32_t* mask;     // draft-token packed mask rows [gen_rows, mask_words] or null
  int32_t mask_words;
  float* part_o;
  float* part_ml;
  int32_t* d_error;
};

struct ContextParams {
  int32_t C, T, Hq, Hkv, group, D, B, NB, max_blocks, num_tiles;
  int32_t num_ctas;         // context mode: persistent CTAs (one per SM at most)
  const int32_t* counts;    // the plan's PlanCount words
  int32_t* cursor;          // context mode: the counts block's work-queue word
  const int32_t* cu_q;
  const int32_t* tile_prefix;
  const int4* unit_info;      // [num_tiles] context units in launch order: (request r, first
                              // q row, past_r + first row, rows of the request from there on)
  const int32_t* ctx_len;
  const int32_t* past;
  const int32_t* tbl;
  const uint8_t* pool;      // for the device-side page checks
  uint16_t* out;
  int64_t out_stride;
  float scale_log2;
  float out_scale;          // multiplies O at the end (the FP8 dequantisation scale, else 1)
  int32_t* d_error;
  // generation kernel (wide generation requests on the tensor cores): CTA = titem_map
  // entry (generation request, split x row group) x KV head
  int32_t G, kv_chunk, num_titems, mask_words;
  int32_t kv_dtype;         // generation kernel: pool element kind (pkv_dtype); 8-bit codes are
                            // converted to f16 in shared memory (head_dim 128 only)
  int64_t total_parts;
  const int2* titem_map;
  const int32_t* split_prefix;
  const int32_t* part_prefix;
  const uint32_t* mask;
  float* part_o;
  float* part_ml;
};

// 8-bit pools with context requests: copies the context requests' pages into a bf16 staging
// pool holding each code's exact value (every E4M3 value and every int8 is a bf16 value), with
// its own block table.
struct StageParams {
  int32_t C, B, Hkv, D, NB, max_blocks, total_pages;
  int32_t kv_dtype;  // PKV_FP8_E4M3 or PKV_INT8
  const int32_t* counts;  // the plan's PlanCount words
  const int32_t* ctx_len;
  const int32_t* past;
  const int32_t* tbl;
  const int32_t* stage_prefix;
  int32_t* stage_tbl;
  const uint8_t* pool;
  uint16_t* stage_pool;
  int32_t* d_error;
};

// Launch `kernel` with programmatic stream serialisation (it may begin while the previous
// kernel on the stream drains; the kernel itself waits with griddepcontrol.wait).
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_append(const AppendParams& p, int kv_dtype, cudaStream_t s);
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);
// wide = false: requests with at most 16 score columns (KV split across warps); true: wider
// requests (columns split across warps, 64 per CTA).
cudaError_t launch_decode(const DecodeParams& p, int kv_dtype, bool wide, cudaStream_t s);
cudaError_t launch_combine(const DecodeParams& p, int max_splits, cudaStream_t s);
cudaError_t launch_stage_q8(const StageParams& p, cudaStream_t s);
// q_map / kv_map are CUtensorMap objects (128-byte, opaque here) built by the front end.
// Context units (persistent kernel, at most num_ctas CTAs); out_map: the output rows as a tiled
// map (box 128 rows x 64 columns of one head) for the full tiles' TMA stores.
cudaError_t launch_context(const ContextParams& p, const void* q_map, const void* kv_map, const void* out_map,
                           cudaStream_t s);
// Wide generation requests on the tensor cores (rows = (token, head) pairs of one KV head, q_map
// boxes g heads x 128/g tokens, partial results for split requests).
cudaError_t launch_gen_tc(const ContextParams& p, const void* q_map, const void* kv_map, cudaStream_t s);

}  // namespace pkv
