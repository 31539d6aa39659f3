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
  kCntCtxCtas = 10,    // context CTAs that take work (the rest exit at once), see context_cta_share
  kCntGenCursor = 11,  // work-queue cursor of the tensor-core generation kernel (zeroed by the plan)
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
  int64_t titem_order;   // [num_titems] int2: titem_map's entries, most KV tiles first
  int64_t item_order;    // [num_items] int2: item_map's entries, most KV tiles first (8-bit pools)
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
#if defined(__CUDACC__)
#define PKV_HD __host__ __device__
#else
#define PKV_HD
#endif

// Persistent context CTAs when the generation kernels run beside the context kernel.  A context
// CTA holds its SM (all of its shared memory and registers) until the unit queue is empty, so
// the generation kernels get only the SMs it leaves free.  On a bf16 pool the generation kernels
// stream at the HBM limit from about two thirds of the SMs, so the context kernel gets the share
// that lets both finish together: the N minimising
//   max(Tc * S / N, Tg * max(1, (2S/3) / (S - N)))
// with Tc the context kernel's time alone (1.45 us per pair of 128-row Q tile and 128-key tile
// and 1.9 us per (unit, query head), per SM, times 1.3 for running beside HBM-bound work) and Tg
// the generation requests' K and V bytes at 6.3 TB/s (calibrated on GB300 over mixes of 2 to 16
// chunked contexts with 64 to 128 decodes and over the 16K prefill beside 8 long decodes: steps
// 5-12% shorter than with every SM).  tile_pairs and units are per query head.
PKV_HD inline int context_cta_share(float tile_pairs, float units, float gen_keys, int Hq, int Hkv, int D, int S) {
  if (S < 8) return S;
  const float t_ctx = 1.3f * (tile_pairs * 1.45f + units * 1.9f) * Hq / S;  // us
  const float t_gen = gen_keys * Hkv * D * 4.0f / 6.3e6f;                   // us
  if (!(t_gen > 0.f)) return S;
  // cost(N) = max(t_ctx S / N, t_gen max(1, m_sat / (S - N))): the first term falls and the
  // second rises with N, so the best N is where they cross (or an end of [S/8, S - 1]); with
  // every SM the generation work mostly waits for the context.  Closed form, no loop: the plan
  // kernel evaluates this on one thread.
  const float a = t_ctx * S, m_sat = 2.0f * S / 3.0f;
  float n = a / t_gen;                                    // crossing with S - N >= m_sat
  if (n > S - m_sat) n = a * S / (a + t_gen * m_sat);    // crossing with S - N < m_sat
  auto cost = [&](int k) {
    const float tc = a / k, tg = t_gen * (m_sat > S - k ? m_sat / (S - k) : 1.0f);
    return tc > tg ? tc : tg;
  };
  int best = S;
  float best_t = t_ctx + t_gen;
  const int lo = S / 8, hi = S - 1;
  const int k0 = static_cast<int>(n);
  for (int k = k0; k <= k0 + 1; ++k) {
    const int kc = k < lo ? lo : (k > hi ? hi : k);
    const float t = cost(kc);
    if (t < best_t) {
      best_t = t;
      best = kc;
    }
  }
  return best;
}

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
  // 1: the plan picks the context CTAs beside the generation kernels (context_cta_share) from
  // the device lengths (bucket plans on a bf16 pool); 0: every launched context CTA takes work
  int32_t ctx_share, num_sms, D;
  // 1 (8-bit pools): the narrow decode CTAs are launched in the order item_order lists them
  // (most KV tiles first); 0: in request order (item_map)
  int32_t sort_items;
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
  int32_t merge_hilo;       // E4M3 narrow kernel: every request has at most 4 columns
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
  int32_t* cursor;          // context kernel: the counts block's work-queue word
  int32_t* gen_cursor;      // generation kernel: its work-queue word
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
  // generation kernel (wide generation requests on the tensor cores): work items = titem_map
  // entry (generation request, split x row group) x KV head
  int32_t G, kv_chunk, num_titems, mask_words;
  int32_t kv_dtype;         // generation kernel: pool element kind (pkv_dtype); 8-bit codes are
                            // converted to f16 in shared memory (head_dim 128 only)
  int32_t half_rows;        // generation kernel: every item has at most 64 rows and 16 % group == 0
                            // (two threads per Q row, the Q map's box 16 / group tokens)
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
