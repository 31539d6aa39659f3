// decode_attn.cu -- launch plan, split-KV ("flash-decoding") paged attention for generation
// requests, and the log-sum-exp combine of the splits.
//
// Pages: "TensorRT-LLM 1.0 源码学习笔记", 6.3 "Paged Attention Kernel 内部" (one query token per
// generation request; loop over the request's KV blocks through the block pointers; QK^T,
// softmax, weighted sum of V) and 6.1 "两者分工" (generation = input length 1);
// "TensorRT-LLM 源码完全拆解(一)", "AttentionMetadata 的字段与它的含义" (packed rows, host and
// device copies of the lengths); "TensorRT-LLM框架概述" (intelliparadigm.com) section 1: decode
// is bound by memory bandwidth; adg.csdn.net/69730cc6 section 1.4 (draft tokens: several new
// tokens per generation request, position offsets, packed masks).
//
// Redesign for GB300 (the pages' kernel gives one CTA per (request, head); here):
//   * the work unit is (generation request, KV head, split of kv_chunk tokens), so short and
//     long requests both fill 152 SMs;
//   * the score tile's columns are the (token, query head) pairs of one KV head, so each KV head
//     is read once for its whole GQA query group and all of the request's draft tokens:
//     S^T = K Q^T and O^T += V^T P^T run on mma.sync with the pairs on N;
//   * narrow kernel (<= 16 columns): a CTA's warps each stream their own run of 16-token tiles
//     with a cp.async ring through shared memory (zero-fill past the sequence end, one
//     block-table lookup per tile) and merge in shared memory at the end;
//     wide kernel (more columns, 8-bit pools or groups that do not divide 128; bf16 pools with
//     such requests otherwise take the tcgen05 generation kernel): the warps share one
//     ring and each owns 16 columns over every tile;
//   * online softmax in base 2 with warp-shuffle column maxima; draft-token visibility as a
//     64-bit mask per column, applied only to tiles that hold new keys;
//   * the splits of one request are merged by a combine kernel with a log-sum-exp rescale (a
//     separate launch: merging inside the decode kernel's last CTA per pair was measured slower,
//     since those merges hold SM slots that would otherwise stream KV).
// FP8 pools (narrow kernel): the codes feed mma.sync m16n8k32 E4M3 directly (K as stored, V after a 4x4 byte
// transpose in registers); Q (scaled by a power of two) and P (times 256) are each split into
// hi + lo E4M3 codes and both halves are multiplied into the same fp32 accumulator, which keeps
// about 8 significant bits of each -- the precision of a bf16 operand -- with no per-element
// conversion of the pool.  The per-pool scale is applied to scores and outputs in fp32.
// INT8 pools, and FP8 pools in the wide kernel: the codes become exact f16 values in
// registers (E4M3 by the hardware conversion; INT8 with the sign bit flipped into the
// mantissa of 1024.0: a permute and a packed subtract per two codes) and run on
// mma.sync m16n8k16 f16 with Q and P in f16; V keeps its +1152 bias through the MMA, which
// comes off at the end as 1152 times the row sum of the same rounded P.
#include <math.h>

#include "common.cuh"

namespace pkv {
namespace {

// --------------------------------------------------------------------------------------------
// plan: prefix sums the other kernels index with (one CTA)
// --------------------------------------------------------------------------------------------
constexpr int kPlanThreads = 256;

// One pass over the requests: exclusive prefix sums of (new tokens, context units of
// kCtxRowsPerCta rows, generation splits, staged FP8 context pages, decode CTAs, partial rows)
// at once, so the whole plan costs a single sweep of block-wide scans.
__device__ __forceinline__ int4 shfl_up4(int4 v, int o) {
  return make_int4(__shfl_up_sync(0xffffffffu, v.x, o), __shfl_up_sync(0xffffffffu, v.y, o),
                   __shfl_up_sync(0xffffffffu, v.z, o), __shfl_up_sync(0xffffffffu, v.w, o));
}
__device__ __forceinline__ int4 add4(int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ int4 sub4(int4 a, int4 b) { return make_int4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }

// Block-wide exclusive scan of a pair of int4 values per thread (one chunk of kPlanThreads
// requests); returns the exclusive prefix within the chunk plus the running carry.
struct Int8v {
  int4 a, b;
};
__device__ __forceinline__ Int8v scan_chunk(const Int8v x, Int8v* s_warp, const Int8v& carry, int lane, int wid) {
  Int8v incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int4 ya = shfl_up4(incl.a, o), yb = shfl_up4(incl.b, o);
    if (lane >= o) {
      incl.a = add4(incl.a, ya);
      incl.b = add4(incl.b, yb);
    }
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int4 z = make_int4(0, 0, 0, 0);
    const Int8v w = lane < kPlanThreads / 32 ? s_warp[lane] : Int8v{z, z};
    Int8v wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int4 ya = shfl_up4(wi.a, o), yb = shfl_up4(wi.b, o);
      if (lane >= o) {
        wi.a = add4(wi.a, ya);
        wi.b = add4(wi.b, yb);
      }
    }
    if (lane < kPlanThreads / 32) s_warp[lane] = Int8v{sub4(wi.a, w.a), sub4(wi.b, w.b)};
  }
  __syncthreads();
  const Int8v sw = s_warp[wid];
  return Int8v{add4(add4(carry.a, sw.a), sub4(incl.a, x.a)), add4(add4(carry.b, sw.b), sub4(incl.b, x.b))};
}

// Exclusive scan, in place, of the plan kernel's kPlanBins-bin shared histogram: each thread owns
// kPlanBins / kPlanThreads bins; shuffles inside each warp, then one warp scans the warps' totals.
// Every thread of the block calls it.
constexpr int kPlanBins = 2048;  // cost bins of the plan's counting sorts (larger costs share the top bin)
__device__ __forceinline__ void plan_hist_scan(int32_t* s_hist, int32_t* s_part, int tid, int lane, int wid) {
  constexpr int kPer = kPlanBins / kPlanThreads;
  int own = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) own += s_hist[tid * kPer + i];
  int incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_part[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < kPlanThreads / 32 ? s_part[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kPlanThreads / 32) s_part[kPlanThreads / 32 + lane] = wi - w;  // exclusive warp offsets
  }
  __syncthreads();
  int run = s_part[kPlanThreads / 32 + wid] + incl - own;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int v = s_hist[tid * kPer + i];
    s_hist[tid * kPer + i] = run;
    run += v;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  __shared__ Int8v s_warp[kPlanThreads / 32];
  __shared__ Int8v s_carry;
  __shared__ int32_t s_ctx_rows;
  __shared__ int32_t s_units, s_titems, s_items;
  __shared__ int32_t s_hist[kPlanBins];
  __shared__ int32_t s_part[kPlanThreads];
  __shared__ unsigned long long s_gen_keys, s_tile_pairs;  // for the context CTA share
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int32_t* counts = p.ws + p.lay.counts;
  int32_t* cu = p.ws + p.lay.cu_q;
  int32_t* tiles = p.ws + p.lay.tile_prefix;
  int32_t* splits = p.ws + p.lay.split_prefix;
  int32_t* items = p.ws + p.lay.item_prefix;
  int32_t* parts = p.ws + p.lay.part_prefix;
  int2* item_map = reinterpret_cast<int2*>(p.ws + p.lay.item_map);
  int4* row_map = reinterpret_cast<int4*>(p.ws + p.lay.row_map);
  int2* witem_map = reinterpret_cast<int2*>(p.ws + p.lay.witem_map);
  int2* titem_map = reinterpret_cast<int2*>(p.ws + p.lay.titem_map);
  int32_t* stage = p.ws + p.lay.stage_prefix;
  const bool staging = p.staging != 0, dyn = p.dyn != 0;
  const int C = p.C, chunk = p.kv_chunk, cols = p.cols_per_cta;
  bool bad = false;
  // The plan reads only the request lengths (written before the append kernel that precedes it,
  // which waited for them) and writes only its own words, so it runs beside that kernel's tail
  // and waits for it just before it ends (griddepcontrol.wait on every exit below): the kernels
  // after the plan start once it has ended, hence after the append too.
  const int4 z4 = make_int4(0, 0, 0, 0);
  if (tid == 0) {
    s_carry = Int8v{z4, z4};
    s_ctx_rows = 0;
    s_gen_keys = 0ull;
    s_tile_pairs = 0ull;
  }
  __syncthreads();
  // rows of the context requests: generation row k is packed row (context rows) + k
  {
    int part = 0;
    for (int r = tid; r < C; r += kPlanThreads) part += max(__ldg(p.ctx_len + r), 0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0 && part) atomicAdd(&s_ctx_rows, part);
  }
  __syncthreads();
  const int gen_row0 = s_ctx_rows;
  unsigned long long gen_keys = 0ull;  // this thread's generation requests' keys
  for (int base = 0; base < p.R; base += kPlanThreads) {
    const int r = base + tid;
    // a: (new tokens, context units, generation splits, staged 8-bit context pages)
    // b: (narrow decode CTAs per KV head, partial-result rows, wide decode CTAs per KV head,
    //     tensor-core generation CTAs per KV head)
    // Without a bucket every request has new tokens.  In a bucket a slot with none is empty,
    // and a slot over the bucket's limits rejects the batch (treated as empty meanwhile).
    Int8v x{z4, z4};
    if (r < p.R) {
      int n = __ldg(p.ctx_len + r);
      const int past = __ldg(p.past + r);
      bool bad_r;
      if (dyn) {
        bad_r = n < 0 || past < 0 || past > p.max_kv_len - n || (r >= C && n > p.max_gen_tokens);
      } else {
        bad_r = n < 1 || (r >= C && n > PKV_MAX_GEN_TOKENS);
      }
      bad |= bad_r;
      if (bad_r) n = 0;
      x.a.x = n;
      if (r < C) {
        x.a.y = (n + kCtxRowsPerCta - 1) / kCtxRowsPerCta;
        if (staging && n > 0) x.a.w = (past + n + p.B - 1) / p.B;
      } else if (n > 0) {
        gen_keys += static_cast<unsigned long long>(past + n);
        const int sr = (past + n + chunk - 1) / chunk, ncols = n * p.group;
        x.a.z = sr;
        if (ncols <= kDecodeNarrowMaxCols) x.b.x = sr * ((ncols + cols - 1) / cols);
        else if (p.tc_wide) x.b.w = sr * ((ncols + kCtxTileM - 1) / kCtxTileM);
        else x.b.z = sr * ((ncols + kDecodeWideCols - 1) / kDecodeWideCols);
        x.b.y = sr * n;
      }
    }
    const Int8v ex = scan_chunk(x, s_warp, s_carry, lane, wid);
    if (r < p.R) {
      cu[r] = ex.a.x;
      if (r < C) {
        tiles[r] = ex.a.y;
        if (staging) stage[r] = ex.a.w;
      } else {
        const int gr = r - C;
        splits[gr] = ex.a.z;
        items[gr] = ex.b.x;
        parts[gr] = ex.b.y;
        // direct maps for the decode CTAs and the combine rows (no searches there); the
        // capacities bound every write
        for (int it = 0; it < x.b.x && ex.b.x + it < p.cap_items; ++it) item_map[ex.b.x + it] = make_int2(gr, it);
        for (int it = 0; it < x.b.z && ex.b.z + it < p.cap_witems; ++it) witem_map[ex.b.z + it] = make_int2(gr, it);
        for (int it = 0; it < x.b.w && ex.b.w + it < p.cap_titems; ++it) titem_map[ex.b.w + it] = make_int2(gr, it);
        for (int i = 0; i < x.a.x; ++i) {
          const int row = ex.a.x + i - gen_row0;
          // (splits, partial row of split 0, rows between splits, token index)
          if (row >= 0 && row < p.gen_rows) row_map[row] = make_int4(x.a.z, ex.b.y + i, x.a.x, i);
        }
      }
    }
    __syncthreads();
    if (tid == kPlanThreads - 1) s_carry = Int8v{add4(ex.a, x.a), add4(ex.b, x.b)};
    __syncthreads();
  }
  bool bad_tot = false;
  if (tid == 0) {
    const Int8v t = s_carry;
    cu[p.R] = t.a.x;
    tiles[C] = t.a.y;
    splits[p.G] = t.a.z;
    items[p.G] = t.b.x;
    parts[p.G] = t.b.y;
    if (staging) stage[C] = t.a.w;
    const int gen_rows = t.a.x - gen_row0;
    if (dyn) {  // the bucket's grids must hold this batch
      bad_tot = t.a.x > p.T || gen_row0 > p.max_ctx_tokens || gen_rows > p.gen_rows || t.a.y > p.cap_tiles ||
                t.a.z > p.cap_splits || t.b.x > p.cap_items || t.b.y > p.cap_parts || t.b.z > p.cap_witems ||
                t.b.w > p.cap_titems || t.a.w > p.cap_stage_pages;
    } else {  // the device lengths must give exactly what the host planned
      bad_tot = t.a.x != p.T || gen_rows != p.gen_rows || t.a.y != p.cap_tiles || t.a.z != p.cap_splits ||
                t.b.x != p.cap_items || t.b.y != p.cap_parts || t.b.z != p.cap_witems || t.b.w != p.cap_titems ||
                (staging && t.a.w != p.cap_stage_pages);
    }
    s_units = t.a.y;
    s_titems = t.b.w;
    s_items = t.b.x;
  }
  const bool any_bad = __syncthreads_or(bad || bad_tot) != 0;
  if (tid == 0) {
    // the counts every later kernel of the call reads; a rejected batch runs nothing
    const Int8v t = s_carry;
    // (the cursor starts at zero; every launched context CTA takes work unless the share below
    // says otherwise)
    const int32_t v[kCntWords] = {t.a.x, gen_row0, t.a.x - gen_row0, t.a.y, t.b.x, t.b.z, t.b.w, t.b.y, t.a.w, 0,
                                  1 << 30};
#pragma unroll
    for (int i = 0; i < kCntWords; ++i) counts[i] = any_bad ? 0 : v[i];
    if (any_bad) flag_error(p.d_error, dyn ? PKV_DEVERR_BUCKET : PKV_DEVERR_PLAN_MISMATCH);
  }
  if (any_bad) {
    pdl_wait();
    return;
  }
  if (p.ctx_share) {  // the generation requests' keys, for the context CTA share below
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gen_keys += __shfl_xor_sync(0xffffffffu, gen_keys, o);
    if (lane == 0 && gen_keys) atomicAdd(&s_gen_keys, gen_keys);
  }

  constexpr int kBins = kPlanBins;

  // ---- tensor-core generation CTAs, most KV tiles first: a counting sort by the tile count of
  // the CTA's split (the generation kernel claims them in this order, so that its last claims
  // are short ones) ----
  const int NT = s_titems;
  if (NT > 0) {
    int2* torder = reinterpret_cast<int2*>(p.ws + p.lay.titem_order);
    auto titem_cost = [&](const int2 im) {
      const int r = C + im.x, n = __ldg(p.ctx_len + r);
      const int L = __ldg(p.past + r) + n, n_rg = max((n * p.group + kCtxTileM - 1) / kCtxTileM, 1);
      const int kt0 = (im.y / n_rg) * chunk, keys = max(min(L, kt0 + chunk) - kt0, 0);
      return min(kBins - 1, (keys + kCtxTileN - 1) / kCtxTileN);
    };
    for (int b = tid; b < kBins; b += kPlanThreads) s_hist[b] = 0;
    __syncthreads();  // titem_map (this block's global writes) and the zeroed histogram are visible
    for (int t = tid; t < NT; t += kPlanThreads) atomicAdd(&s_hist[kBins - 1 - titem_cost(titem_map[t])], 1);
    __syncthreads();
    plan_hist_scan(s_hist, s_part, tid, lane, wid);
    for (int t = tid; t < NT; t += kPlanThreads) {
      const int2 im = titem_map[t];
      torder[atomicAdd(&s_hist[kBins - 1 - titem_cost(im)], 1)] = im;
    }
    __syncthreads();  // the histogram is free again
  }

  // ---- 8-bit pools: narrow decode CTAs, most KV tiles first -- the same counting sort by the
  // tile count of the CTA's split; the decode grid launches them in this order (KV head fastest),
  // so that its last wave is made of short ones.  (Measured: 4 % faster on 8-bit pools, whose
  // splits hold twice the keys of a bf16 split and make fewer waves; on bf16 pools request order
  // was faster, as the long splits first left a last phase of short, overhead-bound CTAs.) ----
  const int NI = p.sort_items ? s_items : 0;
  if (NI > 0) {
    int2* iorder = reinterpret_cast<int2*>(p.ws + p.lay.item_order);
    auto item_cost = [&](const int2 im) {
      const int r = C + im.x, n = __ldg(p.ctx_len + r);
      const int L = __ldg(p.past + r) + n, n_cg = max((n * p.group + cols - 1) / cols, 1);
      const int kt0 = (im.y / n_cg) * chunk, keys = max(min(L, kt0 + chunk) - kt0, 0);
      return min(kBins - 1, (keys + kDecodeTile - 1) / kDecodeTile);
    };
    for (int b = tid; b < kBins; b += kPlanThreads) s_hist[b] = 0;
    __syncthreads();  // item_map (this block's global writes) and the zeroed histogram are visible
    for (int t = tid; t < NI; t += kPlanThreads) atomicAdd(&s_hist[kBins - 1 - item_cost(item_map[t])], 1);
    __syncthreads();
    plan_hist_scan(s_hist, s_part, tid, lane, wid);
    for (int t = tid; t < NI; t += kPlanThreads) {
      const int2 im = item_map[t];
      iorder[atomicAdd(&s_hist[kBins - 1 - item_cost(im)], 1)] = im;
    }
    __syncthreads();  // the histogram is free again
  }

  // ---- context units, most KV tiles first: a counting sort by tile count (descending) ----
  // Each slot gets the unit's descriptor (request, first q row, past + first row, rows left), so
  // a context CTA reads one int4 instead of searching the tile prefix itself.
  const int U = s_units;
  int4* order = reinterpret_cast<int4*>(p.ws + p.lay.unit_info);
  if (U <= 0) {
    pdl_wait();
    return;
  }
  for (int b = tid; b < kBins; b += kPlanThreads) s_hist[b] = 0;
  __syncthreads();  // tiles[] (this block's global writes) and the zeroed histogram are visible
  // the unit's request: the last slot whose unit prefix is <= u (an empty slot shares its
  // prefix with the next slot, so the search lands on the slot that owns the unit)
  auto unit_desc = [&](int u) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tiles[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    const int i0 = (u - tiles[lo]) * kCtxRowsPerCta;
    return make_int4(lo, cu[lo] + i0, __ldg(p.past + lo) + i0, __ldg(p.ctx_len + lo) - i0);
  };
  auto unit_cost = [&](const int4 d) {
    const int keys = d.z + min(kCtxRowsPerCta, d.w);
    return min(kBins - 1, (keys + kCtxTileN - 1) / kCtxTileN);
  };
  unsigned long long tile_pairs = 0ull;
  for (int u = tid; u < U; u += kPlanThreads) {
    const int c = unit_cost(unit_desc(u));
    tile_pairs += static_cast<unsigned long long>(c);
    atomicAdd(&s_hist[kBins - 1 - c], 1);
  }
  if (p.ctx_share) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tile_pairs += __shfl_xor_sync(0xffffffffu, tile_pairs, o);
    if (lane == 0 && tile_pairs) atomicAdd(&s_tile_pairs, tile_pairs);
  }
  __syncthreads();
  if (p.ctx_share && tid == 0)  // bucket plan, bf16 pool, generation kernels beside the context kernel
    counts[kCntCtxCtas] = context_cta_share(static_cast<float>(s_tile_pairs), static_cast<float>(U),
                                            static_cast<float>(s_gen_keys), p.Hq, p.Hkv, p.D, p.num_sms);
  plan_hist_scan(s_hist, s_part, tid, lane, wid);
  for (int u = tid; u < U; u += kPlanThreads) {
    const int4 d = unit_desc(u);
    order[atomicAdd(&s_hist[kBins - 1 - unit_cost(d)], 1)] = d;
  }
  pdl_wait();
}

// --------------------------------------------------------------------------------------------
// split-KV decode
// --------------------------------------------------------------------------------------------
// Tuning knobs (compile-time): cp.async ring depth per warp and tiles per iteration.
#ifndef PKV_DECODE_STAGES_BF16
#define PKV_DECODE_STAGES_BF16 3  // 96 KB per CTA at D = 128: 2 CTAs per SM
#endif
#ifndef PKV_DECODE_STAGES_FP8
#define PKV_DECODE_STAGES_FP8 2   // ring slots of SUB_FP8 tiles: 64 KB per CTA at D = 128
#endif
#ifndef PKV_DECODE_SUB_BF16
#define PKV_DECODE_SUB_BF16 1     // 16-token tiles consumed per iteration (bf16)
#endif

// Pool element kinds of the decode kernel (the pkv_dtype values).
constexpr int kKvBf16 = 0, kKvE4m3 = 1, kKvInt8 = 2;

template <int D, int KVK, bool WIDE>
struct DecodeCfg {
  // Narrow (WIDE = false): each warp streams its own share of the split's tiles through a ring
  // of its own, all warps on the same columns, merged at the end.  Wide: the CTA's warps share
  // one ring and each owns 8*NT columns of its own over every tile (no merge).
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr bool kBytes = KVK != kKvBf16;  // one byte per element (E4M3 or INT8 codes)
  static constexpr int kRowBytes = D * (kBytes ? 1 : 2);
  static constexpr int kChunksPerRow = kRowBytes / 16;
  static constexpr int kTileBytes = kDecodeTile * kRowBytes;  // one 16-token tile of K or V
  static constexpr int kSub = (kBytes || WIDE) ? 2 : PKV_DECODE_SUB_BF16;  // E4M3: PV takes 32 tokens per MMA
  static constexpr int kSlotBytes = 2 * kSub * kTileBytes;      // K then V of kSub tiles
  static constexpr int kStages = WIDE ? 4 : (kBytes ? PKV_DECODE_STAGES_FP8 : PKV_DECODE_STAGES_BF16);
  static constexpr int kRingBytes = kStages * kSlotBytes;       // one ring
  static constexpr int kRingsBytes = (WIDE ? 1 : kWarps) * kRingBytes;
  static constexpr int kLoaders = WIDE ? kThreads : 32;          // threads filling one ring
};

// Physical 16-byte chunk of logical chunk c in tile row `row` (bank-conflict-free layouts for
// the fragment loads below; each is a bijection inside a row).
template <int D, bool BYTES>
__device__ __forceinline__ int swz_k(int row, int c) {
  if constexpr (BYTES && D == 64) return c ^ (row & 3);
  else return c ^ (row & 7);
}
template <int D, bool BYTES>
__device__ __forceinline__ int swz_v(int row, int c) {
  if constexpr (!BYTES) return c ^ (row & 7);
  else if constexpr (D == 128) return c ^ (((row >> 1) & 3) << 1);
  else return c ^ (((row >> 1) & 1) << 1);
}

// 4x4 byte transpose: word j of the result holds byte j of w0, w1, w2, w3 (in that order).
__device__ __forceinline__ void transpose4x4_bytes(const uint32_t (&w)[4], uint32_t (&d)[4]) {
  const uint32_t x0 = __byte_perm(w[0], w[1], 0x5140), x1 = __byte_perm(w[0], w[1], 0x7362);
  const uint32_t y0 = __byte_perm(w[2], w[3], 0x5140), y1 = __byte_perm(w[2], w[3], 0x7362);
  d[0] = __byte_perm(x0, y0, 0x5410);
  d[1] = __byte_perm(x0, y0, 0x7632);
  d[2] = __byte_perm(x1, y1, 0x5410);
  d[3] = __byte_perm(x1, y1, 0x7632);
}

// MRG (E4M3 narrow kernel, one n-tile, at most 4 (token, head) columns per request): the hi and
// lo halves of Q go into the n-tile's columns 0-3 and 4-7 of one MMA instead of two MMAs over
// half-empty tiles, and likewise the hi and lo halves of P; the two halves of the scores are
// added with one shuffle, those of O at the end.
template <int D, int KVK, int NT, bool WIDE, bool MRG = false>
__global__ void __launch_bounds__(DecodeCfg<D, KVK, WIDE>::kThreads)
decode_splitkv_kernel(DecodeParams p) {
  using Cfg = DecodeCfg<D, KVK, WIDE>;
  constexpr bool BYTES = Cfg::kBytes, I8 = KVK == kKvInt8;
  // 8-bit codes either become exact f16 values in registers and run on f16 MMAs (INT8 always;
  // E4M3 in the wide kernel), or feed E4M3 MMAs directly with hi/lo-split Q and P (E4M3 in the
  // narrow kernel).  Measured: the hardware E4M3 -> f16 conversion made the narrow kernel 8%
  // slower than the E4M3 MMAs, while in the wide kernel, whose four sets of hi/lo fragments
  // overflow the register file, converting was 17% faster.
  constexpr bool F16 = I8 || (KVK == kKvE4m3 && WIDE);
  constexpr bool FP8 = KVK == kKvE4m3 && !F16;
  static_assert(!MRG || (FP8 && NT == 1 && !WIDE), "merged hi / lo columns: E4M3 narrow kernel, one n-tile");
  constexpr int KS = D / 16;  // k-steps over the head dim / m-tiles of O^T
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g8 = lane >> 2, q4 = lane & 3;  // fragment row group / column pair
  // narrow: one flat grid over (item in the plan's longest-first order, KV head), head fastest;
  // wide: (item, KV head)
  const int item = WIDE ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) / p.Hkv;
  const int h = WIDE ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.x) % p.Hkv;

  // ---- which generation request, split and column group this CTA owns ----
  // Columns of the score tile are (token i, query head h*group + hl) pairs of this KV head,
  // c = i*group + hl; a CTA takes HNC of them (column group cg), a warp HN.
  constexpr int HN = NT * 8;
  constexpr int HNC = WIDE ? Cfg::kWarps * HN : HN;
  if (item >= (WIDE ? p.total_witems : p.total_items)) return;
  pdl_wait();
  // the plan's counts: CTAs past this batch's share of the grid (a bucket's spare ones) exit
  if (item >= __ldg(p.counts + (WIDE ? kCntWitems : kCntItems))) return;
  const int gen_row0 = __ldg(p.counts + kCntGenRow0), gen_rows = __ldg(p.counts + kCntGenRows);
  const int2 im = (WIDE ? p.witem_map : p.item_map)[item];  // written by the plan kernel
  const int gr = min(max(im.x, 0), p.G - 1), r = p.C + gr, local = im.y;
  const int n_new = __ldg(p.new_len + r);
  const int ncols = n_new * p.group;
  const int n_cg = (ncols + HNC - 1) / HNC;
  const int s_idx = local / max(n_cg, 1), cg = local - s_idx * n_cg;
  const int num_splits = __ldg(p.split_prefix + gr + 1) - __ldg(p.split_prefix + gr);
  const int past = __ldg(p.past + r);
  const int L = past + n_new;
  const int t_begin = s_idx * p.kv_chunk;
  const int t_end = min(L, t_begin + p.kv_chunk);
  if (local < 0 || s_idx >= num_splits || t_begin >= t_end || n_new < 1 || n_new > PKV_MAX_GEN_TOKENS) {
    if (threadIdx.x == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);
    return;
  }
  const int n_tiles = (t_end - t_begin + kDecodeTile - 1) / kDecodeTile;
  const int my_first = WIDE ? 0 : (warp * n_tiles) / Cfg::kWarps;
  const int my_n = WIDE ? n_tiles : ((warp + 1) * n_tiles) / Cfg::kWarps - my_first;
  const int row0 = __ldg(p.cu_q + r);  // packed row of the request's token 0
  const int col0 = cg * HNC;                        // the CTA's first column
  const int wcol0 = col0 + (WIDE ? warp * HN : 0);  // this warp's first column
  const bool warp_cols = wcol0 < ncols;             // wide: a warp past the last pair only loads
  const int64_t part_row0 = static_cast<int64_t>(__ldg(p.part_prefix + gr)) + static_cast<int64_t>(s_idx) * n_new;
  if (row0 < gen_row0 || row0 + n_new > gen_row0 + gen_rows || part_row0 + n_new > p.total_parts) {
    if (threadIdx.x == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // device lengths disagree
    return;
  }

  // which new keys (past + j) the lane's accumulator columns (2*q4 + {0,1} of each n-tile) see:
  // bit j; a column past the last pair sees everything (its result is discarded)
  uint64_t vis[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = wcol0 + nt * 8 + (MRG ? (2 * q4 + j) & 3 : 2 * q4 + j);
      uint64_t v = ~0ull;
      if (c < ncols) {
        const int i = c / p.group;
        if (p.mask != nullptr) {
          const uint32_t* mrow = p.mask + static_cast<int64_t>(row0 + i - gen_row0) * p.mask_words;
          v = __ldg(mrow);
          if (n_new > 32 && p.mask_words > 1) v |= static_cast<uint64_t>(__ldg(mrow + 1)) << 32;
          v |= 1ull << i;
        } else {
          v = (2ull << i) - 1;  // j <= i (i = 63 wraps to all ones)
        }
      }
      vis[nt][j] = v;
    }

  // ---- Q fragments (B operand of S^T = K Q^T): column n = wcol0 + nt*8 + g8 ----
  // bf16: k16 fragments.  FP8 pool: k32 E4M3 fragments of q * 2^e split as hi + lo codes; the
  // lane holds head dims [q4*D/4, (q4+1)*D/4) and k-step kk takes its bytes 8kk .. 8kk+7.
  // INT8 pool: k16 f16 fragments of q * 2^e over the same per-lane segment, k-step kk taking its
  // elements 4kk .. 4kk+3 (the K codes are converted to f16 in the same order).
  constexpr int QW = FP8 ? D / 32 : KS;  // k-steps
  uint32_t qb[NT][QW][2];
  uint32_t ql[NT][FP8 ? QW : 1][2];
  float colscale[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = wcol0 + nt * 8 + (MRG ? g8 & 3 : g8);  // MRG: columns 4-7 repeat 0-3 (lo half)
    const bool valid = c < ncols;
    const int ci = valid ? c / p.group : 0, hl = valid ? c - ci * p.group : 0;
    const uint16_t* qh = p.q + static_cast<int64_t>(row0 + ci) * p.q_stride + static_cast<int64_t>(h * p.group + hl) * D;
    if constexpr (!BYTES) {
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qb[nt][kk][0] = valid ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * q4) : 0u;
        qb[nt][kk][1] = valid ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * q4 + 8) : 0u;
      }
      colscale[nt][0] = colscale[nt][1] = p.scale_log2;
    } else {
      float x[D / 4];
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < D / 4; e += 2) {
        uint32_t w = valid ? *reinterpret_cast<const uint32_t*>(qh + q4 * (D / 4) + e) : 0u;
        x[e] = __uint_as_float(w << 16);
        x[e + 1] = __uint_as_float(w & 0xFFFF0000u);
        amax = fmaxf(amax, fmaxf(fabsf(x[e]), fabsf(x[e + 1])));
      }
      amax = warp_max_xor(amax, 1);
      amax = warp_max_xor(amax, 2);
      int ex = 0;
      if (amax > 0.f) frexpf(amax, &ex);
      // E4M3: amax * up in [128, 256), inside E4M3's 448; f16: in [2^13, 2^14), far from 65504
      const float up = ldexpf(1.f, (F16 ? 14 : 8) - ex);
      if constexpr (F16) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          qb[nt][kk][0] = pack_f16x2(x[4 * kk] * up, x[4 * kk + 1] * up);
          qb[nt][kk][1] = pack_f16x2(x[4 * kk + 2] * up, x[4 * kk + 3] * up);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < QW; ++kk) {
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const float* xs = x + 8 * kk + 4 * b;
            uint32_t h01, l01, h23, l23;
            split_e4m3x2(xs[0] * up, xs[1] * up, h01, l01);
            split_e4m3x2(xs[2] * up, xs[3] * up, h23, l23);
            qb[nt][kk][b] = (MRG && g8 >= 4) ? (l01 | (l23 << 16)) : (h01 | (h23 << 16));
            ql[nt][kk][b] = l01 | (l23 << 16);
          }
        }
      }
      // score columns 2*q4, 2*q4+1 belong to heads held by lanes (2*q4)*4 and (2*q4+1)*4
      const float down = 1.f / up;
      const float d0 = __shfl_sync(0xffffffffu, down, (MRG ? (2 * q4) & 3 : 2 * q4) * 4);
      const float d1 = __shfl_sync(0xffffffffu, down, (MRG ? (2 * q4 + 1) & 3 : 2 * q4 + 1) * 4);
      colscale[nt][0] = d0 * p.kv_scale * p.scale_log2;
      colscale[nt][1] = d1 * p.kv_scale * p.scale_log2;
    }
  }

  float o[NT][KS][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
  }

  uint8_t* wbuf = smem + (WIDE ? 0 : warp * Cfg::kRingBytes);
  const uint32_t wbuf_s = smem_u32(wbuf);
  const int32_t* tbl_r = p.tbl + static_cast<int64_t>(r) * p.max_blocks;
  const int64_t row_pitch = static_cast<int64_t>(p.Hkv) * Cfg::kRowBytes;  // bytes between slots
  const int64_t kv_pitch = static_cast<int64_t>(p.B) * row_pitch;           // K -> V in a page
  const int log2B = 31 - __clz(p.B);                                        // B is a power of two
  constexpr int SUB = Cfg::kSub;
  const int w_begin = t_begin + my_first * kDecodeTile;
  const int w_end = min(t_end, w_begin + my_n * kDecodeTile);  // this warp's tokens
  const int n_iter = (my_n + SUB - 1) / SUB;

  // per-thread pieces of the 16-row tile copy that do not change from tile to tile (a narrow
  // warp fills its own ring, the whole CTA fills the wide ring)
  constexpr int kTileChunks = kDecodeTile * Cfg::kChunksPerRow;
  constexpr int kCopies = (kTileChunks + Cfg::kLoaders - 1) / Cfg::kLoaders;
  const int loader = WIDE ? static_cast<int>(threadIdx.x) : lane;
  int cp_row[kCopies];
  uint32_t cp_dk[kCopies], cp_dv[kCopies], cp_src[kCopies];
#pragma unroll
  for (int i = 0; i < kCopies; ++i) {
    const int c_lin = min(loader + Cfg::kLoaders * i, kTileChunks - 1);
    const int row = c_lin / Cfg::kChunksPerRow, c = c_lin % Cfg::kChunksPerRow;
    cp_row[i] = loader + Cfg::kLoaders * i < kTileChunks ? row : kDecodeTile;  // kDecodeTile: no copy
    cp_src[i] = static_cast<uint32_t>(row * row_pitch + c * 16);
    cp_dk[i] = row * Cfg::kRowBytes + (swz_k<D, BYTES>(row, c) << 4);
    cp_dv[i] = row * Cfg::kRowBytes + (swz_v<D, BYTES>(row, c) << 4);
  }

  auto load_tile = [&](int tile, uint32_t sK, uint32_t sV) {  // one 16-token tile into (sK, sV)
    const int t0 = w_begin + tile * kDecodeTile;
    const int lb = t0 >> log2B, slot0 = t0 & (p.B - 1);
    int page = (t0 < w_end && lb < p.max_blocks) ? __ldg(tbl_r + lb) : 0;
    const bool page_ok = page >= 0 && page < p.NB;
    if (!page_ok) {
      if (loader == 0) flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
      page = 0;
    }
    const uint8_t* kbase = p.pool + (static_cast<int64_t>(page) * 2 * kv_pitch) +
                           static_cast<int64_t>(slot0) * row_pitch + static_cast<int64_t>(h) * Cfg::kRowBytes;
#pragma unroll
    for (int i = 0; i < kCopies; ++i) {
      if (kTileChunks % Cfg::kLoaders != 0 && cp_row[i] >= kDecodeTile) continue;  // no chunk left
      const bool ok = page_ok && (t0 + cp_row[i] < w_end);
      const uint8_t* src = kbase + cp_src[i];
      cp_async_16(sK + cp_dk[i], ok ? src : p.pool, ok ? 16u : 0u);
      cp_async_16(sV + cp_dv[i], ok ? src + kv_pitch : p.pool, ok ? 16u : 0u);
    }
  };
  auto load_slot = [&](int it, int slot) {  // SUB consecutive tiles of this ring
    const uint32_t base = wbuf_s + slot * Cfg::kSlotBytes;
#pragma unroll
    for (int u = 0; u < SUB; ++u)
      load_tile(it * SUB + u, base + u * Cfg::kTileBytes, base + (SUB + u) * Cfg::kTileBytes);
  };

  constexpr int S = Cfg::kStages;
#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < n_iter) load_slot(s, s);
    cp_async_commit();
  }

  for (int it = 0; it < n_iter; ++it) {
    cp_async_wait<S - 2>();
    if constexpr (WIDE) __syncthreads();  // slot `it` filled by all; slot it-1 free for reuse
    else __syncwarp();
    {
      const int nxt = it + S - 1;
      if (nxt < n_iter) load_slot(nxt, nxt % S);
      cp_async_commit();
    }
    if (WIDE && !warp_cols) continue;  // warp-uniform: no columns of its own
    const int slot = it % S;
    const uint32_t sK0 = wbuf_s + slot * Cfg::kSlotBytes;
    const uint32_t sV0 = sK0 + SUB * Cfg::kTileBytes;
    const int t0 = w_begin + it * SUB * kDecodeTile;

    // ---- S^T[16 tokens x 8 columns] = K Q^T for each sub-tile ----
    float sacc[SUB][NT][4];
#pragma unroll
    for (int u = 0; u < SUB; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[u][nt][0] = sacc[u][nt][1] = sacc[u][nt][2] = sacc[u][nt][3] = 0.f;
#pragma unroll
    for (int u = 0; u < SUB; ++u) {
      const uint32_t sK = sK0 + u * Cfg::kTileBytes;
      if constexpr (!BYTES) {
        const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a[4];
          ldmatrix_x4(a, sK + row * Cfg::kRowBytes + (swz_k<D, BYTES>(row, 2 * kk + (lane >> 4)) << 4));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sacc[u][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
        }
      } else {
        constexpr int CPL = D / 64;  // 16-byte chunks per lane per row
        uint4 kw[2][CPL];
        const uint8_t* sKp = wbuf + (sK - wbuf_s);
#pragma unroll
        for (int rs = 0; rs < 2; ++rs) {
          const int row = g8 + 8 * rs;
#pragma unroll
          for (int i = 0; i < CPL; ++i)
            kw[rs][i] = *reinterpret_cast<const uint4*>(sKp + row * Cfg::kRowBytes +
                                                        (swz_k<D, BYTES>(row, q4 * CPL + i) << 4));
        }
        if constexpr (FP8) {
#pragma unroll
          for (int kk = 0; kk < QW; ++kk) {  // K codes feed the E4M3 MMA as they are
            const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&kw[0][(2 * kk) >> 2]);
            const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&kw[1][(2 * kk) >> 2]);
            const uint32_t a[4] = {w0[(2 * kk) & 3], w1[(2 * kk) & 3], w0[(2 * kk + 1) & 3], w1[(2 * kk + 1) & 3]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_e4m3_16832(sacc[u][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
              if constexpr (!MRG) mma_e4m3_16832(sacc[u][nt], a, ql[nt][kk][0], ql[nt][kk][1]);
            }
          }
          if constexpr (MRG) {  // columns j and j + 4 hold the hi and lo halves of column j
#pragma unroll
            for (int i = 0; i < 4; ++i) sacc[u][0][i] += __shfl_xor_sync(0xffffffffu, sacc[u][0][i], 2);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {  // 8-bit codes -> exact f16, four per word
            const uint32_t w0 = reinterpret_cast<const uint32_t*>(&kw[0][kk >> 2])[kk & 3];
            const uint32_t w1 = reinterpret_cast<const uint32_t*>(&kw[1][kk >> 2])[kk & 3];
            uint32_t a[4];
            if constexpr (I8) {
              i8x4_to_f16x2(w0, a[0], a[2]);
              i8x4_to_f16x2(w1, a[1], a[3]);
            } else {
              e4m3x4_to_f16x2(w0, a[0], a[2]);
              e4m3x4_to_f16x2(w1, a[1], a[3]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16_16816(sacc[u][nt], a, qb[nt][kk][0], qb[nt][kk][1]);
          }
        }
      }
    }

    // ---- online softmax over the SUB sub-tiles (columns 2*q4, 2*q4+1) ----
    uint32_t pb[SUB][NT][2];     // bf16: k16 P^T fragments per sub-tile
    uint32_t p8[NT][2][2];       // FP8: [hi/lo][sub-tile] E4M3 P^T words (k32 over both sub-tiles)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sv[SUB][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < SUB; ++u) {
        const int ta = t0 + u * kDecodeTile + g8, tb = ta + 8;
        bool ok[4] = {ta < w_end, ta < w_end, tb < w_end, tb < w_end};
        if (t0 + (u + 1) * kDecodeTile > past) {  // the tile holds new keys: apply visibility
          const int ja = ta - past, jb = tb - past;
          ok[0] = ok[0] && (ja < 0 || ((vis[nt][0] >> ja) & 1ull));
          ok[1] = ok[1] && (ja < 0 || ((vis[nt][1] >> ja) & 1ull));
          ok[2] = ok[2] && (jb < 0 || ((vis[nt][0] >> jb) & 1ull));
          ok[3] = ok[3] && (jb < 0 || ((vis[nt][1] >> jb) & 1ull));
        }
        sv[u][0] = ok[0] ? sacc[u][nt][0] * colscale[nt][0] : -INFINITY;
        sv[u][1] = ok[1] ? sacc[u][nt][1] * colscale[nt][1] : -INFINITY;
        sv[u][2] = ok[2] ? sacc[u][nt][2] * colscale[nt][0] : -INFINITY;
        sv[u][3] = ok[3] ? sacc[u][nt][3] * colscale[nt][1] : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sv[u][0], sv[u][2]));
        mx1 = fmaxf(mx1, fmaxf(sv[u][1], sv[u][3]));
      }
#pragma unroll
      for (int msk = 4; msk < 32; msk <<= 1) {
        mx0 = warp_max_xor(mx0, msk);
        mx1 = warp_max_xor(mx1, msk);
      }
      // a column that has seen no visible key yet keeps m = -inf; its exponents use base 0
      const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
      const float eb0 = mn0 == -INFINITY ? 0.f : mn0, eb1 = mn1 == -INFINITY ? 0.f : mn1;
      if (__any_sync(0xffffffffu, mn0 != m_run[nt][0] || mn1 != m_run[nt][1])) {
        const float al0 = ex2_approx(m_run[nt][0] - eb0), al1 = ex2_approx(m_run[nt][1] - eb1);
        l_run[nt][0] *= al0;
        l_run[nt][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[nt][mt][0] *= al0;
          o[nt][mt][1] *= al1;
          o[nt][mt][2] *= al0;
          o[nt][mt][3] *= al1;
        }
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
      }
#pragma unroll
      for (int u = 0; u < SUB; ++u) {
        const float p0 = ex2_approx(sv[u][0] - eb0), p1 = ex2_approx(sv[u][1] - eb1);
        const float p2 = ex2_approx(sv[u][2] - eb0), p3 = ex2_approx(sv[u][3] - eb1);
        if constexpr (!BYTES) {
          l_run[nt][0] += p0 + p2;
          l_run[nt][1] += p1 + p3;
          pb[u][nt][0] = movmatrix_trans(pack_bf16x2(p0, p1));
          pb[u][nt][1] = movmatrix_trans(pack_bf16x2(p2, p3));
        } else if constexpr (F16) {
          // f16 P; the row sums take the rounded values the MMA multiplies, so that the bias
          // of the V codes (1152 per unit weight) comes off exactly as 1152 * l at the end
          const uint32_t h01 = pack_f16x2(p0, p1), h23 = pack_f16x2(p2, p3);
          const float2 r01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
          const float2 r23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
          l_run[nt][0] += r01.x + r23.x;
          l_run[nt][1] += r01.y + r23.y;
          pb[u][nt][0] = movmatrix_trans(h01);
          pb[u][nt][1] = movmatrix_trans(h23);
        } else {
          l_run[nt][0] += p0 + p2;
          l_run[nt][1] += p1 + p3;
          // 256 * p as hi + lo E4M3 codes, one (hi | lo << 8) 16-bit element per value, so the
          // 8x8 16-bit transpose moves each value whole: lane (g, q) then holds tokens 2q, 2q+1
          // (upper rows) and 2q+8, 2q+9 (lower rows) of head g
          uint32_t h01, l01, h23, l23;
          split_e4m3x2(p0 * 256.f, p1 * 256.f, h01, l01);
          split_e4m3x2(p2 * 256.f, p3 * 256.f, h23, l23);
          const uint32_t up_t = movmatrix_trans(__byte_perm(h01, l01, 0x5140));
          const uint32_t lo_t = movmatrix_trans(__byte_perm(h23, l23, 0x5140));
          p8[nt][0][u] = __byte_perm(up_t, lo_t, 0x6420);  // hi codes of tokens 2q, 2q+1, 2q+8, 2q+9
          p8[nt][1][u] = __byte_perm(up_t, lo_t, 0x7531);  // lo codes
        }
      }
    }

    // ---- O^T[D x 8 columns] += V^T P^T ----
    if constexpr (!BYTES) {
#pragma unroll
      for (int u = 0; u < SUB; ++u) {
        const uint32_t sV = sV0 + u * Cfg::kTileBytes;
        const int row = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, sV + row * Cfg::kRowBytes + (swz_v<D, BYTES>(row, 2 * mt + ((lane >> 3) & 1)) << 4));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[nt][mt], a, pb[u][nt][0], pb[u][nt][1]);
        }
      }
    } else {
      // V^T fragments (m = head dim, k = the 32 tokens in P^T's order): for each sub-tile the lane
      // reads 4 dims of tokens 2q, 2q+1, 2q+8, 2q+9 and transposes them to one word per dim
      const int rows[4] = {2 * q4, 2 * q4 + 1, 2 * q4 + 8, 2 * q4 + 9};
#pragma unroll
      for (int pp = 0; pp < D / 32; ++pp) {
        const int c = 2 * pp + (g8 >> 2), in_chunk = (4 * g8) & 15;
        uint32_t dj[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint8_t* sVp = wbuf + (sV0 - wbuf_s) + u * Cfg::kTileBytes;
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w[i] = *reinterpret_cast<const uint32_t*>(sVp + rows[i] * Cfg::kRowBytes +
                                                      (swz_v<D, BYTES>(rows[i], c) << 4) + in_chunk);
          transpose4x4_bytes(w, dj[u]);
        }
        if constexpr (FP8) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {  // dims 32pp + 4g + 2half + {0, 1}
            const uint32_t a[4] = {dj[0][2 * half], dj[0][2 * half + 1], dj[1][2 * half], dj[1][2 * half + 1]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if constexpr (MRG) {  // hi codes in columns 0-3, lo codes in columns 4-7
                const int hl = g8 >= 4 ? 1 : 0;
                mma_e4m3_16832(o[nt][2 * pp + half], a, p8[nt][hl][0], p8[nt][hl][1]);
              } else {
                mma_e4m3_16832(o[nt][2 * pp + half], a, p8[nt][0][0], p8[nt][0][1]);
                mma_e4m3_16832(o[nt][2 * pp + half], a, p8[nt][1][0], p8[nt][1][1]);
              }
            }
          }
        } else {  // per 16-token sub-tile: dims 32pp + 4g + 2half + {0, 1} as rows
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t a[4];
              if constexpr (I8) {
                i8x4_to_f16x2_biased(dj[u][2 * half], a[0], a[2]);
                i8x4_to_f16x2_biased(dj[u][2 * half + 1], a[1], a[3]);
              } else {
                e4m3x4_to_f16x2(dj[u][2 * half], a[0], a[2]);
                e4m3x4_to_f16x2(dj[u][2 * half + 1], a[1], a[3]);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[nt][2 * pp + half], a, pb[u][nt][0], pb[u][nt][1]);
            }
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- finish per-warp row sums, then merge the warps of this CTA in shared memory ----
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l_run[nt][j];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[nt][j] = v;
    }
  __syncthreads();  // every warp is done with its ring; reuse shared memory for the merge
  float* sm_o = reinterpret_cast<float*>(smem);             // [warps][HN][D]
  float* sm_m = sm_o + Cfg::kWarps * HN * D;                 // [warps][HN]
  float* sm_l = sm_m + Cfg::kWarps * HN;                     // [warps][HN]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (g8 == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        sm_m[warp * HN + nt * 8 + 2 * q4 + j] = m_run[nt][j];
        sm_l[warp * HN + nt * 8 + 2 * q4 + j] = l_run[nt][j];
      }
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rho = g8 + 8 * (j >> 1);
        int d;
        if constexpr (!BYTES) d = 16 * mt + rho;
        else d = 32 * (mt >> 1) + 4 * (rho & 7) + 2 * (mt & 1) + (rho >> 3);
        sm_o[(warp * HN + nt * 8 + 2 * q4 + (j & 1)) * D + d] = o[nt][mt][j];
      }
  }
  __syncthreads();
  const int64_t hq0 = static_cast<int64_t>(h) * p.group;
  const int n_here = min(HNC, ncols - col0);  // valid columns of this CTA
  for (int idx = threadIdx.x; idx < n_here * D; idx += Cfg::kThreads) {
    const int cl = idx / D, d = idx - cl * D;
    const int c = col0 + cl, ci = c / p.group, hl = c - ci * p.group;
    float M = -INFINITY, acc = 0.f, lsum = 0.f;
    if constexpr (WIDE) {  // column cl belongs to warp cl / HN, which saw the whole split
      M = sm_m[cl];
      acc = sm_o[cl * D + d];
      lsum = sm_l[cl];
    } else {
#pragma unroll
      for (int w = 0; w < Cfg::kWarps; ++w) M = fmaxf(M, sm_m[w * HN + cl]);
      const float Mb = M == -INFINITY ? 0.f : M;  // no visible key in this split (draft masks)
#pragma unroll
      for (int w = 0; w < Cfg::kWarps; ++w) {
        const float f = ex2_approx(sm_m[w * HN + cl] - Mb);
        const float ow = sm_o[(w * HN + cl) * D + d] + (MRG ? sm_o[(w * HN + cl + 4) * D + d] : 0.f);
        acc += f * ow;
        lsum += f * sm_l[w * HN + cl];
      }
    }
    if constexpr (I8) acc -= kI8Bias * lsum;  // the V codes entered the MMA as 1152 + code
    acc *= FP8 ? p.kv_scale * (1.f / 256.f) : p.kv_scale;  // FP8: P entered the MMA as 256 p
    if (num_splits == 1) {
      __nv_bfloat16 b = __float2bfloat16_rn(acc / lsum);
      p.out[static_cast<int64_t>(row0 + ci) * p.Hq * D + (hq0 + hl) * D + d] = *reinterpret_cast<uint16_t*>(&b);
    } else {
      const int64_t pi = (part_row0 + ci) * p.Hq + hq0 + hl;
      p.part_o[pi * D + d] = acc;
      if (d == 0) {
        p.part_ml[pi * 2] = M;
        p.part_ml[pi * 2 + 1] = lsum;
      }
    }
  }
}

// --------------------------------------------------------------------------------------------
// log-sum-exp merge of the splits: one CTA of W warps (4, 8 or 16, by the largest split count)
// per (generation row, query head); warp w streams splits w, w+W, ... with an online max (lane
// i owns 4 consecutive head dims), then the W partial results are merged through shared memory
// --------------------------------------------------------------------------------------------
// Few splits: one warp per (generation row, query head), kCombinePairs pairs per CTA, each warp
// an online log-sum-exp over all the row's splits (lane i owns 4 consecutive head dims).
constexpr int kCombinePairs = 8;

__global__ void __launch_bounds__(kCombinePairs * 32) combine_warp_kernel(DecodeParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * kCombinePairs + warp;
  pdl_wait();
  if (pair >= static_cast<int64_t>(__ldg(p.counts + kCntGenRows)) * p.Hq) return;  // this batch's rows only
  const int grow = static_cast<int>(pair / p.Hq), hq = static_cast<int>(pair - static_cast<int64_t>(grow) * p.Hq);
  const int row = __ldg(p.counts + kCntGenRow0) + grow;
  const int4 rm = p.row_map[grow];  // written by the plan kernel earlier on the stream
  const int S = rm.x, n_new = rm.z, i = rm.w;
  if (S <= 1) return;  // written directly by the decode kernel
  const int64_t first = rm.y;  // partial row of split 0; split s: first + s * n_new
  if (i < 0 || i >= n_new || first < 0 || first + static_cast<int64_t>(S - 1) * n_new >= p.total_parts) {
    if (lane == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // device lengths disagree
    return;
  }
  const int D = p.D;
  const bool active = lane < D / 4;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + first * p.Hq + hq;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + (first * p.Hq + hq) * D) + lane;
  const int64_t stride_ml = static_cast<int64_t>(n_new) * p.Hq, stride4 = stride_ml * D / 4;
  float M = -INFINITY, lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < S; ++s) {
    const float2 m_l = ml[s * stride_ml];
    const float4 v = active ? po[s * stride4] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float Mn = fmaxf(M, m_l.x);
    const float Mb = Mn == -INFINITY ? 0.f : Mn;  // splits with no visible key (draft masks)
    const float a = ex2_approx(M - Mb), b = ex2_approx(m_l.x - Mb);
    acc.x = acc.x * a + v.x * b;
    acc.y = acc.y * a + v.y * b;
    acc.z = acc.z * a + v.z * b;
    acc.w = acc.w * a + v.w * b;
    lsum = lsum * a + m_l.y * b;
    M = Mn;
  }
  if (!active) return;
  const float inv = 1.f / lsum;
  uint2 packed = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  *reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(row) * p.Hq * D + static_cast<int64_t>(hq) * D + 4 * lane) = packed;
}

template <int W>  // warps per CTA: more for requests with many splits
__global__ void __launch_bounds__(W * 32) combine_kernel(DecodeParams p) {
  __shared__ float4 s_acc[W][32];
  __shared__ float2 s_ml[W];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grow = blockIdx.x / p.Hq, hq = blockIdx.x - grow * p.Hq;  // generation row, query head
  pdl_wait();
  if (grow >= __ldg(p.counts + kCntGenRows)) return;  // this batch's rows only
  const int row = __ldg(p.counts + kCntGenRow0) + grow;
  const int4 rm = p.row_map[grow];  // written by the plan kernel earlier on the stream
  const int S = rm.x, n_new = rm.z, i = rm.w;
  if (S <= 1) return;  // written directly by the decode kernel
  const int64_t first = rm.y;  // partial row of split 0; split s: first + s * n_new
  if (i < 0 || i >= n_new || first < 0 || first + static_cast<int64_t>(S - 1) * n_new >= p.total_parts) {
    if (threadIdx.x == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // device lengths disagree
    return;
  }
  const int D = p.D;
  const bool active = lane < D / 4;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + first * p.Hq + hq;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + (first * p.Hq + hq) * D) + lane;
  const int64_t stride_ml = static_cast<int64_t>(n_new) * p.Hq, stride4 = stride_ml * D / 4;
  float M = -INFINITY, lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = warp; s < S; s += W) {
    const float2 m_l = ml[s * stride_ml];
    const float4 v = active ? po[s * stride4] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float Mn = fmaxf(M, m_l.x);
    const float Mb = Mn == -INFINITY ? 0.f : Mn;  // splits with no visible key (draft masks)
    const float a = ex2_approx(M - Mb), b = ex2_approx(m_l.x - Mb);
    acc.x = acc.x * a + v.x * b;
    acc.y = acc.y * a + v.y * b;
    acc.z = acc.z * a + v.z * b;
    acc.w = acc.w * a + v.w * b;
    lsum = lsum * a + m_l.y * b;
    M = Mn;
  }
  s_acc[warp][lane] = acc;
  if (lane == 0) s_ml[warp] = make_float2(M, lsum);
  __syncthreads();
  if (warp != 0 || !active) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < W; ++w) Mt = fmaxf(Mt, s_ml[w].x);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float lt = 0.f;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const float f = ex2_approx(s_ml[w].x - Mt);  // a warp with no splits has M = -inf: f = 0
    const float4 a4 = s_acc[w][lane];
    o.x += f * a4.x;
    o.y += f * a4.y;
    o.z += f * a4.z;
    o.w += f * a4.w;
    lt += f * s_ml[w].y;
  }
  const float inv = 1.f / lt;
  uint2 packed = make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
  *reinterpret_cast<uint2*>(p.out + static_cast<int64_t>(row) * p.Hq * D + static_cast<int64_t>(hq) * D + 4 * lane) = packed;
}

template <int D, int KVK, int NT, bool WIDE, bool MRG = false>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  using Cfg = DecodeCfg<D, KVK, WIDE>;
  auto kern = decode_splitkv_kernel<D, KVK, NT, WIDE, MRG>;
  constexpr int kMerge = Cfg::kWarps * NT * 8 * (D + 2) * 4;  // the epilogue's staging
  constexpr int kSmem = Cfg::kRingsBytes > kMerge ? Cfg::kRingsBytes : kMerge;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int items = WIDE ? p.total_witems : p.total_items;
  const dim3 grid = WIDE ? dim3(items, p.Hkv) : dim3(static_cast<unsigned>(items) * p.Hkv, 1);
  return launch_pdl(kern, grid, dim3(Cfg::kThreads), kSmem, s, p);
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, p);
}

cudaError_t launch_combine(const DecodeParams& p, int max_splits, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(p.gen_rows) * p.Hq));
  if (max_splits <= kCombinePairs) {  // one warp per (row, head)
    const int64_t pairs = static_cast<int64_t>(p.gen_rows) * p.Hq;
    return launch_pdl(combine_warp_kernel, dim3(static_cast<unsigned>((pairs + kCombinePairs - 1) / kCombinePairs)),
                      dim3(kCombinePairs * 32), 0, s, p);
  }
  // about 8 splits per warp, 4 to 16 warps
  if (max_splits > 64) return launch_pdl(combine_kernel<16>, grid, dim3(16 * 32), 0, s, p);
  if (max_splits > 32) return launch_pdl(combine_kernel<8>, grid, dim3(8 * 32), 0, s, p);
  return launch_pdl(combine_kernel<4>, grid, dim3(4 * 32), 0, s, p);
}

template <int KVK>
cudaError_t launch_decode_kind(const DecodeParams& p, bool wide, cudaStream_t s) {
  if (wide) {  // 16 columns per warp, 64 per CTA
    return p.D == 128 ? launch_decode_t<128, KVK, 2, true>(p, s) : launch_decode_t<64, KVK, 2, true>(p, s);
  }
  if constexpr (KVK == kKvE4m3) {  // at most 4 columns per request: hi and lo in one n-tile
    if (p.merge_hilo && p.nt == 1)
      return p.D == 128 ? launch_decode_t<128, KVK, 1, false, true>(p, s) : launch_decode_t<64, KVK, 1, false, true>(p, s);
  }
  if (p.D == 128) return p.nt == 1 ? launch_decode_t<128, KVK, 1, false>(p, s) : launch_decode_t<128, KVK, 2, false>(p, s);
  return p.nt == 1 ? launch_decode_t<64, KVK, 1, false>(p, s) : launch_decode_t<64, KVK, 2, false>(p, s);
}

cudaError_t launch_decode(const DecodeParams& p, int kv_dtype, bool wide, cudaStream_t s) {
  if (kv_dtype == PKV_FP8_E4M3) return launch_decode_kind<kKvE4m3>(p, wide, s);
  if (kv_dtype == PKV_INT8) return launch_decode_kind<kKvInt8>(p, wide, s);
  return launch_decode_kind<kKvBf16>(p, wide, s);
}

}  // namespace pkv
