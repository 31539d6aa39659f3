// append_rope.cu -- GPT-NeoX RoPE on Q and K plus the append of K/V into the paged pool.
//
// Pages: "TensorRT-LLM 1.0 源码学习笔记", 二.2 "KVCacheManager 详解" (the attention op writes
// each new token's KV into the blocks named by the block table) and 6.4 "量化" (quantise on
// write with kv_scale_orig_quant); adg.csdn.net/69730cc6 section 1.1 (GPT-NeoX rotary
// embedding); "TensorRT-LLM 源码完全拆解(一)", "KVCacheManager 的三个对外接口" (pool layout
// [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]).
//
// HBM-bound.  Persistent CTAs (two per SM) each stream every (grid)-th token through a ring of
// shared-memory stages:
//   * a producer warp resolves 32 tokens at a time, one per lane (request from an in-CTA prefix
//     scan of context_lengths, slot position, rotation position, pool page), so the dependent
//     lookups of 32 tokens are in flight together; one lane then issues each token's bulk
//     copies (cp.async.bulk: its q row, k row and v row, and the RoPE table row of its rotation
//     position) into the next free stage, completing on the stage's mbarrier;
//   * consumer warps (one thread per 16-element task of a token, up to 12 warps; each thread
//     decodes its task's place once) rotate Q and K with the fixed fp32 recipe, quantise for
//     8-bit pools, and store 16-byte rows of q_out and the pool slot (8-byte for 8-bit pools);
//     each warp releases the stage with one arrive.
// A task is 16 elements of one head (8 rotation pairs, or a pass-through part of a partially
// rotated head); the heads of a token are consecutive tasks, so every row read and written is a
// run of full 32-byte sectors and the lanes of one head can reduce an RMSNorm with shuffles.
// Variants: rotate-half or interleaved pairs, partial rotary dims, the optional RMSNorm of q /
// k heads, and draft tokens rotated for past + offset (adg.csdn.net/69730cc6 section 1.4,
// spec_decoding_position_offsets) while stored at slot past + i.  Every wait is bounded; a
// wait that runs out sets PKV_DEVERR_TIMEOUT, and the producer lets its last copies land before
// the CTA ends.
#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

struct alignas(16) U16x8 {
  uint16_t v[8];
};

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ U16x8 to_bf16x8(const float (&y)[8]) {
  U16x8 r;
#pragma unroll
  for (int e = 0; e < 8; ++e) r.v[e] = f32_to_bf16_bits(y[e]);
  return r;
}

// 8 fp32 values * inv_scale -> 8 E4M3 codes (RNE, saturating), packed little-endian.
__device__ __forceinline__ uint2 to_e4m3x8(const float (&y)[8], float inv_scale) {
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float2 f = make_float2(__fmul_rn(y[4 * h + 2 * e], inv_scale), __fmul_rn(y[4 * h + 2 * e + 1], inv_scale));
      __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      acc |= static_cast<uint32_t>(two) << (16 * e);
    }
    w[h] = acc;
  }
  return make_uint2(w[0], w[1]);
}

// 8 fp32 values * inv_scale -> 8 int8 codes: nearest integer, ties to even, saturated to
// [-128, 127] (NaN -> 0), packed little-endian.
__device__ __forceinline__ uint2 to_int8x8(const float (&y)[8], float inv_scale) {
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float f = __fmul_rn(y[4 * h + e], inv_scale);
      const int c = min(max(__float2int_rn(f), -128), 127);
      acc |= (static_cast<uint32_t>(c) & 0xFFu) << (8 * e);
    }
    w[h] = acc;
  }
  return make_uint2(w[0], w[1]);
}

// ---- the kernel: a producer warp streams tokens into a shared-memory ring with bulk copies;
// W consumer warps (one task per thread per token, W <= 12) rotate / quantise / store them ----
constexpr int kMaxConsumerWarps = 12;
constexpr int kMaxAppendThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kMetaRing = 64;  // resolved tokens kept ahead (32 resolved per producer pass)
#ifndef PKV_APPEND_STAGES
#define PKV_APPEND_STAGES 4  // deepest token ring (measured: 8 no faster)
#endif
#ifndef PKV_APPEND_EARLY
#define PKV_APPEND_EARLY 0  // 1: issue the first stages' q / k / v copies before the request scan
#endif
constexpr int kMaxStages = PKV_APPEND_STAGES;

// Dynamic shared memory of one CTA: the request prefix, the token metadata ring, the ring's
// mbarriers, then the stages (each: the token's q row, k row, v row and RoPE row).
struct AppendSmem {
  int cu_off, meta_off, bar_off, stage_off, stage_bytes, stages, bytes;
  int q_bytes, kv_bytes, rope_bytes;
};
__host__ __device__ inline AppendSmem append_smem(int R, int Hq, int Hkv, int D, int rot, int stages) {
  AppendSmem L;
  L.q_bytes = Hq * D * 2;
  L.kv_bytes = Hkv * D * 2;
  L.rope_bytes = (rot / 2) * 8;
  L.cu_off = 0;
  L.meta_off = ((R + 1) * 4 + 15) & ~15;
  L.bar_off = L.meta_off + kMetaRing * 16;
  L.stage_off = (L.bar_off + 2 * kMaxStages * 8 + 127) & ~127;
  L.stage_bytes = (L.q_bytes + 2 * L.kv_bytes + L.rope_bytes + 127) & ~127;
  L.stages = stages;
  L.bytes = L.stage_off + stages * L.stage_bytes;
  return L;
}

// One task (16 elements of one head of one token, as two groups of 8) in the token's stage and
// destination row; the same for every token, so each thread decodes its tasks once.
struct TaskDesc {
  uint32_t src_a, src_b;  // byte offsets of the two groups in the stage
  int32_t cs;             // byte offset of the task's 8 (cos, sin) pairs in the stage, -1: no rotation
  int32_t dst_a, dst_b;   // element offsets in the destination row (q_out row, or the slot's K / V row)
  int32_t kind;           // 0 = q, 1 = k, 2 = v; -1: no task
  int32_t off;            // element offsets of the groups inside the head: offA | offB << 16
};

__device__ __forceinline__ TaskDesc describe_task(int task, int tasks_per_token, const AppendParams& p,
                                                  const AppendSmem& L) {
  TaskDesc d;
  d.kind = -1;
  d.src_a = d.src_b = 0;
  d.cs = -1;
  d.dst_a = d.dst_b = 0;
  d.off = 0;
  if (task >= tasks_per_token) return d;
  const int D = p.D, per_head = D >> 4, lph = 31 - __clz(per_head);
  const int rot_tasks = p.rot >> 4, rhalf = p.rot >> 1;
  int kind = 0;
  if (task >= p.Hq * per_head) {
    task -= p.Hq * per_head;
    kind = 1;
    if (task >= p.Hkv * per_head) {
      task -= p.Hkv * per_head;
      kind = 2;
    }
  }
  const int h = task >> lph, t = task & (per_head - 1);
  int offA, offB;  // element offsets of the two groups inside the head
  if (p.style == 0 && t < rot_tasks) {
    offA = 8 * t;
    offB = rhalf + 8 * t;
  } else {
    const int base = (p.style == 0) ? p.rot + 16 * (t - rot_tasks) : 16 * t;
    offA = base;
    offB = base + 8;
  }
  const uint32_t row = kind == 0 ? 0u : kind == 1 ? static_cast<uint32_t>(L.q_bytes)
                                                   : static_cast<uint32_t>(L.q_bytes + L.kv_bytes);
  d.kind = kind;
  d.src_a = row + 2u * static_cast<uint32_t>(h * D + offA);
  d.src_b = row + 2u * static_cast<uint32_t>(h * D + offB);
  d.cs = (kind != 2 && t < rot_tasks) ? L.q_bytes + 2 * L.kv_bytes + 8 * (8 * t) : -1;
  d.dst_a = h * D + offA;
  d.dst_b = h * D + offB;
  d.off = offA | (offB << 16);
  return d;
}

template <int KVK>  // pool element kind: 0 bf16, 1 E4M3 codes, 2 int8 codes
__global__ void __launch_bounds__(kMaxAppendThreads, 2) append_rope_kernel(AppendParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t s_warp[kMaxConsumerWarps + 1];
  __shared__ int32_t s_carry;
  __shared__ int32_t s_abort;
  const AppendSmem L = append_smem(p.R, p.Hq, p.Hkv, p.D, p.rot, p.stages);
  int32_t* s_cu = reinterpret_cast<int32_t*>(smem + L.cu_off);  // [R + 1] prefix of context_lengths
  int4* s_meta = reinterpret_cast<int4*>(smem + L.meta_off);   // [kMetaRing] (rotation pos, page, slot, token)
  const uint32_t smem_s = smem_u32(smem);
  const uint32_t bar_full = smem_s + L.bar_off, bar_empty = bar_full + 8 * kMaxStages;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int W = p.consumer_warps, nthreads = (W + 1) * 32;  // blockDim.x
  const int S = L.stages;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(bar_full + 8 * i, 1);   // the producer's arrive + the copies' bytes
      tc::mbar_init(bar_empty + 8 * i, W);  // one arrive per consumer warp
    }
    tc::fence_barrier_init();
    s_carry = 0;
    s_abort = 0;
  }
  __syncthreads();  // the barriers are initialised before anyone uses them
  pdl_wait();
  // The attention call's plan kernel, launched next, reads only request lengths -- visible now
  // (the wait above) and never written here -- so it may run beside this kernel; it waits for
  // this kernel before it ends, so everything after it still sees the appended rows.
  pdl_launch_dependents();
  // The first stages' q / k / v rows depend on nothing but the token index: the producer issues
  // them before the scan below, so their latency overlaps the scan and the first lookups (their
  // RoPE rows follow once the positions are known).  Rows past the batch's rows are still inside
  // the caller's buffers (a bucket's capacity), so the copies are always in bounds.
  const int cap_local = static_cast<int>(blockIdx.x) < p.T ? (p.T - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1 : 0;
  const int n_pre = PKV_APPEND_EARLY ? min(S, cap_local) : 0;
  if (wid == W && lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>(L.q_bytes + 2 * L.kv_bytes + L.rope_bytes);
    for (int j = 0; j < n_pre; ++j) {
      const int64_t token = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(j) * gridDim.x;
      const uint32_t full = bar_full + 8 * j, dst = smem_s + L.stage_off + j * L.stage_bytes;
      tc::mbar_arrive_expect_tx(full, bytes);
      tc::bulk_load_1d(dst, p.q + token * p.q_stride, L.q_bytes, full);
      tc::bulk_load_1d(dst + L.q_bytes, p.k + token * p.k_stride, L.kv_bytes, full);
      tc::bulk_load_1d(dst + L.q_bytes + L.kv_bytes, p.v + token * p.v_stride, L.kv_bytes, full);
    }
  }
  __syncthreads();
  // ---- block-wide exclusive scan of context_lengths (chunks of the block's threads) ----
  bool neg = false;
  for (int base = 0; base < p.R; base += nthreads) {
    const int r = base + tid;
    const int x = r < p.R ? __ldg(p.ctx_len + r) : 0;
    neg |= x < 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int w = lane <= W ? s_warp[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane <= W) s_warp[lane] = wi - w;  // exclusive warp offsets
    }
    __syncthreads();
    const int carry = s_carry;
    if (r < p.R) s_cu[r] = carry + s_warp[wid] + incl - x;
    __syncthreads();
    if (tid == nthreads - 1) s_carry = carry + s_warp[wid] + incl;
    __syncthreads();
  }
  if (tid == 0) s_cu[p.R] = s_carry;
  // Without a bucket the device lengths must add up to the host's token count; in a bucket
  // (p.T = the rows' capacity) the batch may use fewer rows, never more, and empty slots
  // (no new tokens) own no row
  const bool bad = __syncthreads_or(neg) != 0 || (p.dyn ? s_cu[p.R] > p.T : s_cu[p.R] != p.T);
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) flag_error(p.d_error, p.dyn ? PKV_DEVERR_BUCKET : PKV_DEVERR_PLAN_MISMATCH);
    if (wid == W && lane == 0) {  // complete the early stages (RoPE row 0) and let them land
      for (int j = 0; j < n_pre; ++j)
        tc::bulk_load_1d(smem_s + L.stage_off + j * L.stage_bytes + L.q_bytes + 2 * L.kv_bytes, p.rope, L.rope_bytes,
                         bar_full + 8 * j);
      for (int j = 0; j < n_pre; ++j) tc::mbar_wait(bar_full + 8 * j, 0, 200000000LL);
    }
    return;
  }
  const int T = s_cu[p.R];          // packed rows of this batch
  const int gen_row0 = s_cu[p.C];   // first row of the generation requests
  // this CTA's tokens: blockIdx.x, + gridDim.x, ...
  const int n_local = static_cast<int>(blockIdx.x) < T ? (T - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1 : 0;
  auto stage_addr = [&](int st) { return smem_s + L.stage_off + st * L.stage_bytes; };

  if (wid == W) {
    // ======================= producer =======================
    // Resolves 32 tokens at a time (one per lane: request, positions, page; every dependent
    // lookup of 32 tokens in flight together), then one lane issues each token's bulk copies
    // into the next free stage.
    const int log2B = 31 - __clz(p.B);
    const int rhalf = p.rot >> 1;
    int issued = 0;
    bool ok_all = true;
    for (int j = 0; j < n_local && ok_all; ++j) {
      if ((j & 31) == 0) {
        const int jj = j + lane;
        if (jj < n_local) {
          const int token = static_cast<int>(blockIdx.x) + jj * static_cast<int>(gridDim.x);
          int lo = 0, hi = p.R - 1;  // request of this token: largest r with s_cu[r] <= token
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_cu[mid] <= token) lo = mid;
            else hi = mid - 1;
          }
          const int r = lo;
          const int past_r = __ldg(p.past + r);
          const int pos = past_r + (token - s_cu[r]);  // slot position
          int rpos = pos;                               // rotation position
          bool ok = true;
          if (p.pos_off != nullptr && token >= gen_row0) {  // a draft token
            const int off = __ldg(p.pos_off + (token - gen_row0));
            if (off < 0 || off >= __ldg(p.ctx_len + r)) {
              flag_error(p.d_error, PKV_DEVERR_BAD_OFFSET);
              ok = false;
            }
            rpos = past_r + off;
          }
          if (ok && (pos < 0 || pos >= p.max_pos || rpos < 0 || rpos >= p.max_pos)) {
            flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // device lengths disagree with the host-checked ones
            ok = false;
          }
          int page = -1;
          const int lb = pos >> log2B, slot = pos & (p.B - 1);
          if (ok) {
            page = lb < p.max_blocks ? __ldg(p.tbl + static_cast<size_t>(r) * p.max_blocks + lb) : -1;
            if (page < 0 || page >= p.NB) {
              flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);  // q_out is still written, the pool is not
              page = -1;
            }
          }
          s_meta[jj & (kMetaRing - 1)] = make_int4(ok ? rpos : -1, page, slot, token);
        }
        __syncwarp();
      }
      const int st = j % S;
      if (j >= S && !__all_sync(0xffffffffu, tc::mbar_wait(bar_empty + 8 * st, ((j / S) - 1) & 1))) {
        ok_all = false;
        break;
      }
      if (lane == 0) {
        const int4 m = s_meta[j & (kMetaRing - 1)];
        const bool ok = m.x >= 0;
        const uint32_t full = bar_full + 8 * st, dst = stage_addr(st);
        if (j < n_pre) {  // q / k / v already on their way: the RoPE row (row 0 for a skipped token)
          tc::bulk_load_1d(dst + L.q_bytes + 2 * L.kv_bytes, p.rope + static_cast<size_t>(ok ? m.x : 0) * rhalf,
                           L.rope_bytes, full);
        } else {
        const uint32_t bytes = ok ? static_cast<uint32_t>(L.q_bytes + 2 * L.kv_bytes + L.rope_bytes) : 0u;
        tc::mbar_arrive_expect_tx(full, bytes);
        if (ok) {
          const int64_t token = m.w;
          tc::bulk_load_1d(dst, p.q + token * p.q_stride, L.q_bytes, full);
          tc::bulk_load_1d(dst + L.q_bytes, p.k + token * p.k_stride, L.kv_bytes, full);
          tc::bulk_load_1d(dst + L.q_bytes + L.kv_bytes, p.v + token * p.v_stride, L.kv_bytes, full);
          tc::bulk_load_1d(dst + L.q_bytes + 2 * L.kv_bytes, p.rope + static_cast<size_t>(m.x) * rhalf, L.rope_bytes,
                           full);
        }
        }
      }
      __syncwarp();
      ++issued;
    }
    // early stages of rows past this batch's last row (a bucket batch smaller than its
    // capacity): complete them with RoPE row 0 so that they land like the rest
    if (lane == 0)
      for (int j = issued; j < n_pre; ++j)
        tc::bulk_load_1d(stage_addr(j) + L.q_bytes + 2 * L.kv_bytes, p.rope, L.rope_bytes, bar_full + 8 * j);
    __syncwarp();
    issued = max(issued, n_pre);
    if (!ok_all && lane == 0) {
      flag_error(p.d_error, PKV_DEVERR_TIMEOUT);
      s_abort = 1;
    }
    // the last copies issued have landed before the CTA may wind down (whether or not the
    // consumers got to them): no bulk copy is ever in flight into a finished CTA's memory
    for (int j = (issued > S ? issued - S : 0); j < issued; ++j)
      tc::mbar_wait(bar_full + 8 * (j % S), (j / S) & 1, 200000000LL);
  } else {
    // ======================= consumers =======================
    // Thread tid takes tasks tid, tid + 32 W, ... of every token: 16 elements of one head (two
    // groups of 8, A and B, placed by the rope style).  The heads of a token are consecutive
    // tasks, so the lanes of one head are D/16 consecutive lanes of a warp (D/16 divides 32) --
    // the norm reduces over them.
    const int D = p.D, per_head = D >> 4;
    const int tasks_per_token = (p.Hq + 2 * p.Hkv) * per_head;
    const int stride = 32 * W;
    const int rounds = (tasks_per_token + stride - 1) / stride;
    const size_t esz = KVK != 0 ? 1 : 2;
    const TaskDesc d0 = describe_task(tid, tasks_per_token, p, L);
    const TaskDesc d1 = describe_task(tid + stride, tasks_per_token, p, L);
    const size_t kv_page_elems = static_cast<size_t>(p.B) * p.Hkv * D;  // K -> V of a page
    for (int j = 0; j < n_local; ++j) {
      const int st = j % S;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(bar_full + 8 * st, (j / S) & 1))) {
        if (lane == 0) {
          flag_error(p.d_error, PKV_DEVERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      const int4 m = s_meta[j & (kMetaRing - 1)];
      const uint8_t* stage = smem + L.stage_off + st * L.stage_bytes;
      const int64_t token = m.w;
      // the slot's K row in the pool (V is one page half further)
      const size_t slot_elem = (static_cast<size_t>(m.y) * 2 * p.B + m.z) * p.Hkv * D;
      if (m.x >= 0) {
        for (int rr = 0; rr < rounds; ++rr) {  // warp-uniform: inactive lanes join the norm shuffles
          const TaskDesc d = rr == 0 ? d0 : rr == 1 ? d1 : describe_task(tid + rr * stride, tasks_per_token, p, L);
          const bool active = d.kind >= 0;
          const U16x8 a8 = *reinterpret_cast<const U16x8*>(stage + d.src_a);
          const U16x8 b8 = *reinterpret_cast<const U16x8*>(stage + d.src_b);
          float xa[8], xb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            xa[e] = bf16_bits_to_f32(a8.v[e]);
            xb[e] = bf16_bits_to_f32(b8.v[e]);
          }
          // ---- optional RMSNorm of q / k heads (uniform per warp group of D/16 lanes) ----
          const float* nw = d.kind == 0 ? p.q_norm_w : d.kind == 1 ? p.k_norm_w : nullptr;
          if (__any_sync(0xffffffffu, nw != nullptr)) {  // every lane shuffles; xor stays inside a head
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = __fmaf_rn(xa[e], xa[e], __fmaf_rn(xb[e], xb[e], ss));
            for (int mm = 1; mm < per_head; mm <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, mm);
            if (nw != nullptr) {
              const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), p.norm_eps)));
              const int offA = d.off & 0xFFFF, offB = d.off >> 16;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                xa[e] = __fmul_rn(__fmul_rn(xa[e], inv), __ldg(nw + offA + e));
                xb[e] = __fmul_rn(__fmul_rn(xb[e], inv), __ldg(nw + offB + e));
              }
            }
          }
          if (!active) continue;
          // ---- rotation: the fixed fp32 recipe y_a = fma(a, c, -(b*s)), y_b = fma(b, c, a*s) ----
          float ya[8], yb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            ya[e] = xa[e];
            yb[e] = xb[e];
          }
          if (d.cs >= 0) {
            const float4* cs4 = reinterpret_cast<const float4*>(stage + d.cs);
            float c[8], sn[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 f = cs4[e];
              c[2 * e] = f.x;
              sn[2 * e] = f.y;
              c[2 * e + 1] = f.z;
              sn[2 * e + 1] = f.w;
            }
            if (p.style == 0) {  // rotate-half pairs (xa[e], xb[e]), pair index 8t + e
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                ya[e] = __fmaf_rn(xa[e], c[e], -__fmul_rn(xb[e], sn[e]));
                yb[e] = __fmaf_rn(xb[e], c[e], __fmul_rn(xa[e], sn[e]));
              }
            } else {  // interleaved pairs (xa[2e], xa[2e+1]) then (xb[2e], xb[2e+1])
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                ya[2 * e] = __fmaf_rn(xa[2 * e], c[e], -__fmul_rn(xa[2 * e + 1], sn[e]));
                ya[2 * e + 1] = __fmaf_rn(xa[2 * e + 1], c[e], __fmul_rn(xa[2 * e], sn[e]));
                yb[2 * e] = __fmaf_rn(xb[2 * e], c[4 + e], -__fmul_rn(xb[2 * e + 1], sn[4 + e]));
                yb[2 * e + 1] = __fmaf_rn(xb[2 * e + 1], c[4 + e], __fmul_rn(xb[2 * e], sn[4 + e]));
              }
            }
          }
          if (d.kind == 0) {
            uint16_t* dst = p.q_out + token * p.q_out_stride;
            *reinterpret_cast<U16x8*>(dst + d.dst_a) = to_bf16x8(ya);
            *reinterpret_cast<U16x8*>(dst + d.dst_b) = to_bf16x8(yb);
            continue;
          }
          if (m.y < 0) continue;  // bad page: flagged once by the producer
          uint8_t* dst = static_cast<uint8_t*>(p.pool) + (slot_elem + (d.kind == 2 ? kv_page_elems : 0)) * esz;
          if constexpr (KVK == 2) {
            *reinterpret_cast<uint2*>(dst + d.dst_a) = to_int8x8(ya, p.inv_scale);
            *reinterpret_cast<uint2*>(dst + d.dst_b) = to_int8x8(yb, p.inv_scale);
          } else if constexpr (KVK == 1) {
            *reinterpret_cast<uint2*>(dst + d.dst_a) = to_e4m3x8(ya, p.inv_scale);
            *reinterpret_cast<uint2*>(dst + d.dst_b) = to_e4m3x8(yb, p.inv_scale);
          } else if (d.kind == 2) {  // V is stored as given
            *reinterpret_cast<U16x8*>(dst + 2 * d.dst_a) = a8;
            *reinterpret_cast<U16x8*>(dst + 2 * d.dst_b) = b8;
          } else {
            *reinterpret_cast<U16x8*>(dst + 2 * d.dst_a) = to_bf16x8(ya);
            *reinterpret_cast<U16x8*>(dst + 2 * d.dst_b) = to_bf16x8(yb);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar_empty + 8 * st);  // this warp is done with the stage
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int32_t*>(&s_abort) != 0)) break;
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int kv_dtype, cudaStream_t s) {
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 152;
  }
  AppendParams q = p;
  // one consumer thread per task of a token, up to 12 warps (wider models loop over rounds)
  const int tasks_per_token = (p.Hq + 2 * p.Hkv) * (p.D / 16);
  q.consumer_warps = std::max(1, std::min(kMaxConsumerWarps, (tasks_per_token + 31) / 32));
  // ring depth: up to eight stages, as many as fit two CTAs per SM (the q row of very wide
  // models may leave room for fewer)
  const AppendSmem one = append_smem(p.R, p.Hq, p.Hkv, p.D, p.rot, 1);
  const int budget = 112 * 1024;  // per CTA, two CTAs per SM
  int stages = static_cast<int>(std::min<int64_t>(kMaxStages, (budget - one.stage_off) / one.stage_bytes));
  if (stages < 2) stages = 2;
  q.stages = stages;
  const AppendSmem L = append_smem(p.R, p.Hq, p.Hkv, p.D, p.rot, stages);
  if (L.bytes > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = kv_dtype == PKV_FP8_E4M3 ? append_rope_kernel<1>
              : kv_dtype == PKV_INT8   ? append_rope_kernel<2>
                                       : append_rope_kernel<0>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.bytes);
  if (e != cudaSuccess) return e;
  // persistent CTAs (two per SM), each streaming every (grid)-th token
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(p.T, 2LL * num_sms));
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3((q.consumer_warps + 1) * 32), L.bytes, s, q);
}

}  // namespace pkv
