// append_rope.cu -- GPT-NeoX RoPE on Q and K plus the append of K/V into the paged pool.
//
// Pages: "TensorRT-LLM 1.0 源码学习笔记", 二.2 "KVCacheManager 详解" (the attention op writes
// each new token's KV into the blocks named by the block table) and 6.4 "量化" (quantise on
// write with kv_scale_orig_quant); adg.csdn.net/69730cc6 section 1.1 (GPT-NeoX rotary
// embedding); "TensorRT-LLM 源码完全拆解(一)", "KVCacheManager 的三个对外接口" (pool layout
// [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]).
//
// HBM-bound.  One thread handles 16 elements of one head of one token (8 rotation pairs, or a
// pass-through part of a partially rotated head): two 16-byte loads, two 16-byte stores (8-byte
// stores into an FP8 or INT8 pool).  (A warp-per-token layout with the rotation coefficients
// loaded once per token measured no faster.)  Variants: rotate-half or interleaved pairs, partial rotary dims,
// an optional RMSNorm of q / k heads reduced across the head's lanes with shuffles, and
// draft tokens rotated for past + offset (adg.csdn.net/69730cc6 section 1.4,
// spec_decoding_position_offsets) while stored at slot past + i.
// Threads of a warp cover consecutive heads of the same token, so every row read and written
// is a run of full 32-byte sectors.  The token -> request map comes from an in-CTA prefix scan
// of context_lengths (no workspace needed).
#include "common.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

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

// Rotate 8 rotate-half pairs (lo[e], hi[e]) with the fixed fp32 recipe:
// y_lo = fma(lo, c, -(hi*s)), y_hi = fma(hi, c, lo*s).
__device__ __forceinline__ void rotate8(const float (&lo)[8], const float (&hi)[8], const float2* cs,
                                        float (&ylo)[8], float (&yhi)[8]) {
  const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float4 t = __ldg(cs4 + e);
    const float c0 = t.x, s0 = t.y, c1 = t.z, s1 = t.w;
    const float a0 = lo[2 * e], b0 = hi[2 * e], a1 = lo[2 * e + 1], b1 = hi[2 * e + 1];
    ylo[2 * e] = __fmaf_rn(a0, c0, -__fmul_rn(b0, s0));
    yhi[2 * e] = __fmaf_rn(b0, c0, __fmul_rn(a0, s0));
    ylo[2 * e + 1] = __fmaf_rn(a1, c1, -__fmul_rn(b1, s1));
    yhi[2 * e + 1] = __fmaf_rn(b1, c1, __fmul_rn(a1, s1));
  }
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

template <int KVK>  // pool element kind: 0 bf16, 1 E4M3 codes, 2 int8 codes
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(AppendParams p) {
  extern __shared__ int32_t s_cu[];  // [R + 1] exclusive prefix of context_lengths
  // ---- block-wide exclusive scan of context_lengths (chunks of blockDim.x) ----
  __shared__ int32_t s_warp[kAppendThreads / 32];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_wait();
  if (tid == 0) s_carry = 0;
  __syncthreads();
  bool neg = false;
  for (int base = 0; base < p.R; base += kAppendThreads) {
    int r = base + tid;
    int x = r < p.R ? __ldg(p.ctx_len + r) : 0;
    neg |= x < 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int w = lane < kAppendThreads / 32 ? s_warp[lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < kAppendThreads / 32) s_warp[lane] = wi - w;  // exclusive warp offsets
    }
    __syncthreads();
    int carry = s_carry;
    if (r < p.R) s_cu[r] = carry + s_warp[wid] + incl - x;
    __syncthreads();
    if (tid == kAppendThreads - 1) s_carry = carry + s_warp[wid] + incl;
    __syncthreads();
  }
  if (tid == 0) s_cu[p.R] = s_carry;
  // Without a bucket the device lengths must add up to the host's token count; in a bucket
  // (p.T = the rows' capacity) the batch may use fewer rows, never more, and empty slots
  // (no new tokens) own no row
  const bool bad = __syncthreads_or(neg) != 0 || (p.dyn ? s_cu[p.R] > p.T : s_cu[p.R] != p.T);
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) flag_error(p.d_error, p.dyn ? PKV_DEVERR_BUCKET : PKV_DEVERR_PLAN_MISMATCH);
    return;
  }
  const int T = s_cu[p.R];          // packed rows of this batch
  const int gen_row0 = s_cu[p.C];   // first row of the generation requests

  // Each lane handles 16 elements of one head of one token: two groups of 8 (A and B) whose
  // place depends on the rope style; heads of a token are consecutive tasks, so the lanes of one
  // head are D/16 consecutive lanes of a warp (D/16 divides 32) -- the norm reduces over them.
  const int D = p.D, per_head = D >> 4;
  const int rot_tasks = p.rot >> 4, rhalf = p.rot >> 1;
  const int tasks_per_token = (p.Hq + 2 * p.Hkv) * per_head;
  const int total = T * tasks_per_token;  // < 2^31, checked on the host
  const int lph = 31 - __clz(per_head);      // per_head is 4 or 8
  const size_t esz = KVK != 0 ? 1 : 2;
  const int stride = gridDim.x * kAppendThreads;
  for (int wbase = blockIdx.x * kAppendThreads + (tid & ~31); wbase < total;
       wbase += stride) {  // warp-uniform loop: inactive lanes still join the norm shuffles
    const int gi = wbase + lane;
    const bool active = gi < total;
    const int token = active ? gi / tasks_per_token : 0;
    int task = active ? gi - token * tasks_per_token : 0;
    int lo = 0, hi = p.R - 1;  // request of this token: largest r with s_cu[r] <= token
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (s_cu[mid] <= token) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo;
    const int past_r = __ldg(p.past + r);
    const int pos = past_r + (token - s_cu[r]);  // slot position
    int rpos = pos;                               // rotation position
    bool ok = active;
    if (active && p.pos_off != nullptr && token >= gen_row0) {  // a draft token
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
    // kind: 0 = q, 1 = k, 2 = v; head h; task t within the head
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
    const bool rotate = kind != 2 && t < rot_tasks;
    int offA, offB;  // element offsets of the two 8-element groups inside the head
    if (p.style == 0 && t < rot_tasks) {
      offA = 8 * t;
      offB = rhalf + 8 * t;
    } else {
      const int base = (p.style == 0) ? p.rot + 16 * (t - rot_tasks) : 16 * t;
      offA = base;
      offB = base + 8;
    }
    const uint16_t* src = (kind == 0 ? p.q + token * p.q_stride : kind == 1 ? p.k + token * p.k_stride
                                                                          : p.v + token * p.v_stride) +
                          h * D;
    U16x8 a8 = {}, b8 = {};
    if (ok) {
      a8 = *reinterpret_cast<const U16x8*>(src + offA);
      b8 = *reinterpret_cast<const U16x8*>(src + offB);
    }
    float xa[8], xb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      xa[e] = bf16_bits_to_f32(a8.v[e]);
      xb[e] = bf16_bits_to_f32(b8.v[e]);
    }
    // ---- optional RMSNorm of q / k heads (uniform per warp group of D/16 lanes) ----
    const float* nw = kind == 0 ? p.q_norm_w : kind == 1 ? p.k_norm_w : nullptr;
    if (__any_sync(0xffffffffu, nw != nullptr)) {  // every lane shuffles; xor stays inside a head
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = __fmaf_rn(xa[e], xa[e], __fmaf_rn(xb[e], xb[e], ss));
      for (int m = 1; m < per_head; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      if (nw != nullptr) {
        const float inv = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(D)), p.norm_eps)));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xa[e] = __fmul_rn(__fmul_rn(xa[e], inv), __ldg(nw + offA + e));
          xb[e] = __fmul_rn(__fmul_rn(xb[e], inv), __ldg(nw + offB + e));
        }
      }
    }
    if (!ok) continue;
    // ---- rotation: the fixed fp32 recipe y_a = fma(a, c, -(b*s)), y_b = fma(b, c, a*s) ----
    float ya[8], yb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ya[e] = xa[e];
      yb[e] = xb[e];
    }
    if (rotate) {
      const float2* cs = p.rope + static_cast<size_t>(rpos) * rhalf + 8 * t;
      if (p.style == 0) {
        rotate8(xa, xb, cs, ya, yb);
      } else {
        float c[8], sn[8];
        const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 f = __ldg(cs4 + e);
          c[2 * e] = f.x;
          sn[2 * e] = f.y;
          c[2 * e + 1] = f.z;
          sn[2 * e + 1] = f.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // pairs (xa[2e], xa[2e+1]) then (xb[2e], xb[2e+1])
          ya[2 * e] = __fmaf_rn(xa[2 * e], c[e], -__fmul_rn(xa[2 * e + 1], sn[e]));
          ya[2 * e + 1] = __fmaf_rn(xa[2 * e + 1], c[e], __fmul_rn(xa[2 * e], sn[e]));
          yb[2 * e] = __fmaf_rn(xb[2 * e], c[4 + e], -__fmul_rn(xb[2 * e + 1], sn[4 + e]));
          yb[2 * e + 1] = __fmaf_rn(xb[2 * e + 1], c[4 + e], __fmul_rn(xb[2 * e], sn[4 + e]));
        }
      }
    }
    if (kind == 0) {
      uint16_t* dst = p.q_out + token * p.q_out_stride + h * D;
      *reinterpret_cast<U16x8*>(dst + offA) = to_bf16x8(ya);
      *reinterpret_cast<U16x8*>(dst + offB) = to_bf16x8(yb);
      continue;
    }
    const int lb = pos >> (31 - __clz(p.B)), slot = pos & (p.B - 1);
    const int page = lb < p.max_blocks ? __ldg(p.tbl + static_cast<size_t>(r) * p.max_blocks + lb) : -1;
    if (page < 0 || page >= p.NB) {
      flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
      continue;
    }
    const int is_v = kind == 2;
    const size_t elem = ((static_cast<size_t>(page) * 2 + is_v) * p.B + slot) * p.Hkv * D + static_cast<size_t>(h) * D;
    uint8_t* dst = static_cast<uint8_t*>(p.pool) + elem * esz;
    if constexpr (KVK == 2) {
      *reinterpret_cast<uint2*>(dst + offA) = to_int8x8(ya, p.inv_scale);
      *reinterpret_cast<uint2*>(dst + offB) = to_int8x8(yb, p.inv_scale);
    } else if constexpr (KVK == 1) {
      *reinterpret_cast<uint2*>(dst + offA) = to_e4m3x8(ya, p.inv_scale);
      *reinterpret_cast<uint2*>(dst + offB) = to_e4m3x8(yb, p.inv_scale);
    } else if (is_v) {  // V is stored as given
      *reinterpret_cast<U16x8*>(dst + 2 * offA) = a8;
      *reinterpret_cast<U16x8*>(dst + 2 * offB) = b8;
    } else {
      *reinterpret_cast<U16x8*>(dst + 2 * offA) = to_bf16x8(ya);
      *reinterpret_cast<U16x8*>(dst + 2 * offB) = to_bf16x8(yb);
    }
  }
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
  const int64_t tasks = static_cast<int64_t>(p.T) * (p.Hq + 2 * p.Hkv) * (p.D / 16);
  if (tasks + kAppendThreads * 8LL * num_sms >= (int64_t(1) << 31)) return cudaErrorInvalidValue;  // int32 task index
  int64_t blocks = (tasks + kAppendThreads - 1) / kAppendThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // grid-stride beyond 8 CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t smem = sizeof(int32_t) * (p.R + 1);
  auto kern = kv_dtype == PKV_FP8_E4M3 ? append_rope_kernel<1>
              : kv_dtype == PKV_INT8   ? append_rope_kernel<2>
                                       : append_rope_kernel<0>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kAppendThreads), smem, s, p);
}

}  // namespace pkv
