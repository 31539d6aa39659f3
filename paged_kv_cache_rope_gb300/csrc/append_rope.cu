// append_rope.cu -- GPT-NeoX RoPE on Q and K plus the append of K/V into the paged pool.
//
// Pages: "TensorRT-LLM 1.0 源码学习笔记", 二.2 "KVCacheManager 详解" (the attention op writes
// each new token's KV into the blocks named by the block table) and 6.4 "量化" (quantise on
// write with kv_scale_orig_quant); adg.csdn.net/69730cc6 section 1.1 (GPT-NeoX rotary
// embedding); "TensorRT-LLM 源码完全拆解(一)", "KVCacheManager 的三个对外接口" (pool layout
// [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim]).
//
// HBM-bound.  One thread handles 8 rotation pairs (x_j .. x_{j+7}, x_{j+D/2} .. x_{j+D/2+7}) of
// one head of one token: two 16-byte loads, two 16-byte stores (8-byte stores into an FP8 pool).
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

// Rotate 8 pairs with the fixed fp32 recipe: y_lo = fma(lo, c, -(hi*s)), y_hi = fma(hi, c, lo*s).
__device__ __forceinline__ void rotate8(const U16x8& lo, const U16x8& hi, const float2* cs,
                                        float (&ylo)[8], float (&yhi)[8]) {
  const float4* cs4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float4 t = __ldg(cs4 + e);
    float c0 = t.x, s0 = t.y, c1 = t.z, s1 = t.w;
    float a0 = bf16_bits_to_f32(lo.v[2 * e]), b0 = bf16_bits_to_f32(hi.v[2 * e]);
    float a1 = bf16_bits_to_f32(lo.v[2 * e + 1]), b1 = bf16_bits_to_f32(hi.v[2 * e + 1]);
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

template <bool FP8>
__global__ void __launch_bounds__(kAppendThreads) append_rope_kernel(AppendParams p) {
  extern __shared__ int32_t s_cu[];  // [R + 1] exclusive prefix of context_lengths
  // ---- block-wide exclusive scan of context_lengths (chunks of blockDim.x) ----
  __shared__ int32_t s_warp[kAppendThreads / 32];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  pdl_wait();
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < p.R; base += kAppendThreads) {
    int r = base + tid;
    int x = r < p.R ? __ldg(p.ctx_len + r) : 0;
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
  __syncthreads();
  if (s_cu[p.R] != p.T) {  // device lengths disagree with the host's token count
    if (blockIdx.x == 0 && tid == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);
    return;
  }

  const int D = p.D, half = D >> 1, per_head = D >> 4;  // 8-pair tasks per head
  const int tasks_per_token = (p.Hq + 2 * p.Hkv) * per_head;
  const int64_t total = static_cast<int64_t>(p.T) * tasks_per_token;
  const size_t esz = FP8 ? 1 : 2;
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * kAppendThreads + tid; gi < total;
       gi += static_cast<int64_t>(gridDim.x) * kAppendThreads) {
    const int token = static_cast<int>(gi / tasks_per_token);
    int task = static_cast<int>(gi - static_cast<int64_t>(token) * tasks_per_token);
    // request of this token: largest r with s_cu[r] <= token
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (s_cu[mid] <= token) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo;
    const int pos = __ldg(p.past + r) + (token - s_cu[r]);
    if (pos < 0 || pos >= p.max_pos) {  // device lengths disagree with the host-checked ones
      flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);
      continue;
    }
    const float2* cs = p.rope + static_cast<size_t>(pos) * half;
    if (task < p.Hq * per_head) {  // ---- Q head: rotate, bf16 out ----
      const int h = task / per_head, j0 = (task - h * per_head) * 8;
      const uint16_t* src = p.q + token * p.q_stride + h * D;
      U16x8 lo8 = *reinterpret_cast<const U16x8*>(src + j0);
      U16x8 hi8 = *reinterpret_cast<const U16x8*>(src + half + j0);
      float ylo[8], yhi[8];
      rotate8(lo8, hi8, cs + j0, ylo, yhi);
      uint16_t* dst = p.q_out + token * p.q_out_stride + h * D;
      *reinterpret_cast<U16x8*>(dst + j0) = to_bf16x8(ylo);
      *reinterpret_cast<U16x8*>(dst + half + j0) = to_bf16x8(yhi);
      continue;
    }
    task -= p.Hq * per_head;
    const int is_v = task >= p.Hkv * per_head;
    if (is_v) task -= p.Hkv * per_head;
    const int h = task / per_head, j0 = (task - h * per_head) * 8;
    const int lb = pos / p.B, slot = pos - lb * p.B;
    const int page = lb < p.max_blocks ? __ldg(p.tbl + static_cast<size_t>(r) * p.max_blocks + lb) : -1;
    if (page < 0 || page >= p.NB) {
      flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
      continue;
    }
    const size_t elem = ((static_cast<size_t>(page) * 2 + is_v) * p.B + slot) * p.Hkv * D + static_cast<size_t>(h) * D;
    uint8_t* dst = static_cast<uint8_t*>(p.pool) + elem * esz;
    const uint16_t* src = (is_v ? p.v + token * p.v_stride : p.k + token * p.k_stride) + h * D;
    U16x8 lo8 = *reinterpret_cast<const U16x8*>(src + j0);
    U16x8 hi8 = *reinterpret_cast<const U16x8*>(src + half + j0);
    float ylo[8], yhi[8];
    if (!is_v) {
      rotate8(lo8, hi8, cs + j0, ylo, yhi);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ylo[e] = bf16_bits_to_f32(lo8.v[e]);
        yhi[e] = bf16_bits_to_f32(hi8.v[e]);
      }
    }
    if constexpr (FP8) {
      *reinterpret_cast<uint2*>(dst + j0) = to_e4m3x8(ylo, p.inv_scale);
      *reinterpret_cast<uint2*>(dst + half + j0) = to_e4m3x8(yhi, p.inv_scale);
    } else {
      if (is_v) {  // V is stored as given
        *reinterpret_cast<U16x8*>(dst + 2 * j0) = lo8;
        *reinterpret_cast<U16x8*>(dst + 2 * (half + j0)) = hi8;
      } else {
        *reinterpret_cast<U16x8*>(dst + 2 * j0) = to_bf16x8(ylo);
        *reinterpret_cast<U16x8*>(dst + 2 * (half + j0)) = to_bf16x8(yhi);
      }
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, bool fp8, cudaStream_t s) {
  static int num_sms = 0;
  if (num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (num_sms <= 0) num_sms = 152;
  }
  const int64_t tasks = static_cast<int64_t>(p.T) * (p.Hq + 2 * p.Hkv) * (p.D / 16);
  int64_t blocks = (tasks + kAppendThreads - 1) / kAppendThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // grid-stride beyond 8 CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t smem = sizeof(int32_t) * (p.R + 1);
  auto kern = fp8 ? append_rope_kernel<true> : append_rope_kernel<false>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(kAppendThreads), smem, s, p);
}

}  // namespace pkv
