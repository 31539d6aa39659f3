// common.cuh -- device helpers shared by the library's kernels (sm_103a only).
//
// Thin wrappers over PTX that the CUDA C++ front end does not expose directly: cp.async with
// zero-fill, ldmatrix, movmatrix, warp-level mma.sync, plus error-word helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "internal.h"

namespace pkv {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: every kernel of the library is launched so that it may start
// while the previous kernel on the stream drains; it must wait here before touching memory that
// earlier work produces.  A no-op when launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets the next kernel on the stream (launched with programmatic serialisation) start before this
// one ends; every such kernel here still runs griddepcontrol.wait before it reads what the
// kernels before it wrote.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void flag_error(int32_t* d_error, uint32_t bits) {
  if (d_error) atomicOr(reinterpret_cast<unsigned int*>(d_error), bits);
}

// 16-byte global -> shared copy; src_bytes == 0 zero-fills the destination without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Transpose an 8x8 matrix of 16-bit elements held one row pair per lane (fragment layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// D(16x8, fp32) += A(16x16) * B(16x8), A row-major, B column-major fragments.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8, fp32) += A(16x32) * B(32x8), E4M3 operands (4 codes per register).
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 -> two E4M3 codes (RNE, saturating), x.x in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// x ~= hi + lo with hi = e4m3(x) and lo = e4m3(x - hi) (two codes per output, low byte first):
// about 8 significant bits between them, so a pair of E4M3 MMAs reproduces a bf16 operand.
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t& hi2, uint32_t& lo2) {
  hi2 = f32x2_to_e4m3x2(x0, x1);
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(hi2), __NV_E4M3);
  const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&h));
  lo2 = f32x2_to_e4m3x2(x0 - hv.x, x1 - hv.y);
}

// The same split for 0 <= x <= 448 without a round trip through E4M3: hi is x cut to three
// mantissa bits (an E4M3 value from 2^-6 up, converted exactly) and lo = e4m3(x - hi); together
// about seven significant bits (below 2^-6 hi rounds to E4M3's 2^-9 steps, an absolute error
// under 2^-10).
__device__ __forceinline__ void split_cut_e4m3x2(float x0, float x1, uint32_t& hi2, uint32_t& lo2) {
  const float h0 = __uint_as_float(__float_as_uint(x0) & 0xFFF00000u);
  const float h1 = __uint_as_float(__float_as_uint(x1) & 0xFFF00000u);
  hi2 = f32x2_to_e4m3x2(h0, h1);
  lo2 = f32x2_to_e4m3x2(x0 - h0, x1 - h1);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two E4M3 codes (low byte first) -> f16x2, exact (every E4M3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Four int8 codes (byte j = code j) -> two f16x2 with lo = (code0, code1), hi = (code2, code3),
// each value 1152 + code exactly: with the sign bit flipped a byte reads u = code + 128, and the
// f16 pattern 0x64:u is 1024 + u (f16 values are spaced exactly 1 apart in [1024, 2048)).
__device__ __forceinline__ void i8x4_to_f16x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}
// The same with the bias removed: lo, hi hold the codes themselves (exact in f16).
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  i8x4_to_f16x2_biased(w, lo, hi);
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
  __half2 l = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
  __half2 h = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
  lo = *reinterpret_cast<uint32_t*>(&l);
  hi = *reinterpret_cast<uint32_t*>(&h);
}
constexpr float kI8Bias = 1152.f;

// Four E4M3 codes (byte j = code j) -> two exact f16x2, lo = (code0, code1), hi = (code2, code3).
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w));
  hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// 2^x with the MUFU instruction alone (flush-to-zero; relative error ~2^-22, and results below
// 2^-126 -- probabilities of masked or vanishing keys -- become 0).  -inf gives 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Blackwell packed / three-operand fp32 instructions (one issue slot for two lanes of work).
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {  // a * b + c, per lane
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float warp_max_xor(float v, int mask) {
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, mask));
}

}  // namespace pkv
