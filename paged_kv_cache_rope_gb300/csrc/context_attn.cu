// context_attn.cu -- causal context / chunked-context attention over the paged pool on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM, operands fed by TMA).
//
// Pages: "TensorRT-LLM 1.0 源码学习笔记", 6.1 "两者分工" (input length > 1 takes the flash-
// attention path, fused with the paged KV cache) and 6.2 "Flash Attention算法核心" (outer loop
// over Q tiles, inner loop over KV tiles; GEMM1 S = Q K^T, online max / sum, GEMM2 O += P V with
// the running rescale); adg.csdn.net/69730cc6 section 1.3 (chunked context: a chunk attends to
// the cached prefix plus itself); "TensorRT-LLM框架概述" section 2.2.1 (flash attention cuts HBM
// traffic).
//
// The pages' kernel keeps S and O in registers of warp-level MMA fragments.  On sm_103a the
// contraction runs on tcgen05 with both accumulators in TMEM instead:
//   CTA = (query head, 128-row query tile of one context request), 6 warps:
//     warps 0-3  softmax: thread i owns row i (TMEM lane i) -- reads S from TMEM, masks,
//                online max / sum in base 2 (O is rescaled in TMEM only when the running max
//                grows by more than 2^8), writes P (bf16) to shared memory, final O / l;
//     warp 4     TMA producer: Q once, then per 128-key tile the pool pages of K and V through
//                the block table (one box per page and 64-wide head-dim half);
//     warp 5     TMEM owner and MMA issuer: S_j = Q K_j^T into one of two TMEM S buffers, then
//                O += P_{j-1} V_{j-1}; completion is signalled with tcgen05.commit on mbarriers.
//   TMEM: S0 | S1 | O  (128 + 128 + D columns of 128 lanes, 512 allocated).
//   Shared memory (128-byte swizzle, K-major Q/K/P, MN-major V): Q, K[2], V[2], P[2].
// Rows past the request's end and keys past the causal limit are masked by select (never by
// arithmetic on the loaded values); V rows past the sequence end are zeroed before PV, so
// stale or poisoned pool slots cannot reach the output.  Every wait is bounded.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kSoftmaxWarps = 4;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O once P could exceed 2^8

template <int D>
struct CtxSmem {
  static constexpr int kHalf = 128 * 128;                    // one 64-wide half of a 128-row tile
  static constexpr int kQ = (D / 64) * kHalf;                 // Q tile
  static constexpr int kKV = (D / 64) * kHalf;                // one K or V stage
  static constexpr int kP = 2 * kHalf;                        // P tile (128 keys)
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQ;
  static constexpr int kVOff = kKOff + 2 * kKV;
  static constexpr int kPOff = kVOff + 2 * kKV;
  static constexpr int kBarOff = kPOff + 2 * kP;
  static constexpr int kBarBytes = 256;
  static constexpr int kBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
};

// barrier indices
enum {
  BAR_Q = 0,
  BAR_KFULL = 1,   // +2
  BAR_KEMPTY = 3,  // +2
  BAR_VFULL = 5,   // +2
  BAR_VEMPTY = 7,  // +2
  BAR_SFULL = 9,   // +2
  BAR_SFREE = 11,  // +2
  BAR_PFULL = 13,  // +2
  BAR_PFREE = 15,  // +2
  BAR_MMADONE = 17,
  NUM_BARS = 18
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
context_attn_kernel(const ContextParams p, const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap kv_map) {
  using L = CtxSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  const uint32_t bar0 = base_s + L::kBarOff;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L::kBarOff + 8 * NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kBarOff + 8 * NUM_BARS + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.x;
  const int hk = hq / p.group;

  // ---- which context request / query tile (heaviest tiles first) ----
  const int tile = p.num_tiles - 1 - static_cast<int>(blockIdx.y);
  int lo = 0, hi = p.C - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.tile_prefix + mid) <= tile) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int i0 = (tile - __ldg(p.tile_prefix + r)) * kCtxTileM;
  const int n_r = __ldg(p.ctx_len + r);
  const int past = __ldg(p.past + r);
  const int n_valid = min(kCtxTileM, n_r - i0);
  const int row0 = __ldg(p.cu_q + r) + i0;
  const int L_r = past + n_r;
  if (n_valid <= 0 || tile < 0) {  // plan disagrees with the launch
    if (threadIdx.x == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);
    return;
  }
  const int kv_len = past + i0 + n_valid;  // keys visible to the last valid row
  const int n_kv_tiles = (kv_len + kCtxTileN - 1) / kCtxTileN;

  const uint32_t sQ = base_s + L::kQOff;
  auto sK = [&](int st) { return base_s + L::kKOff + st * L::kKV; };
  auto sV = [&](int st) { return base_s + L::kVOff + st * L::kKV; };
  auto sP = [&](int st) { return base_s + L::kPOff + st * L::kP; };

  // ---- set-up: barriers, TMEM ----
  if (threadIdx.x == 0) {
    tc::mbar_init(bar(BAR_Q), 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(BAR_KFULL + s), 1);
      tc::mbar_init(bar(BAR_KEMPTY + s), 1);
      tc::mbar_init(bar(BAR_VFULL + s), 1);
      tc::mbar_init(bar(BAR_VEMPTY + s), 1);
      tc::mbar_init(bar(BAR_SFULL + s), 1);
      tc::mbar_init(bar(BAR_SFREE + s), kSoftmaxWarps * 32);
      tc::mbar_init(bar(BAR_PFULL + s), kSoftmaxWarps * 32);
      tc::mbar_init(bar(BAR_PFREE + s), 1);
    }
    tc::mbar_init(bar(BAR_MMADONE), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(base_s + L::kBarOff + 8 * NUM_BARS, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tc::prefetch_tmap(&q_map);
    tc::prefetch_tmap(&kv_map);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  auto fail = [&]() {
    flag_error(p.d_error, PKV_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };
  // Softmax warps execute tcgen05.ld/st (.sync.aligned): every branch around them must be
  // uniform across the warp, so waits and the abort flag are voted on.
  auto warp_wait = [&](uint32_t b, uint32_t parity) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b, parity)) != 0;
  };
  auto warp_abort = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0) != 0; };

  if (warp == kProducerWarp) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      const int32_t* tbl = p.tbl + static_cast<int64_t>(r) * p.max_blocks;
      const int box_rows = p.B < kCtxTileN ? p.B : kCtxTileN;
      const int pages_per_tile = kCtxTileN / box_rows;
      const int n_pages_seq = (L_r + p.B - 1) / p.B;
      tc::mbar_arrive_expect_tx(bar(BAR_Q), kCtxTileM * D * 2);
      for (int dh = 0; dh < D / 64; ++dh)
        tc::tma_load_4d(sQ + dh * L::kHalf, &q_map, bar(BAR_Q), 0, dh, hq, row0);
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_kv_tiles && !*abort_flag; ++j) {
        const int st = j & 1;
        // pages of this tile that exist in the sequence and have a valid id
        int pages[kCtxTileN / 16];
        int n_ok = 0;
        for (int pp = 0; pp < pages_per_tile; ++pp) {
          const int lb = (j * kCtxTileN) / p.B + pp;  // B <= 128: whole pages per tile
          int pg = -1;
          if (lb < n_pages_seq && lb < p.max_blocks) {
            pg = __ldg(tbl + lb);
            if (pg < 0 || pg >= p.NB) {
              flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
              pg = -1;
            }
          }
          pages[pp] = pg;
          n_ok += pg >= 0;
        }
        const uint32_t bytes = static_cast<uint32_t>(n_ok) * box_rows * D * 2;
        if (j >= 2 && !tc::mbar_wait(bar(BAR_KEMPTY + st), ((j - 2) >> 1) & 1)) { fail(); break; }
        tc::mbar_arrive_expect_tx(bar(BAR_KFULL + st), bytes);
        for (int pp = 0; pp < pages_per_tile; ++pp) {
          if (pages[pp] < 0) continue;
          const int row = (pages[pp] * 2 + 0) * p.B;
          for (int dh = 0; dh < D / 64; ++dh)
            tc::tma_load_4d(sK(st) + dh * L::kHalf + pp * box_rows * 128, &kv_map, bar(BAR_KFULL + st), 0, dh, hk,
                            row);
        }
        ++issued_k;
        if (j >= 2 && !tc::mbar_wait(bar(BAR_VEMPTY + st), ((j - 2) >> 1) & 1)) { fail(); break; }
        tc::mbar_arrive_expect_tx(bar(BAR_VFULL + st), bytes);
        for (int pp = 0; pp < pages_per_tile; ++pp) {
          if (pages[pp] < 0) continue;
          const int row = (pages[pp] * 2 + 1) * p.B;
          for (int dh = 0; dh < D / 64; ++dh)
            tc::tma_load_4d(sV(st) + dh * L::kHalf + pp * box_rows * 128, &kv_map, bar(BAR_VFULL + st), 0, dh, hk,
                            row);
        }
        ++issued_v;
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA winds down
        for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j)
          tc::mbar_wait(bar(BAR_KFULL + (j & 1)), (j >> 1) & 1, 200000000LL);
        for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j)
          tc::mbar_wait(bar(BAR_VFULL + (j & 1)), (j >> 1) & 1, 200000000LL);
        tc::mbar_wait(bar(BAR_Q), 0, 200000000LL);
      }
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(128, kCtxTileN, 0);
      constexpr uint32_t idesc_o = tc::idesc_bf16(128, D, 1);
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj & 1;
        if (!tc::mbar_wait(bar(BAR_PFULL + st), (jj >> 1) & 1)) return false;
        if (!tc::mbar_wait(bar(BAR_VFULL + st), (jj >> 1) & 1)) return false;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kCtxTileN / 16; ++kk) {
          const uint64_t a = tc::sdesc_sw128(sP(st) + (kk >> 2) * L::kHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t b = tc::sdesc_sw128(sV(st) + kk * 16 * 128, L::kHalf, 1024);
          tc::mma_bf16_ss(tO, a, b, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar(BAR_PFREE + st));
        tc::mma_commit(bar(BAR_VEMPTY + st));
        return true;
      };
      bool ok = tc::mbar_wait(bar(BAR_Q), 0);
      for (int j = 0; ok && j < n_kv_tiles && !*abort_flag; ++j) {
        const int st = j & 1;
        if (!tc::mbar_wait(bar(BAR_KFULL + st), (j >> 1) & 1)) { ok = false; break; }
        if (j >= 2 && !tc::mbar_wait(bar(BAR_SFREE + st), ((j - 2) >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = tc::sdesc_sw128(sQ + (kk >> 2) * L::kHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t b = tc::sdesc_sw128(sK(st) + (kk >> 2) * L::kHalf + (kk & 3) * 32, 16, 1024);
          tc::mma_bf16_ss(tS0 + st * kCtxTileN, a, b, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(BAR_SFULL + st));
        tc::mma_commit(bar(BAR_KEMPTY + st));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !*abort_flag) ok = issue_pv(n_kv_tiles - 1);
      if (!ok) fail();
      tc::mma_commit(bar(BAR_MMADONE));
      tc::mbar_wait(bar(BAR_MMADONE), 0, 200000000LL);  // nothing of ours still runs on TMEM
    }
  } else {
    // ======================= softmax warps =======================
    const int row = warp * 32 + lane;                   // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int q_pos = past + i0 + min(row, n_valid - 1);  // padding rows mirror the last row
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv_tiles; ++j) {
      const int st = j & 1;
      if (warp_abort() || !warp_wait(bar(BAR_SFULL + st), (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t tS = tS0 + st * kCtxTileN + lane_off;
      const int lim = q_pos - j * kCtxTileN;  // key column c is visible iff c <= lim
      // pass 1: row max of the visible, scaled scores
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < kCtxTileN / 32; ++cc) {
        uint32_t v[32];
        tc::tmem_ld32(tS + cc * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float s = __uint_as_float(v[e]) * sl2;
          mx = (cc * 32 + e <= lim) ? fmaxf(mx, s) : mx;
        }
      }
      const float m_new = fmaxf(m_run, mx);
      float m_use = m_run;
      if (j == 0) {
        m_use = m_new;  // first tile: O is still empty
      } else if (__any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold)) {
        // the whole warp rescales (lanes below the threshold too, each to its own new max);
        // O must hold every earlier P V before it is rescaled
        if (!warp_wait(bar(BAR_PFREE + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const float f = exp2f(m_run - m_new);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t v[32];
          tc::tmem_ld32(tO + lane_off + cc * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
          tc::tmem_st32(tO + lane_off + cc * 32, v);
        }
        tc::tmem_wait_st();
        l_run *= f;
        m_use = m_new;
      }
      m_run = m_use;
      // P buffer `st` is free once P_{j-2} V_{j-2} has completed
      if (j >= 2 && !warp_wait(bar(BAR_PFREE + st), ((j - 2) >> 1) & 1)) { ok = false; break; }
      // pass 2: P = exp2(s - m) for visible keys, 0 otherwise; bf16 into the swizzled P tile
      uint8_t* prow = base + (sP(st) - base_s) + row * 128;
#pragma unroll
      for (int cc = 0; cc < kCtxTileN / 32; ++cc) {
        uint32_t v[32];
        tc::tmem_ld32(tS + cc * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c = cc * 32 + e;
          const float p0 = (c <= lim) ? exp2f(__uint_as_float(v[e]) * sl2 - m_use) : 0.f;
          const float p1 = (c + 1 <= lim) ? exp2f(__uint_as_float(v[e + 1]) * sl2 - m_use) : 0.f;
          l_run += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        // 32 keys = 4 chunks of 16 bytes in key-half (cc >> 1), chunks (cc & 1) * 4 .. +3
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (cc & 1) * 4 + k;
          uint4* dst = reinterpret_cast<uint4*>(prow + (cc >> 1) * L::kHalf + ((chunk ^ (row & 7)) << 4));
          *dst = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(bar(BAR_SFREE + st));
      if (j == n_kv_tiles - 1) {
        // zero V rows past the end of the sequence (stale or unloaded slots)
        if (!warp_wait(bar(BAR_VFULL + st), (j >> 1) & 1)) { ok = false; break; }
        if (j * kCtxTileN + row >= L_r) {
          uint8_t* vrow = base + (sV(st) - base_s) + row * 128;
#pragma unroll
          for (int dh = 0; dh < D / 64; ++dh)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              reinterpret_cast<uint4*>(vrow + dh * L::kHalf)[k] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar(BAR_PFULL + st));
    }
    if (!ok) fail();
    // ---- epilogue: O / l -> bf16 rows ----
    const int jl = n_kv_tiles - 1;
    if (ok && !warp_abort() && warp_wait(bar(BAR_PFREE + (jl & 1)), (jl >> 1) & 1)) {
      tc::fence_after_sync();
      const float inv_l = 1.f / l_run;
      uint16_t* orow = p.out + static_cast<int64_t>(row0 + row) * p.out_stride + static_cast<int64_t>(hq) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tc::tmem_ld32(tO + lane_off + cc * 32, v);
        if (row < n_valid && row0 + row < p.T) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pk[e >> 1] = pack_bf16x2(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            reinterpret_cast<uint4*>(orow + cc * 32)[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
    } else if (ok) {
      fail();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_context(const ContextParams& p, const void* q_map, const void* kv_map, bool fp8,
                           cudaStream_t s) {
  if (fp8) return cudaErrorNotSupported;
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(kv_map);
  dim3 grid(p.Hq, p.num_tiles);
  cudaError_t e;
  if (p.D == 128) {
    e = cudaFuncSetAttribute(context_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, CtxSmem<128>::kBytes);
    if (e != cudaSuccess) return e;
    context_attn_kernel<128><<<grid, kThreads, CtxSmem<128>::kBytes, s>>>(p, qm, km);
  } else {
    e = cudaFuncSetAttribute(context_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, CtxSmem<64>::kBytes);
    if (e != cudaSuccess) return e;
    context_attn_kernel<64><<<grid, kThreads, CtxSmem<64>::kBytes, s>>>(p, qm, km);
  }
  return cudaGetLastError();
}

}  // namespace pkv
