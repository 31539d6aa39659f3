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
// contraction runs on tcgen05 with both accumulators in TMEM instead.
//
// context_attn_kernel: persistent, one CTA per SM at most.  Work item = (context unit of 256
// query rows, query head) = two 128-row Q tiles A and B that share every K/V tile and take turns
// on the tensor core.  A CTA claims items from a queue (longest unit first, as the plan sorted
// them) and keeps its TMEM, barriers and K/V ring across items.  12 warps (3 warpgroups, with
// setmaxnreg moving registers from the control warpgroup to the two softmax warpgroups):
//     warps 0-3 / 4-7  softmax of tile A / B: thread i owns row i (TMEM lane i).  It reads its
//                S row from TMEM in one pass (128 registers), masks by select, keeps the running
//                max / sum in base 2 (O is rescaled in TMEM only when the max grows by more than
//                2^8), and writes P as bf16 back into the first 64 columns of its own S buffer;
//     warp 8     item queue and TMA producer: per item Q once per tile, then per 128-key tile
//                the pool pages of K and V through the block table (lane i looks up and loads
//                page i: one box per page and 64-wide head-dim half); it claims the next item
//                as soon as it has issued the current one's last tile;
//     warp 9     TMEM owner and MMA issuer (warps 10-11 only complete the warpgroup), in the order
//                  S_A(0) S_B(0) | PV_A(0) S_A(1) PV_B(0) S_B(1) | PV_A(1) S_A(2) ...
//                so one tile's softmax overlaps the other tile's MMAs, and from the last PV of
//                one item straight on to the first S of the next.  PV takes P straight from TMEM
//                (A operand in tensor memory) and V from shared memory (MN-major).
//   Warps 8 and 9 share their sub-partitions with busy softmax warps and get few issue slots,
//   so they run converged, one elect.sync lane issues, and an 8-step MMA batch is a single
//   inline-asm statement over descriptors built once per operand tile: every instruction they
//   spend between MMA batches leaves the tensor pipe idle.
//   A full 128-row output tile leaves through a staging tile of its own (handed from epilogue to
//   epilogue in order) and two TMA stores, so no Q slot waits for an output store; per-thread
//   row stores would scatter each warp instruction over 32 rows.
//   TMEM columns: S_A | S_B | O_A | O_B (4 x 128 of 128 lanes).  tcgen05 work issued by one
//   thread completes in order, so a commit after S_X(j) also covers PV_X(j-1): the softmax of
//   tile j may rescale O_X as soon as S_X(j) has landed.
// 8-bit pools (E4M3 or int8 codes): stage_q8_kernel first copies the context requests' pages
// into a bf16 staging pool (exact code values) with its own block table; the context kernel then
// runs unchanged on it, with the pool scale folded into the score scale and into the output scale.
//
// gen_attn_kernel: generation requests with more (token, query head) pairs than the mma.sync
// decode kernel's columns, on the same tcgen05 pipeline; bf16 pools, or 8-bit pools at head_dim
// 128 whose codes TMA lands raw: on E4M3 pools S and PV both run on kind::f8f6f4 straight from
// the raw K and V codes, against Q and P split into hi + lo E4M3 codes (P in TMEM); on INT8
// pools K and V are converted to f16 by the softmax warpgroup that will read the tile, Q is made
// f16, and S and PV run on kind::f16.  Q takes a power-of-two scale per row that the scores give
// back.  Persistent like the context
// kernel: work item = (request, KV head, split, 128 rows), claimed longest first; a 128-row tile
// is 128/g draft tokens x the g query heads of one KV head (the Q box spans g heads), so each
// K / V tile serves the whole group; the two softmax warpgroups
// take the even and the odd KV tiles of one split of kv_chunk keys against the same Q tile; at
// the end B hands its (max, sum) over through shared memory, A merges O_A and O_B from TMEM and
// writes the output row (one split) or a partial row for the combine kernel.  Visibility of the
// new keys comes from the draft-token mask words (bitmaps per row), applied only to the tiles
// that hold new keys.  When no request has more than 64 rows (e.g. 8 draft tokens x 8 heads) and
// g divides 16, the Q rows sit in the first 16 TMEM lanes of each warp's quarter and two threads
// share a row through the 16x32bx2 TMEM shape, each taking half of a tile's keys (max and sum
// combined with one shuffle) and half of the output columns: the softmax of a tile is spread over
// all four sub-partitions instead of running on the two whose lanes hold the rows.
//
// Rows past the request's end and keys past the causal limit are masked by select (never by
// arithmetic on the loaded values); V rows past the sequence end are zeroed before PV, so
// stale or poisoned pool slots cannot reach the output.  Every wait is bounded.
#include <cuda.h>
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;  // generation kernel: the V copies (warp 8: item ring, Q and K)
constexpr int kThreads = 12 * 32;  // three warpgroups: softmax A, softmax B, producer + MMA (+2 idle)
// Registers: 168 per thread at launch (64512 per CTA).  The softmax warpgroups take 216 each and
// the producer / MMA warpgroup keeps 64: 2 * 128 * 216 + 128 * 64 = 63488 <= 64512.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 64;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O once P could exceed 2^8
// E4M3 P (generation kernel, E4M3 pool): P is emitted as 2^4 * exp2(s - m) with m at most 4 below
// the row's true running maximum, so a code never exceeds 2^8 (E4M3 tops out at 448) and values
// down to 2^-10 of the maximum keep E4M3's normal range; O and l carry the same 2^4.
constexpr float kRescaleThresholdE4M3 = 4.0f;
constexpr float kPScaleLog2E4M3 = 4.0f;

// Generation kernel: one Q tile (A and B share it), K[3], V[3] -- each K / V tile has one
// consumer and the two halves alternate.
// With an INT8 pool: Q, K[2], V[2] (f16), a ring of the raw codes (K[2], V[2]) that TMA fills
// and the softmax warpgroups convert, and the per-row Q scales.  With an E4M3 pool nothing is
// converted: the scores read the raw K codes and Q's hi and lo E4M3 tiles, which replace the
// bf16 Q tile in place (a row's two 128-code halves take the 256 bytes of its bf16 codes), and
// PV reads the raw V codes against P's hi and lo E4M3 codes in TMEM: Q, raw K[5], raw V[5].
// Then B's (m, l) per row for A's merge (its own area: the K ring already holds the next item's
// tiles when an item ends).
template <int D, int KV = 0>
struct GenSmem {
  static constexpr bool kQ8 = KV != 0;
  static constexpr bool kF8S = KV == PKV_FP8_E4M3;
  static constexpr int kHalf = 128 * 128;         // one 64-wide half of a 128-row tile (bytes)
  static constexpr int kTile = (D / 64) * kHalf;  // one Q tile or one K / V stage
  static constexpr int kStages = kF8S ? 0 : (kQ8 ? 2 : 3);  // f16 / bf16 V stages (and K stages)
  static constexpr int kKStages = kStages;
  static constexpr int kRawStages = kF8S ? 5 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kTile;
  static constexpr int kVOff = kKOff + kKStages * kTile;
  static constexpr int kRawTile = 128 * D;        // 128 rows of D one-byte codes
  static constexpr int kRawKOff = kVOff + kStages * kTile;
  static constexpr int kRawVOff = kRawKOff + (kQ8 ? kRawStages : 0) * kRawTile;
  static constexpr int kBarOff = kRawVOff + (kQ8 ? kRawStages : 0) * kRawTile;
  static constexpr int kBarBytes = 512;
  static constexpr int kQScaleOff = kBarOff + kBarBytes;  // [128] floats: 1 / (Q row's power-of-two scale)
  static constexpr int kXchOff = kQScaleOff + (kQ8 ? 128 * 4 : 0);  // [2][128] floats: B's m, l
  static constexpr int kBytes = kXchOff + 2 * 128 * 4 + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per CTA");
  static_assert(!kQ8 || D == 128, "8-bit codes only at head_dim 128");
};

enum {
  BAR_Q = 0,
  BAR_KFULL = 1,   // +3 stages
  BAR_KEMPTY = 4,  // +3
  BAR_VFULL = 7,   // +3
  BAR_VEMPTY = 10, // +3
  BAR_SFULL = 13,  // +2 Q tiles
  BAR_PFULL = 15,  // +2
  BAR_ODONE = 17,  // +2
  BAR_MMADONE = 19,
  BAR_MERGE = 20,  // generation: tile B's softmax state is in shared memory
  BAR_RAWK = 21,   // +6: 8-bit pool, raw K codes landed (TMA)
  BAR_RAWV = 27,   // +6: raw V codes landed
  BAR_RAWKEMPTY = 33, // +6: a raw K stage may be refilled (E4M3: its S is done; INT8: converted)
  BAR_RAWVEMPTY = 39, // +6: a raw V stage may be refilled (E4M3: its PV is done; INT8: converted)
  BAR_QRAW = 45,   // the bf16 Q tile landed (warpgroup B rescales and re-encodes it)
  BAR_QFREE = 46,  // an item's last S MMA is done: its Q tile (and re-encoding) may be replaced
  BAR_ITEM = 47,   // +2: item ring entry written
  BAR_ITEMFREE = 49,  // +2: item ring entry read by the V producer, the MMA warp and the eight softmax warps
  BAR_IDONE = 51,  // an item is finished by the MMA warp (issued) and the eight softmax warps
  BAR_QSREAD = 52, // 8-bit pool: warpgroup A has read the item's Q row scales
  BAR_Q2 = 53,     // the same four for the second set of Q rows (two threads per row)
  BAR_QRAW2 = 54,
  BAR_QFREE2 = 55,
  BAR_QSREAD2 = 56,
  NUM_BARS = 57
};
constexpr int kMaxRawStages = 6;


template <int D, int KV, bool HALF>
__global__ void __launch_bounds__(kThreads, 1)
gen_attn_kernel(const ContextParams p, const __grid_constant__ CUtensorMap q_map,
                const __grid_constant__ CUtensorMap kv_map) {
  using L = GenSmem<D, KV>;
  // 8-bit pool: the producer lands raw codes and the softmax warpgroups re-encode what the MMAs
  // cannot read as stored (Q, and on INT8 pools K and V)
  constexpr bool Q8 = L::kQ8;
  // E4M3 pools: scores and PV on kind::f8f6f4 straight from the raw K and V codes, with Q and P
  // split into hi + lo E4M3 codes (7-8 significant bits together); nothing is converted
  constexpr bool F8S = KV == PKV_FP8_E4M3;
  constexpr int S = L::kStages > 0 ? L::kStages : 1;  // (E4M3: no f16 ring; one nominal stage)
  constexpr int R = L::kRawStages;
  static_assert(R <= kMaxRawStages, "raw ring barriers");
  // Q row sets: with two threads per row (HALF) an item's 64 Q rows take 16 of the 32 lanes of
  // each warp's quarter, so consecutive items alternate between lanes 0-15 and 16-31 and the
  // next item's Q is copied (and, on 8-bit pools, re-encoded) while the current item still runs.
  constexpr int QS = HALF ? 2 : 1;
  // set s's barriers: Q landed / re-encoded (the MMAs may read it), raw bf16 landed (8-bit), the
  // set's last S MMA done (it may be refilled), its row scales read by warpgroup A (8-bit)
  auto b_qready = [](int s) { return s ? BAR_Q2 : BAR_Q; };
  auto b_qraw = [](int s) { return s ? BAR_QRAW2 : BAR_QRAW; };
  auto b_qfree = [](int s) { return s ? BAR_QFREE2 : BAR_QFREE; };
  auto b_qsread = [](int s) { return s ? BAR_QSREAD2 : BAR_QSREAD; };
  // ring stage and phase of the g-th K / V tile of the stream (f16 / bf16 rings, raw rings)
  auto stg = [](int g) { return g % S; };
  auto phs = [](int g) { return (g / S) & 1; };
  auto rstg = [](int g) { return g % R; };
  auto rphs = [](int g) { return (g / R) & 1; };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  const uint32_t bar0 = base_s + L::kBarOff;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L::kBarOff + 8 * NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kBarOff + 8 * NUM_BARS + 4);
  volatile int* s_item = reinterpret_cast<volatile int*>(base + L::kBarOff + 8 * NUM_BARS + 8);  // [2]
  static_assert(8 * NUM_BARS + 16 <= L::kBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up: barriers, TMEM (reads nothing earlier kernels write, so it runs before the
  // grid-dependency wait and overlaps the previous kernel's tail) ----
  if (threadIdx.x == 0) {
    // Q / K / V ready: the producer's transaction arrive, or (8-bit) one arrive per warp of the
    // softmax warpgroup that converted them
    const uint32_t ready_count = Q8 ? 4 : 1;
    tc::mbar_init(bar(BAR_Q), ready_count);
    tc::mbar_init(bar(BAR_Q2), ready_count);
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(bar(BAR_KFULL + s), ready_count);
      tc::mbar_init(bar(BAR_KEMPTY + s), 1);
      tc::mbar_init(bar(BAR_VFULL + s), ready_count);
      tc::mbar_init(bar(BAR_VEMPTY + s), 1);
    }
    if (Q8) {
      for (int s = 0; s < R; ++s) {
        tc::mbar_init(bar(BAR_RAWK + s), 1);
        tc::mbar_init(bar(BAR_RAWV + s), 1);
        tc::mbar_init(bar(BAR_RAWKEMPTY + s), F8S ? 1 : 4);
        tc::mbar_init(bar(BAR_RAWVEMPTY + s), F8S ? 1 : 4);  // E4M3: its PV is done
      }
      tc::mbar_init(bar(BAR_QRAW), 1);
      tc::mbar_init(bar(BAR_QRAW2), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(BAR_SFULL + s), 1);
      tc::mbar_init(bar(BAR_PFULL + s), 4);  // one arrive per softmax warp
      tc::mbar_init(bar(BAR_ODONE + s), 1);
    }
    tc::mbar_init(bar(BAR_MMADONE), 1);
    tc::mbar_init(bar(BAR_MERGE), 128);
    tc::mbar_init(bar(BAR_QFREE), 1);
    tc::mbar_init(bar(BAR_QFREE2), 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(BAR_ITEM + s), 1);
      tc::mbar_init(bar(BAR_ITEMFREE + s), 10);  // the V producer, the MMA warp and the eight softmax warps
    }
    tc::mbar_init(bar(BAR_IDONE), 9);
    tc::mbar_init(bar(BAR_QSREAD), 4);
    tc::mbar_init(bar(BAR_QSREAD2), 4);
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

  pdl_wait();

  // ---- work items: (tensor-core generation CTA of the plan, KV head hk) ----
  // Item = (generation request, KV head hk, split of the keys, group of 128 rows); rows are the
  // (token i, query head hk*g + hl) pairs r = i*g + hl of the request's new tokens, keys
  // kt0 .. kend-1 of the split, visibility per draft-token mask; partial results go to the split
  // workspace when the request has several splits.  A CTA claims items from a queue (a cursor
  // the plan zeroes), keeps its TMEM, barriers and rings across them, and every role derives the
  // same geometry from the item index.  The softmax warps start an item, and the MMA warp its
  // first PV, only once all nine have finished the previous one (the item's first S MMAs go out
  // before); the producer runs ahead (the next item's Q once the previous item's last S MMA is
  // done, its K / V tiles as stages free up).
  const int n_items = __ldg(p.counts + kCntTitems) * p.Hkv;
  const int gen_row0 = __ldg(p.counts + kCntGenRow0);
  struct Item {
    int hk, r, past, L_r, nv0, nv1, nkt0, nkt1, kt0, kend, q_row, gr, n_new, s_idx, num_splits, pr0, tok0;
    bool ok;
  };
  auto item_of = [&](int w) {
    Item it;
    const int ti = w / p.Hkv;
    it.hk = w - ti * p.Hkv;
    const int2 im = p.titem_map[ti];
    it.gr = min(max(im.x, 0), p.G - 1);
    it.r = p.C + it.gr;
    it.n_new = __ldg(p.ctx_len + it.r);
    it.past = __ldg(p.past + it.r);
    it.L_r = it.past + it.n_new;
    const int rows = it.n_new * p.group;
    const int n_rg = (rows + kCtxTileM - 1) / kCtxTileM;
    it.s_idx = im.y / max(n_rg, 1);
    const int rg = im.y - it.s_idx * n_rg;
    it.num_splits = __ldg(p.split_prefix + it.gr + 1) - __ldg(p.split_prefix + it.gr);
    it.kt0 = it.s_idx * p.kv_chunk;
    it.kend = min(it.L_r, it.kt0 + p.kv_chunk);
    it.pr0 = rg * kCtxTileM;  // first (token, head) pair of the item: one Q tile of 128 pairs
    it.tok0 = __ldg(p.cu_q + it.r);
    it.q_row = it.tok0 + it.pr0 / p.group;
    it.nv0 = max(0, min(128, rows - it.pr0));
    // both halves of the pipeline serve the same rows: A takes the split's even KV tiles, B the
    // odd ones, each with its own S, P, O and softmax state, merged at the end
    const int nk = (it.kend - it.kt0 + kCtxTileN - 1) / kCtxTileN;
    it.nkt0 = (nk + 1) / 2;
    it.nkt1 = nk / 2;
    it.nv1 = it.nkt1 > 0 ? it.nv0 : 0;
    it.ok = im.y >= 0 && it.s_idx < it.num_splits && it.kt0 < it.kend && it.nv0 > 0 && it.n_new >= 1 &&
            it.n_new <= PKV_MAX_GEN_TOKENS && it.tok0 >= gen_row0 && it.tok0 + it.n_new <= p.T &&
            static_cast<int64_t>(__ldg(p.part_prefix + it.gr)) + static_cast<int64_t>(it.num_splits) * it.n_new <=
                p.total_parts;
    return it;
  };

  const uint32_t sQ = base_s + L::kQOff;
  auto sK = [&](int st) { return base_s + L::kKOff + st * L::kTile; };
  auto sV = [&](int st) { return base_s + L::kVOff + st * L::kTile; };

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
  // consumers: item k of this CTA from the ring (-1: no more work), entry handed back
  auto take_item = [&](int k, int& w) {
    const int slot = k & 1;
    if (!warp_wait(bar(BAR_ITEM + slot), (k >> 1) & 1)) return false;
    w = *(s_item + slot);
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(BAR_ITEMFREE + slot));
    return true;
  };
  // the end of an item for the MMA warp and the softmax warps; the next one starts when all nine
  // warps have got here (n: items this CTA has finished so far)
  auto item_done = [&]() {
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(BAR_IDONE));
  };
  auto wait_prev = [&](int n) { return n == 0 || warp_wait(bar(BAR_IDONE), (n - 1) & 1); };

  if (warp >= 8) {
    // one setmaxnreg instruction for all four warps of the control warpgroup
    tc::regs_dec<kRegsControl>();
    // The producer and MMA warps run their loops with all 32 lanes (waits and control flow
    // warp-uniform) and let one elected lane issue the TMA copies / MMAs: a warp that sits
    // diverged on one lane gets issue slots far less often next to a busy softmax warp on the
    // same sub-partition, and the tensor pipe then runs dry between MMA batches.
    if (warp == kProducerWarp || warp == kVProducerWarp) {
      // ======================= item queue + TMA producers =======================
      // Warp 8 publishes the items and copies Q and K, warp 10 (its own sub-partition) takes
      // the items from the ring like a consumer and copies V: each tile's copies are issued by
      // two warps that share their sub-partitions with busy softmax warps, instead of one.
      const bool vwarp = warp == kVProducerWarp;
      int w = static_cast<int>(blockIdx.x);
      int issued_k = 0, issued_v = 0;  // K / V stream tiles issued (all items; each warp its kind)
      int nq = 0;                      // Q tiles loaded
      auto q_bar = [&](int qs) { return Q8 ? b_qraw(qs) : b_qready(qs); };  // 8-bit: warpgroup B re-encodes Q first
      bool pok = true;
      for (int k = 0; pok; ++k) {
        if (vwarp) {
          if (!take_item(k, w)) { pok = false; break; }
          if (w < 0) break;
        } else {
          const int slot = k & 1;
          if (k >= 2 && !warp_wait(bar(BAR_ITEMFREE + slot), ((k - 2) >> 1) & 1)) { pok = false; break; }
          const bool more = w < n_items;
          if (lane == 0) {
            *(s_item + slot) = more ? w : -1;
            tc::mbar_arrive(bar(BAR_ITEM + slot));
          }
          __syncwarp();
          if (!more) break;
        }
        const Item it = item_of(w);
        if (!it.ok) {
          if (lane == 0 && !vwarp) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // plan disagrees
        } else {
          const int nT = it.nkt0 + it.nkt1;
          const int32_t* tbl = p.tbl + static_cast<int64_t>(it.r) * p.max_blocks;
          const int box_rows = p.B < kCtxTileN ? p.B : kCtxTileN;
          const int pages_per_tile = kCtxTileN / box_rows;  // <= 8 (B >= 16)
          const int n_pages_seq = (it.L_r + p.B - 1) / p.B;
          // lane pp < pages_per_tile holds page pp of tile j (B <= 128: whole pages per tile)
          auto has_page = [&](int j) {
            const int lb = (it.kt0 + j * kCtxTileN) / p.B + lane;
            return lane < pages_per_tile && lb < n_pages_seq && lb < p.max_blocks;
          };
          // The split's table entries, 32 at a time: lane l holds entry 32 w + l of window w (the
          // split starts on a page boundary: kt0 is a multiple of 128), and the next window's load
          // is in flight while the current one serves its tiles, so a tile's copies never wait for
          // a table read (one read per tile, a tile ahead, paced the copies at the read latency
          // under the batch's own traffic)
          const int page0 = it.kt0 / p.B;
          auto load_win = [&](int wn) {
            const int lb = page0 + 32 * wn + lane;
            return (lb < n_pages_seq && lb < p.max_blocks) ? __ldg(tbl + lb) : -1;
          };
          int win = 0;
          int pg_win = load_win(0), pg_win_next = load_win(1);
          auto lookup = [&](int j) {
            const int pi = (j * kCtxTileN) / p.B;  // the tile's first page within the split
            if ((pi >> 5) != win) {                 // tiles go in order: the next window
              win = pi >> 5;
              pg_win = pg_win_next;
              pg_win_next = load_win(win + 1);
            }
            const int pg = __shfl_sync(0xffffffffu, pg_win, (pi & 31) + (lane < pages_per_tile ? lane : 0));
            return has_page(j) ? pg : -1;
          };
          // tile j of the item (table entries pg) into the next stage of the CTA's stream
          auto issue_tile = [&](int j, int pg) {
            if (warp_abort()) return false;
            const int g = vwarp ? issued_v : issued_k;  // the tile's place in the CTA's stream
            if (has_page(j) && (pg < 0 || pg >= p.NB)) {
              if (!vwarp) flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
              pg = -1;
            }
            const uint32_t bytes =
                static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, pg >= 0))) * box_rows * D * (Q8 ? 1 : 2);
            if constexpr (Q8) {
              // raw codes of page `lane` into the raw rings; K and V stages are freed separately
              // (a raw K stage once its S is done (E4M3) or its codes are converted (INT8), a raw
              // V stage once its PV is done (E4M3) or its codes are converted (INT8))
              const uint32_t roff = static_cast<uint32_t>(lane * box_rows * D);
              const int rs = rstg(g), rph = rphs(g - R);
              if (!vwarp) {
                if (g >= R && !warp_wait(bar(BAR_RAWKEMPTY + rs), rph)) return false;
                if (lane == 0) tc::mbar_arrive_expect_tx(bar(BAR_RAWK + rs), bytes);
                __syncwarp();
                if (pg >= 0)
                  tc::tma_load_3d(base_s + L::kRawKOff + rs * L::kRawTile + roff, &kv_map, bar(BAR_RAWK + rs), 0, it.hk,
                                  (pg * 2 + 0) * p.B);
                __syncwarp();
                ++issued_k;
              } else {
                if (g >= R && !warp_wait(bar(BAR_RAWVEMPTY + rs), rph)) return false;
                if (lane == 0) tc::mbar_arrive_expect_tx(bar(BAR_RAWV + rs), bytes);
                __syncwarp();
                if (pg >= 0)
                  tc::tma_load_3d(base_s + L::kRawVOff + rs * L::kRawTile + roff, &kv_map, bar(BAR_RAWV + rs), 0, it.hk,
                                  (pg * 2 + 1) * p.B);
                __syncwarp();
                ++issued_v;
              }
              return true;
            }
            // one lane registers the tile's bytes, then every lane with a page issues its own
            // copies (no shuffles, no serial issue loop on one lane)
            const int st = stg(g);
            const uint32_t koff = static_cast<uint32_t>(lane * box_rows * 128);
            if (!vwarp) {
              if (g >= S && !warp_wait(bar(BAR_KEMPTY + st), phs(g - S))) return false;
              if (lane == 0) tc::mbar_arrive_expect_tx(bar(BAR_KFULL + st), bytes);
              __syncwarp();
              if (pg >= 0)
                for (int dh = 0; dh < D / 64; ++dh)
                  tc::tma_load_4d(sK(st) + dh * L::kHalf + koff, &kv_map, bar(BAR_KFULL + st), 0, dh, it.hk,
                                  (pg * 2 + 0) * p.B);
              __syncwarp();
              ++issued_k;
            } else {
              if (g >= S && !warp_wait(bar(BAR_VEMPTY + st), phs(g - S))) return false;
              if (lane == 0) tc::mbar_arrive_expect_tx(bar(BAR_VFULL + st), bytes);
              __syncwarp();
              if (pg >= 0)
                for (int dh = 0; dh < D / 64; ++dh)
                  tc::tma_load_4d(sV(st) + dh * L::kHalf + koff, &kv_map, bar(BAR_VFULL + st), 0, dh, it.hk,
                                  (pg * 2 + 1) * p.B);
              __syncwarp();
              ++issued_v;
            }
            return true;
          };
          // the item's Q tile goes out as soon as the previous item's last S MMA is done, then its
          // tiles as stages free up; the first table window loads meanwhile
#ifdef PKV_SELFTEST
          // Self-test build only (compiled by the tests, never into libpaged_kv.so): no K / V
          // copy is issued, so the MMA warp's wait for the first K tile and the softmax warps'
          // waits for their first S run out after the short self-test budget and the CTA winds
          // down through the timeout path; the Q tile lands before the teardown (waited below).
          const int n_issue = 0;
#else
          const int n_issue = nT;
#endif
          const int qset = nq % QS;  // the item's Q rows, refilled once their previous item's last S is done
          if (!vwarp && pok && nq >= QS && !warp_wait(bar(b_qfree(qset)), ((nq / QS) - 1) & 1)) pok = false;
          if (!pok) break;
          // one Q tile (128 / g tokens x the group's g heads), shared by A and B; HALF: 64 rows,
          // rows 16k .. 16k+15 into tile rows 32k .. 32k+15 (a box of g heads x 16 / g tokens)
          if (!vwarp && tc::elect_one()) {
            if constexpr (HALF) {
              tc::mbar_arrive_expect_tx(bar(q_bar(qset)), 64 * D * 2);
              for (int kq = 0; kq < 4; ++kq)
                for (int dh = 0; dh < D / 64; ++dh)
                  tc::tma_load_4d(sQ + dh * L::kHalf + (kq * 32 + qset * 16) * 128, &q_map, bar(q_bar(qset)), 0, dh,
                                  it.hk * p.group, it.q_row + kq * 16 / p.group);
            } else {
              tc::mbar_arrive_expect_tx(bar(q_bar(0)), 128 * D * 2);
              for (int dh = 0; dh < D / 64; ++dh)
                tc::tma_load_4d(sQ + dh * L::kHalf, &q_map, bar(q_bar(0)), 0, dh, it.hk * p.group, it.q_row);
            }
          }
          __syncwarp();
          if (!vwarp) ++nq;
          for (int j = 0; pok && j < n_issue; ++j) pok = issue_tile(j, lookup(j));
        }
        if (!pok) break;
        if (!vwarp) {
          // claim the next item while this one's tiles are still being consumed
          int nxt = 0;
          if (lane == 0) nxt = atomicAdd(p.gen_cursor, 1) + static_cast<int>(gridDim.x);
          w = __shfl_sync(0xffffffffu, nxt, 0);
        }
      }
      if (!pok && lane == 0) fail();
      __syncwarp();
      // the last copy into each stage and the last Q tile have landed before the CTA can wind
      // down, however the consumers fare (on the normal path these phases completed long ago)
      if constexpr (Q8) {
        for (int j = (issued_k > R ? issued_k - R : 0); j < issued_k; ++j)
          tc::mbar_wait(bar(BAR_RAWK + rstg(j)), rphs(j), 200000000LL);
        for (int j = (issued_v > R ? issued_v - R : 0); j < issued_v; ++j)
          tc::mbar_wait(bar(BAR_RAWV + rstg(j)), rphs(j), 200000000LL);
      } else {
        for (int j = (issued_k > S ? issued_k - S : 0); j < issued_k; ++j)
          tc::mbar_wait(bar(BAR_KFULL + stg(j)), phs(j), 200000000LL);
        for (int j = (issued_v > S ? issued_v - S : 0); j < issued_v; ++j)
          tc::mbar_wait(bar(BAR_VFULL + stg(j)), phs(j), 200000000LL);
      }
      for (int i = (nq > QS ? nq - QS : 0); i < nq; ++i) tc::mbar_wait(bar(q_bar(i % QS)), (i / QS) & 1, 200000000LL);
    } else if (warp == kMmaWarp) {
      // ======================= MMA issuer =======================
      // tcgen05.commit tracks the MMAs of the thread that issues it: elect.sync on a converged
      // warp picks the same (lowest) lane every time, so MMAs and commits share one thread.
      constexpr uint32_t idesc_s = Q8 ? tc::idesc_f16(128, kCtxTileN, 0) : tc::idesc_bf16(128, kCtxTileN, 0);
      constexpr uint32_t idesc_o = Q8 ? tc::idesc_f16(128, D, 1) : tc::idesc_bf16(128, D, 1);
      // Descriptors are built once per operand tile and advanced by adding the byte offset / 16
      // (the start address occupies the low bits and never carries out inside a tile): this
      // warp competes for issue slots with a busy softmax warp, so every instruction counts.
      const uint64_t dq0 = tc::sdesc_sw128(sQ, 16, 1024);
      // per-stage K / V descriptors: stages are L::kTile apart, i.e. kTile / 16 descriptor units
      const uint64_t dk0 = tc::sdesc_sw128(sK(0), 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(sV(0), L::kHalf, 1024);
      // E4M3: raw V stages, MN-major (a 128-code row per key, one 128-byte swizzle atom wide;
      // 8-row groups 1 KB apart)
      const uint64_t dv8 = tc::sdesc_sw128(base_s + L::kRawVOff, L::kRawTile, 1024);
      auto stage_off = [](int st) { return static_cast<uint64_t>(st) * (L::kTile / 16); };
      int G = 0;             // K / V stream tiles of earlier items
      int sc0 = 0, sc1 = 0;  // S / P tiles of earlier items, per half
      int nq = 0, ndone = 0; // Q tiles consumed, items finished
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int w = -1;
        if (!take_item(k, w)) { ok = false; break; }
        if (w < 0) break;
        const Item it = item_of(w);
        if (!it.ok) continue;
        const int nkt0 = it.nkt0, nkt1 = it.nkt1;
        const bool hasB = it.nv1 > 0;
        const int qset = nq % QS;  // the item's Q rows
        auto uses = [&](int j, int x) { return j < (x ? nkt1 : nkt0); };
        // tile j of half x: the (G + 2j + x)-th K / V tile of the CTA's stream
        auto gtile = [&](int j, int x) { return G + 2 * j + x; };
        auto kfull = [&](int j, int x) {
          const int g = gtile(j, x);
          if constexpr (F8S) return warp_wait(bar(BAR_RAWK + rstg(g)), rphs(g));  // raw codes landed
          return warp_wait(bar(BAR_KFULL + stg(g)), phs(g));
        };
        auto issue_s = [&](int j, int x) {
          const int g = gtile(j, x);
          const int st = stg(g);
          const uint64_t a0 = dq0;  // A and B share the Q tile
          const uint64_t b0 = dk0 + stage_off(st);
          if constexpr (F8S) {
            // Q hi and lo tiles (one 128-byte row of codes per Q row) replace the bf16 Q tile's
            // two halves; K is the raw tile: four K=32 steps of 32 bytes, hi then lo
            const uint64_t aq = dq0;
            const uint64_t bk = tc::sdesc_sw128(base_s + L::kRawKOff + rstg(g) * L::kRawTile, 16, 1024);
            constexpr uint64_t kLo = L::kHalf / 16;  // lo tile: the Q tile's second half
            if (tc::elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc::mma_e4m3_ss(tmem + 128 * x, aq + 2 * kk, bk + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) tc::mma_e4m3_ss(tmem + 128 * x, aq + kLo + 2 * kk, bk + 2 * kk, idesc_s, 1u);
              tc::mma_commit(bar(BAR_SFULL + x));
              tc::mma_commit(bar(BAR_RAWKEMPTY + rstg(g)));  // the raw K stage may be refilled
              if (2 * j + x == nkt0 + nkt1 - 1) tc::mma_commit(bar(b_qfree(qset)));  // the item's last S
            }
            __syncwarp();
            return;
          }
          if (tc::elect_one()) {
            if constexpr (D == 128) {
              // steps kk: ((kk / 4) * 16 KB + (kk % 4) * 32 B) / 16
              tc::mma_bf16_ss_x8<0, 2, 4, 6, L::kHalf / 16, L::kHalf / 16 + 2, L::kHalf / 16 + 4, L::kHalf / 16 + 6>(
                  tmem + 128 * x, a0, b0, idesc_s, 0u);
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4);
                tc::mma_bf16_ss(tmem + 128 * x, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u);
              }
            }
            tc::mma_commit(bar(BAR_SFULL + x));
            tc::mma_commit(bar(BAR_KEMPTY + st));  // each K / V tile has one user
            // the item's last S: the Q tile (and its re-encoding) may be replaced once it is done
            if (2 * j + x == nkt0 + nkt1 - 1) tc::mma_commit(bar(b_qfree(qset)));
          }
          __syncwarp();
        };
        ok = warp_wait(bar(b_qready(qset)), (nq / QS) & 1) && kfull(0, 0);
        ++nq;
        if (ok) {
          tc::fence_after_sync();
          issue_s(0, 0);
          if (hasB) {
            ok = kfull(0, 1);  // B's first tile is the stream's second
            if (ok) {
              tc::fence_after_sync();
              issue_s(0, 1);
            }
          }
        }
        // The item's first S MMAs go out while the previous item's epilogue runs (they touch
        // only S); its first PV waits until every warp has finished that item (A's merge reads
        // both O halves).
        if (ok && !wait_prev(ndone)) ok = false;
        // no abort-flag poll per tile: a shared-memory load here sits on the critical path
        // (P ready -> next MMA); if another warp gave up, the waits below run out instead
        for (int j = 0; ok && j < nkt0; ++j) {
          for (int x = 0; x < 2 && ok; ++x) {
            if (!uses(j, x)) continue;
            const int g = gtile(j, x);
            if (!warp_wait(bar(BAR_PFULL + x), ((x ? sc1 : sc0) + j) & 1)) { ok = false; break; }
            if constexpr (F8S) {
              if (!warp_wait(bar(BAR_RAWV + rstg(g)), rphs(g))) { ok = false; break; }
              tc::fence_after_sync();
              const uint64_t bv = dv8 + static_cast<uint64_t>(rstg(g)) * (L::kRawTile / 16);
              if (tc::elect_one()) {
                // P's hi codes (the tile's TMEM columns 0-31), then its lo codes (32-63), against
                // the raw V codes read MN-major: four K=32 steps of 32 rows (4 KB) each
                static_assert(kCtxTileN == 128, "four K=32 steps per KV tile");
                tc::mma_e4m3_ts_x4<32 * 128 / 16>(tmem + 256 + 128 * x, tmem + 128 * x, bv, idesc_o, j > 0 ? 1u : 0u);
                tc::mma_e4m3_ts_x4<32 * 128 / 16>(tmem + 256 + 128 * x, tmem + 128 * x + 32, bv, idesc_o, 1u);
                tc::mma_commit(bar(BAR_RAWVEMPTY + rstg(g)));  // the raw V stage may be refilled
                if (j == (x ? nkt1 : nkt0) - 1) tc::mma_commit(bar(BAR_ODONE + x));
              }
              __syncwarp();
            } else {
              if (!warp_wait(bar(BAR_VFULL + stg(g)), phs(g))) { ok = false; break; }
              tc::fence_after_sync();
              const uint64_t v0 = dv0 + stage_off(stg(g));
              if (tc::elect_one()) {
                static_assert(kCtxTileN == 128, "eight K=16 steps per KV tile");
                tc::mma_bf16_ts_x8<16 * 128 / 16>(tmem + 256 + 128 * x, tmem + 128 * x, v0, idesc_o, j > 0 ? 1u : 0u);
                tc::mma_commit(bar(BAR_VEMPTY + stg(g)));
                if (j == (x ? nkt1 : nkt0) - 1) tc::mma_commit(bar(BAR_ODONE + x));
              }
              __syncwarp();
            }
            if (uses(j + 1, x)) {
              if (!kfull(j + 1, x)) { ok = false; break; }
              tc::fence_after_sync();
              issue_s(j + 1, x);
            }
          }
        }
        if (!ok) break;
        G += nkt0 + nkt1;
        sc0 += nkt0;
        sc1 += nkt1;
        item_done();
        ++ndone;
      }
      if (!ok && lane == 0) fail();
      if (tc::elect_one()) {
        tc::mma_commit(bar(BAR_MMADONE));
        tc::mbar_wait(bar(BAR_MMADONE), 0, 200000000LL);  // nothing of ours still runs on TMEM
      }
      __syncwarp();
    }
  } else {
    // ======================= softmax warpgroups =======================
    tc::regs_inc<kRegsSoftmax>();
    const int x = warp >> 2;                 // Q tile A (0) or B (1)
    const int row = (warp & 3) * 32 + lane;  // tile row == TMEM lane (K / V rows, Q re-encoding)
    // HALF (at most 64 Q rows): Q row qrow sits in tile row srow, the first 16 lanes of each
    // warp's quarter; threads t and t + 16 of a warp share it, each on one half (kh) of the keys
    // of a tile and of the output columns.  Otherwise a thread owns tile row `row` whole.
    const int qrow = HALF ? (warp & 3) * 16 + (lane & 15) : row;
    const int srow0 = HALF ? (warp & 3) * 32 + (lane & 15) : row;
    const int kh = HALF ? (lane >> 4) : 0;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS0 = tmem + 128 * x + lane_off;
    const uint32_t tO0 = tmem + 256 + 128 * x + lane_off;
    float* xch = reinterpret_cast<float*>(base + L::kXchOff);  // [2][128]: B's m, l per row
    // E4M3 P: 32 scores (v) -> P' = exp2(s * sl2 - m + kPOff), summed into ls, as 8 words of hi
    // codes and 8 of lo codes (four keys per word, key 4i + b in byte b) at hw / lw[w0 ..]
    auto emit_e4m3 = [&](uint32_t(&v)[32], float2& ls, uint32_t(&hw)[16], uint32_t(&lw)[16], int w0, float2 sl2x2,
                         float2 negm) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float2 xa = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2, negm);
        const float2 xb = ffma2(make_float2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), sl2x2, negm);
        const float2 pa = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
        const float2 pb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
        ls = fadd2(ls, pa);
        ls = fadd2(ls, pb);
        uint32_t h01, l01, h23, l23;
        split_cut_e4m3x2(pa.x, pa.y, h01, l01);
        split_cut_e4m3x2(pb.x, pb.y, h23, l23);
        hw[w0 + (e >> 2)] = __byte_perm(h01, h23, 0x5410);
        lw[w0 + (e >> 2)] = __byte_perm(l01, l23, 0x5410);
      }
    };
    // ---- INT8 pool: this warpgroup turns the raw codes of its own tiles into f16 ----
    // (E4M3 pools read their codes as stored.)  Thread `row` converts tile row `row`: 128 codes
    // in the 128-byte swizzle TMA wrote (16-byte chunk j at j ^ (row % 8)) become 16 f16 chunks of
    // the K-major 128-byte-swizzled layout the MMAs read, in 64-wide head-dim halves; every int8
    // is exact in f16.  A warpgroup converts its next tile right after handing over its P, while
    // its own PV and the other warpgroup's MMAs run.  A V row past the end of the sequence (stale
    // or unloaded slot) is written as zeros instead.
    auto cvt_row = [&](uint32_t raw_off, uint32_t dst_s, bool zero) {
#pragma unroll
      for (int jc = 0; jc < 8; ++jc) {
        const uint4 w = zero ? make_uint4(0u, 0u, 0u, 0u)
                             : *reinterpret_cast<const uint4*>(base + raw_off + row * 128 + ((jc ^ (row & 7)) << 4));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        uint32_t f[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (KV == PKV_INT8) {
            i8x4_to_f16x2(wv[k], f[2 * k], f[2 * k + 1]);
          } else {
            e4m3x4_to_f16x2(wv[k], f[2 * k], f[2 * k + 1]);
          }
        }
        const uint32_t drow = dst_s + (jc >> 2) * L::kHalf + row * 128;
        const uint32_t c0 = static_cast<uint32_t>(2 * (jc & 3));
        st_shared_v4(drow + ((c0 ^ static_cast<uint32_t>(row & 7)) << 4), f[0], f[1], f[2], f[3]);
        st_shared_v4(drow + (((c0 + 1) ^ static_cast<uint32_t>(row & 7)) << 4), f[4], f[5], f[6], f[7]);
      }
    };
    // tile g of the stream (this warpgroup's), whose first vrows rows hold keys of the split: raw
    // stage g % R into f16 stage g % S -- K once the stage's previous S is done, then V once its
    // previous PV is done; each step frees a raw stage (INT8 pools only)
    auto convert_tile = [&](int g, int vrows) {
      const int rs = rstg(g), rph = rphs(g), st = stg(g), ph_prev = phs(g - S);
      if constexpr (!F8S) {
        if (!warp_wait(bar(BAR_RAWK + rs), rph) || (g >= S && !warp_wait(bar(BAR_KEMPTY + st), ph_prev))) return false;
        cvt_row(L::kRawKOff + rs * L::kRawTile, sK(st), false);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(bar(BAR_KFULL + st));
          tc::mbar_arrive(bar(BAR_RAWKEMPTY + rs));
        }
      }
      if (!warp_wait(bar(BAR_RAWV + rs), rph) || (g >= S && !warp_wait(bar(BAR_VEMPTY + st), ph_prev))) return false;
      cvt_row(L::kRawVOff + rs * L::kRawTile, sV(st), row >= vrows);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(bar(BAR_VFULL + st));
        tc::mbar_arrive(bar(BAR_RAWVEMPTY + rs));
      }
      return true;
    };
    int G = 0, sc = 0, nq = 0;        // stream tiles, this half's S / P tiles, Q tiles of earlier items
    int n_epi = 0, n_merge = 0, ndone = 0;  // this half's epilogues, merges, items finished
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int w = -1;
      if (!take_item(k, w)) { ok = false; break; }
      if (w < 0) break;
      const Item it = item_of(w);
      if (!it.ok) continue;
      // the item's Q rows: lanes 16 qset .. 16 qset + 15 of each quarter (HALF), else all
      const int qset = nq % QS;
      const int srow = srow0 + 16 * qset;
      const uint32_t tS = tS0 + (static_cast<uint32_t>(16 * qset) << 16);
      const uint32_t tO = tO0 + (static_cast<uint32_t>(16 * qset) << 16);
      const int nvx = x ? it.nv1 : it.nv0, nk = x ? it.nkt1 : it.nkt0;
      const int nT = it.nkt0 + it.nkt1;  // KV tiles of the item (A the even ones, B the odd ones)
      const int zero_x = (nT - 1) & 1;   // the user of the last V tile zeroes its tail
      auto gtile = [&](int j) { return G + 2 * j + x; };  // this half's j-th tile in the CTA's stream
      // the row's token and the new keys it sees (bit j: key past + j)
      uint64_t vis = ~0ull;
      int tok_i = 0, hl = 0;
      {
        const int pr = it.pr0 + qrow;  // A and B hold the same rows
        if (qrow < nvx) {
          tok_i = pr / p.group;
          hl = pr - tok_i * p.group;
          if (p.mask != nullptr) {
            const uint32_t* mrow = p.mask + static_cast<int64_t>(it.tok0 + tok_i - gen_row0) * p.mask_words;
            vis = __ldg(mrow);
            if (it.n_new > 32 && p.mask_words > 1) vis |= static_cast<uint64_t>(__ldg(mrow + 1)) << 32;
            vis |= 1ull << tok_i;
          } else {
            vis = (2ull << tok_i) - 1;  // j <= i (i = 63 wraps to all ones)
          }
        }
      }
      // 8-bit pool: warpgroup B (whose epilogue is the short one) re-encodes the item's Q and (INT8)
      // each warpgroup converts its first tile, before waiting for the previous item to end:
      // they touch shared memory only, and their barriers order them against its MMAs.
      float sl2 = p.scale_log2;
      float* qscale = reinterpret_cast<float*>(base + L::kQScaleOff);
      if constexpr (Q8) {
        if (x == 1) {
          // Q row `row`: bf16 -> f16 times 2^(14 - e), e the exponent of the row's largest |q| (far
          // below f16's 65504), in place; the scores take 2^(e - 14) back
          ok = warp_wait(bar(b_qraw(qset)), (nq / QS) & 1);
          if constexpr (F8S && HALF) {
            // 64 rows, two threads per row: thread kh splits head-dim half kh of row srow (both
            // halves of every row are read before any code is written: the lo codes of half 0
            // land where half 1's bf16 codes sat)
            if (ok) {
              const uint32_t rbase = static_cast<uint32_t>(L::kQOff + kh * L::kHalf + srow * 128);
              uint4 qr[8];
              float amax = 0.f;
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                qr[c] = *reinterpret_cast<const uint4*>(base + rbase + ((c ^ (srow & 7)) << 4));
                const uint32_t u[4] = {qr[c].x, qr[c].y, qr[c].z, qr[c].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  amax = max3f(amax, fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u)));
              }
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));  // the row's other half
              int ex = 0;
              if (amax > 0.f) frexpf(amax, &ex);
              const float up = ldexpf(1.f, 8 - ex);  // |q| * up in [128, 256), under 448
              if (nq >= QS && !warp_wait(bar(b_qsread(qset)), ((nq / QS) - 1) & 1)) { ok = false; break; }
              __syncwarp();
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {  // code chunk jc = 4 kh + jj from bf16 chunks 2 jj, 2 jj + 1
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                  const uint4 w = qr[2 * jj + hc];
                  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int k = 0; k < 4; k += 2) {
                    uint32_t h0, l0, h1, l1;
                    split_e4m3x2(__uint_as_float(u[k] << 16) * up, __uint_as_float(u[k] & 0xFFFF0000u) * up, h0, l0);
                    split_e4m3x2(__uint_as_float(u[k + 1] << 16) * up, __uint_as_float(u[k + 1] & 0xFFFF0000u) * up, h1,
                                 l1);
                    hw[2 * hc + (k >> 1)] = (h0 & 0xFFFFu) | (h1 << 16);
                    lw[2 * hc + (k >> 1)] = (l0 & 0xFFFFu) | (l1 << 16);
                  }
                }
                const uint32_t off = static_cast<uint32_t>(srow * 128 + (((4 * kh + jj) ^ (srow & 7)) << 4));
                st_shared_v4(sQ + off, hw[0], hw[1], hw[2], hw[3]);
                st_shared_v4(sQ + L::kHalf + off, lw[0], lw[1], lw[2], lw[3]);
              }
              if (kh == 0) qscale[srow] = 1.f / up;
              tc::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(bar(b_qready(qset)));
            }
          } else if constexpr (HALF) {
            // INT8 pool, 64 rows, two threads per row: thread kh makes head-dim half kh of row
            // srow f16 in place (the row's scale from both halves)
            if (ok) {
              const uint32_t rbase = static_cast<uint32_t>(L::kQOff + kh * L::kHalf + srow * 128);
              uint4 qr[8];
              float amax = 0.f;
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                qr[c] = *reinterpret_cast<const uint4*>(base + rbase + ((c ^ (srow & 7)) << 4));
                const uint32_t u[4] = {qr[c].x, qr[c].y, qr[c].z, qr[c].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  amax = max3f(amax, fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u)));
              }
              amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
              int ex = 0;
              if (amax > 0.f) frexpf(amax, &ex);
              const float up = ldexpf(1.f, 14 - ex);  // |q| * up in [2^13, 2^14)
              if (nq >= QS && !warp_wait(bar(b_qsread(qset)), ((nq / QS) - 1) & 1)) { ok = false; break; }
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint32_t u[4] = {qr[c].x, qr[c].y, qr[c].z, qr[c].w};
                uint32_t hh[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  hh[k] = pack_f16x2(__uint_as_float(u[k] << 16) * up, __uint_as_float(u[k] & 0xFFFF0000u) * up);
                st_shared_v4(base_s + rbase + ((c ^ (srow & 7)) << 4), hh[0], hh[1], hh[2], hh[3]);
              }
              if (kh == 0) qscale[srow] = 1.f / up;
              tc::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(bar(b_qready(qset)));
            }
          } else if (ok) {
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const uint4 w = *reinterpret_cast<const uint4*>(base + L::kQOff + (c >> 3) * L::kHalf + row * 128 +
                                                              (((c & 7) ^ (row & 7)) << 4));
              const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k)
                amax = max3f(amax, fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u)));
            }
            int ex = 0;
            if (amax > 0.f) frexpf(amax, &ex);
            // f16: |q| * up in [2^13, 2^14); E4M3 hi + lo: |q| * up in [128, 256), under 448
            const float up = ldexpf(1.f, (F8S ? 8 : 14) - ex);
            // the previous item's scales are read by both warpgroups before they are replaced
            if (nq >= QS && !warp_wait(bar(b_qsread(qset)), ((nq / QS) - 1) & 1)) { ok = false; break; }
            if constexpr (F8S) {
              // code chunk jc (16 codes = q elements 16 jc ..) from bf16 chunks 2 (jc % 4) and
              // 2 (jc % 4) + 1 of head-dim half jc / 4; the hi tile replaces the row's first half
              // and the lo tile its second, so the whole row is read before any of it is written
              uint4 qr[16];
#pragma unroll
              for (int c = 0; c < 16; ++c)
                qr[c] = *reinterpret_cast<const uint4*>(base + L::kQOff + (c >> 3) * L::kHalf + row * 128 +
                                                        (((c & 7) ^ (row & 7)) << 4));
#pragma unroll
              for (int jc = 0; jc < 8; ++jc) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                  const uint4 w = qr[(jc >> 2) * 8 + 2 * (jc & 3) + hc];
                  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int k = 0; k < 4; k += 2) {
                    uint32_t h0, l0, h1, l1;
                    split_e4m3x2(__uint_as_float(u[k] << 16) * up, __uint_as_float(u[k] & 0xFFFF0000u) * up, h0, l0);
                    split_e4m3x2(__uint_as_float(u[k + 1] << 16) * up, __uint_as_float(u[k + 1] & 0xFFFF0000u) * up, h1,
                                 l1);
                    hw[2 * hc + (k >> 1)] = (h0 & 0xFFFFu) | (h1 << 16);
                    lw[2 * hc + (k >> 1)] = (l0 & 0xFFFFu) | (l1 << 16);
                  }
                }
                const uint32_t off = static_cast<uint32_t>(row * 128 + ((jc ^ (row & 7)) << 4));
                st_shared_v4(sQ + off, hw[0], hw[1], hw[2], hw[3]);
                st_shared_v4(sQ + L::kHalf + off, lw[0], lw[1], lw[2], lw[3]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const uint32_t a = base_s + L::kQOff + (c >> 3) * L::kHalf + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                const uint4 w = *reinterpret_cast<const uint4*>(base + (a - base_s));
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                uint32_t h[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  h[k] = pack_f16x2(__uint_as_float(u[k] << 16) * up, __uint_as_float(u[k] & 0xFFFF0000u) * up);
                st_shared_v4(a, h[0], h[1], h[2], h[3]);
              }
            }
            qscale[row] = 1.f / up;
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(b_qready(qset)));
          }
        }
        if constexpr (!F8S) {
          if (ok && nk > 0) ok = convert_tile(gtile(0), it.kend - (it.kt0 + x * kCtxTileN));  // its first tile
        }
        if (!ok) break;
      }
      if (!wait_prev(ndone)) { ok = false; break; }
      if constexpr (Q8) {
        ok = warp_wait(bar(b_qready(qset)), (nq / QS) & 1);
        if (ok) sl2 *= qscale[srow];
        if (!ok) break;
        __syncwarp();
        if (x == 0 && lane == 0) tc::mbar_arrive(bar(b_qsread(qset)));
      }
      ++nq;  // every pool: the next item's Q rows are the other set
      const int kt0 = it.kt0, kend = it.kend, past = it.past;
      constexpr float kThr = F8S ? kRescaleThresholdE4M3 : kRescaleThreshold;
      constexpr float kPOff = F8S ? kPScaleLog2E4M3 : 0.f;  // P is emitted as 2^kPOff * exp2(s - m)
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; ok && j < nk; ++j) {
        if (!warp_wait(bar(BAR_SFULL + x), (sc + j) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        if constexpr (HALF) {
          // the thread's half of the tile row: keys 64 kh + [0, 32) in v0, 64 kh + [32, 64) in v1
          uint32_t v0[32], v1[32];
          tc::tmem_ld16x2_x32_async<64>(tS + 0, v0);
          tc::tmem_ld16x2_x32_async<64>(tS + 32, v1);
          tc::tmem_wait_ld_dep(v0);
          tc::reg_dep(v1);
          const int tb = kt0 + (2 * j + x) * kCtxTileN;  // key of column 0
          if (__any_sync(0xffffffffu, tb + kCtxTileN > kend || tb + kCtxTileN > past)) {
            auto low = [](int c) { return c >= 32 ? 0xffffffffu : (c <= 0 ? 0u : (1u << c) - 1u); };
            auto word = [&](int wd) {
              const int t0 = tb + 32 * wd, sh = t0 - past;
              uint32_t nv = 0u;
              if (sh >= 0) nv = sh < 64 ? static_cast<uint32_t>(vis >> sh) : 0u;
              else if (sh > -32) nv = static_cast<uint32_t>(vis << (-sh));
              return (low(past - t0) | nv) & low(kend - t0);
            };
            const uint32_t m0 = word(2 * kh), m1 = word(2 * kh + 1);
            const uint32_t all = 0xffffffffu;
            if (__any_sync(all, m0 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v0[e] = (m0 >> e) & 1u ? v0[e] : __float_as_uint(-INFINITY);
            }
            if (__any_sync(all, m1 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v1[e] = (m1 >> e) & 1u ? v1[e] : __float_as_uint(-INFINITY);
            }
          }
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            mx0 = max3f(mx0, __uint_as_float(v0[e]), __uint_as_float(v0[e + 1]));
            mx1 = max3f(mx1, __uint_as_float(v1[e]), __uint_as_float(v1[e + 1]));
          }
          float mt = fmaxf(mx0, mx1);
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the row's other half
          const float m_new = fmaxf(m_run, mt * sl2);
          float m_use = m_run;
          if (j == 0) {
            m_use = m_new;  // O is still empty
          } else if (__any_sync(0xffffffffu, m_new > m_run + kThr)) {
            // each thread rescales its half of the row's O columns
            const float f = ex2_approx(m_run - m_new);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
              uint32_t o[32];
              tc::tmem_ld16x2_x32_async<D / 2>(tO + cc * 32, o);
              tc::tmem_wait_ld_dep(o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              tc::tmem_st16x2_x32<D / 2>(tO + cc * 32, o);
            }
            l_run *= f;
            m_use = m_new;
          }
          m_run = m_use;
          // P pairs of keys 64 kh + [0, 64) into S columns 32 kh + [0, 32) of the shared lane
          // (E4M3: hi codes of the keys into columns 16 kh + [0, 16), lo codes 32 further on)
          float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          const float m_base = m_use == -INFINITY ? 0.f : m_use;
          const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(kPOff - m_base, kPOff - m_base);
          if constexpr (F8S) {
            uint32_t hw[16], lw[16];
            emit_e4m3(v0, ls[0], hw, lw, 0, sl2x2, negm);
            emit_e4m3(v1, ls[1], hw, lw, 8, sl2x2, negm);
            tc::tmem_st16x2_x16<16>(tS + 0, hw);
            tc::tmem_st16x2_x16<16>(tS + 32, lw);
          }
          auto emit = [&](uint32_t(&v)[32], int c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 xa = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2, negm);
              const float2 pv = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
              ls[c] = fadd2(ls[c], pv);
              pk[e >> 1] = Q8 ? pack_f16x2(pv.x, pv.y) : pack_bf16x2(pv.x, pv.y);
            }
            tc::tmem_st16x2_x16<32>(tS + 16 * c, pk);
          };
          if constexpr (!F8S) {
            emit(v0, 0);
            emit(v1, 1);
          }
          const float2 lsum = fadd2(ls[0], ls[1]);
          l_run += lsum.x + lsum.y;  // this thread's half; the pair's halves are added at the end
          tc::tmem_wait_st();
        } else {
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tc::tmem_ld32_async(tS + 0, v0);
          tc::tmem_ld32_async(tS + 32, v1);
          tc::tmem_ld32_async(tS + 64, v2);
          tc::tmem_ld32_async(tS + 96, v3);
          tc::tmem_wait_ld_dep(v0);
          tc::reg_dep(v1);
          tc::reg_dep(v2);
          tc::reg_dep(v3);
          const int tb = kt0 + (2 * j + x) * kCtxTileN;  // key of column 0
          if (__any_sync(0xffffffffu, tb + kCtxTileN > kend || tb + kCtxTileN > past)) {
            // visibility of columns 32w .. 32w+31 as one word: cached keys (t < past), the new
            // keys this row's token sees (bits of vis), nothing at or past the split's end
            auto low = [](int c) { return c >= 32 ? 0xffffffffu : (c <= 0 ? 0u : (1u << c) - 1u); };
            auto word = [&](int wd) {
              const int t0 = tb + 32 * wd, sh = t0 - past;
              uint32_t nv = 0u;
              if (sh >= 0) nv = sh < 64 ? static_cast<uint32_t>(vis >> sh) : 0u;
              else if (sh > -32) nv = static_cast<uint32_t>(vis << (-sh));
              return (low(past - t0) | nv) & low(kend - t0);
            };
            // a select per key only in the words where some row misses some key
            const uint32_t m0 = word(0), m1 = word(1), m2 = word(2), m3 = word(3);
            const uint32_t all = 0xffffffffu;
            if (__any_sync(all, m0 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v0[e] = (m0 >> e) & 1u ? v0[e] : __float_as_uint(-INFINITY);
            }
            if (__any_sync(all, m1 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v1[e] = (m1 >> e) & 1u ? v1[e] : __float_as_uint(-INFINITY);
            }
            if (__any_sync(all, m2 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v2[e] = (m2 >> e) & 1u ? v2[e] : __float_as_uint(-INFINITY);
            }
            if (__any_sync(all, m3 != all)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) v3[e] = (m3 >> e) & 1u ? v3[e] : __float_as_uint(-INFINITY);
            }
          }
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            mx[0] = max3f(mx[0], __uint_as_float(v0[e]), __uint_as_float(v0[e + 1]));
            mx[1] = max3f(mx[1], __uint_as_float(v1[e]), __uint_as_float(v1[e + 1]));
            mx[2] = max3f(mx[2], __uint_as_float(v2[e]), __uint_as_float(v2[e + 1]));
            mx[3] = max3f(mx[3], __uint_as_float(v3[e]), __uint_as_float(v3[e + 1]));
          }
          const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2);
          float m_use = m_run;
          if (j == 0) {
            m_use = m_new;  // O is still empty
          } else if (__any_sync(0xffffffffu, m_new > m_run + kThr)) {
            // PV_x(j-1) completed before S_x(j) was signalled; rescale O (whole warp, per-row factor)
            const float f = ex2_approx(m_run - m_new);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t o[32];
              tc::tmem_ld32(tO + cc * 32, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              tc::tmem_st32(tO + cc * 32, o);
            }
            l_run *= f;
            m_use = m_new;
          }
          m_run = m_use;
          // P = exp2(s * scale_log2 - m) as bf16 pairs into S columns 0..63 (keys 2c, 2c+1 in column c)
          float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          const float m_base = m_use == -INFINITY ? 0.f : m_use;  // no visible key yet (generation splits)
          const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(kPOff - m_base, kPOff - m_base);
          if constexpr (F8S) {  // E4M3: hi codes of keys 4c .. 4c+3 in column c, lo codes in 32 + c
            uint32_t hw[16], lw[16];
            emit_e4m3(v0, ls[0], hw, lw, 0, sl2x2, negm);
            emit_e4m3(v1, ls[1], hw, lw, 8, sl2x2, negm);
            tc::tmem_st16(tS + 0, hw);
            tc::tmem_st16(tS + 32, lw);
            emit_e4m3(v2, ls[2], hw, lw, 0, sl2x2, negm);
            emit_e4m3(v3, ls[3], hw, lw, 8, sl2x2, negm);
            tc::tmem_st16(tS + 16, hw);
            tc::tmem_st16(tS + 48, lw);
          }
          auto emit = [&](uint32_t(&v)[32], int c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 xa = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2, negm);
              const float2 pv = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
              ls[c] = fadd2(ls[c], pv);
              pk[e >> 1] = Q8 ? pack_f16x2(pv.x, pv.y) : pack_bf16x2(pv.x, pv.y);
            }
            tc::tmem_st16(tS + 16 * c, pk);
          };
          if constexpr (!F8S) {
            emit(v0, 0);
            emit(v1, 1);
            emit(v2, 2);
            emit(v3, 3);
          }
          const float2 lsum = fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3]));
          l_run += lsum.x + lsum.y;
          tc::tmem_wait_st();
        }
        if (F8S && 2 * j + x == nT - 1 && x == zero_x) {
          // E4M3: zero the raw V rows past the end of the split (stale or unloaded slots; a zero
          // P against a NaN code would still poison the row) before its PV
          const int g = G + nT - 1;
          if (!warp_wait(bar(BAR_RAWV + rstg(g)), rphs(g))) { ok = false; break; }
          if (kt0 + (nT - 1) * kCtxTileN + row >= kend) {
            uint4* vrow = reinterpret_cast<uint4*>(base + L::kRawVOff + rstg(g) * L::kRawTile + row * 128);
#pragma unroll
            for (int kq = 0; kq < 8; ++kq) vrow[kq] = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_proxy_async_smem();
        }
        if (!Q8 && 2 * j + x == nT - 1 && x == zero_x) {
          // zero V rows past the end of the sequence (stale or unloaded slots) before any PV (an
          // 8-bit pool's conversion writes them as zeros)
          const int g = G + nT - 1;
          if (!warp_wait(bar(BAR_VFULL + stg(g)), phs(g))) { ok = false; break; }
          if (kt0 + (nT - 1) * kCtxTileN + row >= kend) {
            uint8_t* vrow = base + (sV(stg(g)) - base_s) + row * 128;
#pragma unroll
            for (int dh = 0; dh < D / 64; ++dh)
#pragma unroll
              for (int kq = 0; kq < 8; ++kq)
                reinterpret_cast<uint4*>(vrow + dh * L::kHalf)[kq] = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_proxy_async_smem();
        }
        // one arrive per warp after the warp has synchronised (fewer atomics on one word)
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_PFULL + x));
        if constexpr (Q8 && !F8S) {  // the warpgroup's next tile, while its PV and the other tile's MMAs run
          if (j + 1 < nk && !convert_tile(gtile(j + 1), kend - (kt0 + (2 * j + 2 + x) * kCtxTileN))) { ok = false; break; }
        }
      }
      if (!ok) break;
      // ---- epilogue: the two halves of the split's keys: B hands its (m, l) over through
      // shared memory and A merges O_A and O_B from TMEM into the output row or a partial row ----
      if (nk > 0) {
        if (warp_abort() || !warp_wait(bar(BAR_ODONE + x), n_epi & 1)) { ok = false; break; }
        ++n_epi;
        tc::fence_after_sync();
        // HALF: the row's sum is its two threads' halves added (both hold the same running max)
        const float l_row = HALF ? l_run + __shfl_xor_sync(0xffffffffu, l_run, 16) : l_run;
        if (x == 1) {
          if (kh == 0) {
            xch[qrow] = m_run;
            xch[128 + qrow] = l_row;
          }
          tc::mbar_arrive(bar(BAR_MERGE));
        } else {
          float mB = -INFINITY, lB = 0.f;
          if (it.nkt1 > 0) {
            if (!warp_wait(bar(BAR_MERGE), n_merge & 1)) { ok = false; break; }
            tc::fence_after_sync();
            mB = xch[qrow];
            lB = xch[128 + qrow];
          }
          const float M = fmaxf(m_run, mB), Mb = M == -INFINITY ? 0.f : M;
          const float fA = ex2_approx(m_run - Mb), fB = ex2_approx(mB - Mb);
          const float l = fA * l_row + fB * lB;
          const bool store = qrow < nvx;
          const int64_t head = static_cast<int64_t>(it.hk) * p.group + hl;
          const bool whole = it.num_splits == 1;  // else a partial result for the combine
          const float osc = p.out_scale;
          const float sA = whole ? fA * osc / l : fA * osc;
          const float sB = whole ? fB * osc / l : fB * osc;
          uint16_t* orow = p.out + static_cast<int64_t>(it.tok0 + tok_i) * p.out_stride + head * D;
          const int64_t pi = (static_cast<int64_t>(__ldg(p.part_prefix + it.gr)) +
                              static_cast<int64_t>(it.s_idx) * it.n_new + tok_i) * p.Hq + head;
          float* prow = p.part_o + pi * D;
          // HALF: each of the row's two threads takes D / 2 of its output columns
          constexpr int kChunks = HALF ? D / 64 : D / 32;
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc) {
            uint32_t va[32], vb[32];
            if constexpr (HALF) {
              tc::tmem_ld16x2_x32_async<D / 2>(tO + cc * 32, va);
              tc::tmem_wait_ld_dep(va);
            } else {
              tc::tmem_ld32(tO + cc * 32, va);
            }
            if (it.nkt1 > 0) {  // O_B, same lanes
              if constexpr (HALF) {
                tc::tmem_ld16x2_x32_async<D / 2>(tO + 128 + cc * 32, vb);
                tc::tmem_wait_ld_dep(vb);
              } else {
                tc::tmem_ld32(tO + 128 + cc * 32, vb);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) vb[e] = 0u;
            }
            const int c0 = kh * (D / 2) + cc * 32;  // output column of o[0]
            float o[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(va[e]) * sA + __uint_as_float(vb[e]) * sB;
            if (store && whole) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(o[e], o[e + 1]);
#pragma unroll
              for (int kq = 0; kq < 4; ++kq)
                reinterpret_cast<uint4*>(orow + c0)[kq] =
                    make_uint4(pk[4 * kq], pk[4 * kq + 1], pk[4 * kq + 2], pk[4 * kq + 3]);
            } else if (store) {
#pragma unroll
              for (int kq = 0; kq < 8; ++kq)
                reinterpret_cast<float4*>(prow + c0)[kq] =
                    make_float4(o[4 * kq], o[4 * kq + 1], o[4 * kq + 2], o[4 * kq + 3]);
            }
          }
          if (store && !whole && kh == 0) {
            p.part_ml[pi * 2] = M;
            p.part_ml[pi * 2 + 1] = l;
          }
        }
      }
      if (it.nkt1 > 0) ++n_merge;
      G += nT;
      sc += nk;
      item_done();
      ++ndone;
    }
    if (!ok) fail();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- context attention: one CTA per SM walks a queue of (unit, query head) items ----
// A CTA keeps its TMEM, barriers and rings across items, so one item's fill and drain overlap
// its neighbours:
//   - the producer claims the next item (an atomic cursor the plan zeroes) as soon as it has
//     issued the current item's last K / V tile, publishes it through a two-entry ring in
//     shared memory, and loads the next Q tile into a slot as soon as the slot's last S MMA is
//     done and the next K / V tiles as soon as stages free up;
//   - the producer publishes each item with its unit descriptor (read while the previous
//     item's tiles were still in flight), so no consumer waits on a global load between items;
//   - the MMA warp goes from the last PV of one item straight to the first S of the next;
//   - output tiles leave through their own staging tile (one, handed from epilogue to epilogue
//     in order), so a Q slot never waits for an output store.
// The ring counters (K / V stream tile, S / P tile per Q tile, Q loads per slot) run on across
// items; every phase is derived from them.  Items are claimed longest unit first, as the plan
// sorted them.
template <int D>
struct CtxSmem {
  static constexpr int kHalf = 128 * 128;
  static constexpr int kTile = (D / 64) * kHalf;
  static constexpr int kStages = 2;
  static constexpr int kQOff = 0;                          // Q_A, Q_B
  static constexpr int kKOff = 2 * kTile;                  // K ring
  static constexpr int kVOff = kKOff + kStages * kTile;    // V ring
  static constexpr int kOOff = kVOff + kStages * kTile;    // output staging tile
  static constexpr int kBarOff = kOOff + kTile;
  static constexpr int kBarBytes = 512;
  static constexpr int kBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

enum {
  PB_Q = 0,          // +2: Q tile of slot x landed
  PB_QFREE = 2,      // +2: the last S MMA on slot x is done (the slot may be refilled)
  PB_KFULL = 4,      // +2 stages
  PB_KEMPTY = 6,     // +2
  PB_VFULL = 8,      // +2
  PB_VEMPTY = 10,    // +2
  PB_SFULL = 12,     // +2 Q tiles
  PB_PFULL = 14,     // +2
  PB_ODONE = 16,     // +2
  PB_ITEM = 18,      // +2: item ring entry written
  PB_ITEMFREE = 20,  // +2: item ring entry read by the MMA warp and the eight softmax warps
  PB_OSTG = 22,      // the staging tile's last store has been read out
  PB_OWRITTEN = 23,  // +2: the four warps of Q tile x have written the staging tile
  PB_MMADONE = 25,
  PB_NUM = 26
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
context_attn_kernel(const ContextParams p, const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap out_map) {
  using L = CtxSmem<D>;
  constexpr int S = L::kStages;
  static_assert(S == 2, "ring stage and phase below are bit operations");
  // ring stage and phase of the g-th K / V tile of the stream (g >= 0)
  auto stg = [](int g) { return g & 1; };
  auto phs = [](int g) { return (g >> 1) & 1; };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  const uint32_t bar0 = base_s + L::kBarOff;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + L::kBarOff + 8 * PB_NUM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kBarOff + 8 * PB_NUM + 4);
  // item ring: [2][8] ints, entry = item index (-1: no more work) and the unit's descriptor
  volatile int* s_item = reinterpret_cast<volatile int*>(base + L::kBarOff + 8 * PB_NUM + 16);
  static_assert(8 * PB_NUM + 16 + 2 * 8 * 4 <= L::kBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up (before the grid-dependency wait: reads nothing earlier kernels write) ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar(PB_Q + s), 1);
      tc::mbar_init(bar(PB_QFREE + s), 1);
      tc::mbar_init(bar(PB_KFULL + s), 1);
      tc::mbar_init(bar(PB_KEMPTY + s), 1);
      tc::mbar_init(bar(PB_VFULL + s), 1);
      tc::mbar_init(bar(PB_VEMPTY + s), 1);
      tc::mbar_init(bar(PB_SFULL + s), 1);
      tc::mbar_init(bar(PB_PFULL + s), 4);  // one arrive per softmax warp
      tc::mbar_init(bar(PB_ODONE + s), 1);
      tc::mbar_init(bar(PB_ITEM + s), 1);
      tc::mbar_init(bar(PB_ITEMFREE + s), 9);  // the MMA warp and the eight softmax warps
      tc::mbar_init(bar(PB_OWRITTEN + s), 4);
    }
    tc::mbar_init(bar(PB_OSTG), 1);
    tc::mbar_init(bar(PB_MMADONE), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(base_s + L::kBarOff + 8 * PB_NUM, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tc::prefetch_tmap(&q_map);
    tc::prefetch_tmap(&kv_map);
    tc::prefetch_tmap(&out_map);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  pdl_wait();

  const int n_items = __ldg(p.counts + kCntUnits) * p.Hq;
  // CTAs that take work: the grid, or fewer when the plan leaves SMs to the generation kernels
  // running beside this one (the others go straight to the teardown)
  const int active = min(static_cast<int>(gridDim.x), __ldg(p.counts + kCntCtxCtas));
  // An item: query head hq of unit y (the plan's descriptor: request, first q row, key position
  // of that row, rows of the request from there on).  Every role derives the same geometry.
  struct Item {
    int hq, hk, r, q_row, past, L_r, nv0, nv1, nkt0, nkt1, nT;
    bool ok, hasB, fullA, fullB;
  };
  auto item_of = [&](int w, const int4 u) {
    Item it;
    const int y = w / p.Hq;
    it.hq = w - y * p.Hq;
    it.hk = it.hq / p.group;
    it.r = u.x;
    it.q_row = u.y;
    it.past = u.z;
    const int n_rem = u.w;
    it.L_r = it.past + n_rem;
    it.nv0 = max(0, min(128, n_rem));
    it.nv1 = max(0, min(128, n_rem - 128));
    it.nkt0 = it.nv0 > 0 ? (it.past + it.nv0 + kCtxTileN - 1) / kCtxTileN : 0;
    it.nkt1 = it.nv1 > 0 ? (it.past + 128 + it.nv1 + kCtxTileN - 1) / kCtxTileN : 0;
    it.ok = it.nv0 > 0 && it.r >= 0 && it.r < p.C && it.past >= 0 && it.q_row >= 0 && it.q_row + it.nv0 + it.nv1 <= p.T;
    it.hasB = it.nv1 > 0;
    it.nT = it.ok ? (it.hasB ? it.nkt1 : it.nkt0) : 0;
    // full output tiles leave through the staging tile and a TMA store, A before B
    it.fullA = it.ok && it.nv0 == 128 && it.q_row + 128 <= p.T;
    it.fullB = it.ok && it.nv1 == 128 && it.q_row + 256 <= p.T;
    return it;
  };

  const uint32_t sQ = base_s + L::kQOff;
  const uint32_t sO = base_s + L::kOOff;
  auto sK = [&](int st) { return base_s + L::kKOff + st * L::kTile; };
  auto sV = [&](int st) { return base_s + L::kVOff + st * L::kTile; };
  auto fail = [&]() {
    flag_error(p.d_error, PKV_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };
  auto warp_wait = [&](uint32_t b, uint32_t parity) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b, parity)) != 0;
  };
  auto warp_abort = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0) != 0; };
  // consumers: item k of this CTA from the ring (-1: no more work), entry handed back
  auto take_item = [&](int k, int& w, int4& u) {
    const int slot = k & 1;
    if (!warp_wait(bar(PB_ITEM + slot), (k >> 1) & 1)) return false;
    const volatile int* e = s_item + 8 * slot;
    w = e[0];
    u = make_int4(e[1], e[2], e[3], e[4]);
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(PB_ITEMFREE + slot));
    return true;
  };

  if (warp >= 8) {
    tc::regs_dec<kRegsControl>();
    if (warp == kProducerWarp) {
      // ======================= item queue + TMA producer =======================
      int w = static_cast<int>(blockIdx.x) < active ? static_cast<int>(blockIdx.x) : n_items;
      // the first unit's descriptor, loaded beside the item count (in bounds: the grid has at
      // most num_tiles x Hq CTAs and unit_info num_tiles entries; unused past the item count)
      int4 u = __ldg(p.unit_info + static_cast<int>(blockIdx.x) / p.Hq);
      int issued_k = 0, issued_v = 0;  // K / V stream tiles issued (all items)
      int nq0 = 0, nq1 = 0;            // Q loads per slot
      bool pok = true;
      for (int k = 0; pok; ++k) {
        const int slot = k & 1;
        if (k >= 2 && !warp_wait(bar(PB_ITEMFREE + slot), ((k - 2) >> 1) & 1)) { pok = false; break; }
        const bool more = w < n_items;
        if (lane == 0) {
          volatile int* e = s_item + 8 * slot;
          e[0] = more ? w : -1;
          e[1] = u.x;
          e[2] = u.y;
          e[3] = u.z;
          e[4] = u.w;
          tc::mbar_arrive(bar(PB_ITEM + slot));
        }
        __syncwarp();
        if (!more) break;
        const Item it = item_of(w, u);
        if (!it.ok) {
          if (lane == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);  // plan disagrees
        } else {
          // Q tiles: slot x once its previous item's last S MMA is done
          for (int x = 0; x < (it.hasB ? 2 : 1); ++x) {
            const int n = x ? nq1 : nq0;
            if (n > 0 && !warp_wait(bar(PB_QFREE + x), (n - 1) & 1)) { pok = false; break; }
            if (tc::elect_one()) {
              tc::mbar_arrive_expect_tx(bar(PB_Q + x), 128 * D * 2);
              for (int dh = 0; dh < D / 64; ++dh)
                tc::tma_load_4d(sQ + x * L::kTile + dh * L::kHalf, &q_map, bar(PB_Q + x), 0, dh, it.hq,
                                it.q_row + 128 * x);
            }
            __syncwarp();
            if (x) ++nq1; else ++nq0;
          }
          const int32_t* tbl = p.tbl + static_cast<int64_t>(it.r) * p.max_blocks;
          const int box_rows = p.B < kCtxTileN ? p.B : kCtxTileN;
          const int pages_per_tile = kCtxTileN / box_rows;  // <= 8 (B >= 16)
          const int n_pages_seq = (it.L_r + p.B - 1) / p.B;
#ifdef PKV_SELFTEST
          // Self-test build only (compiled by the tests, never into libpaged_kv.so): no K / V
          // copy is issued, so the MMA warp's wait for the first K tile and the softmax warps'
          // waits for their first S run out after the short self-test budget and the CTA winds
          // down through the timeout path; the Q tiles land before the teardown (waited below).
          const int n_issue = 0;
#else
          const int n_issue = it.nT;
#endif
          for (int j = 0; pok && j < n_issue; ++j) {
            if (warp_abort()) { pok = false; break; }
            const int g = issued_k;  // == issued_v
            const int st = stg(g);
            // lane pp < pages_per_tile looks up page pp of the tile (whole pages per tile)
            const int lb = (j * kCtxTileN) / p.B + lane;
            int pg = -1;
            if (lane < pages_per_tile && lb < n_pages_seq && lb < p.max_blocks) {
              pg = __ldg(tbl + lb);
              if (pg < 0 || pg >= p.NB) {
                flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
                pg = -1;
              }
            }
            const uint32_t bytes =
                static_cast<uint32_t>(__popc(__ballot_sync(0xffffffffu, pg >= 0))) * box_rows * D * 2;
            const uint32_t koff = static_cast<uint32_t>(lane * box_rows * 128);
            if (g >= S && !warp_wait(bar(PB_KEMPTY + st), phs(g - S))) { pok = false; break; }
            if (lane == 0) tc::mbar_arrive_expect_tx(bar(PB_KFULL + st), bytes);
            __syncwarp();
            if (pg >= 0)
              for (int dh = 0; dh < D / 64; ++dh)
                tc::tma_load_4d(sK(st) + dh * L::kHalf + koff, &kv_map, bar(PB_KFULL + st), 0, dh, it.hk,
                                (pg * 2 + 0) * p.B);
            __syncwarp();
            ++issued_k;
            if (g >= S && !warp_wait(bar(PB_VEMPTY + st), phs(g - S))) { pok = false; break; }
            if (lane == 0) tc::mbar_arrive_expect_tx(bar(PB_VFULL + st), bytes);
            __syncwarp();
            if (pg >= 0)
              for (int dh = 0; dh < D / 64; ++dh)
                tc::tma_load_4d(sV(st) + dh * L::kHalf + koff, &kv_map, bar(PB_VFULL + st), 0, dh, it.hk,
                                (pg * 2 + 1) * p.B);
            __syncwarp();
            ++issued_v;
          }
        }
        if (!pok) break;
        // claim the next item while this one's tiles are still being consumed
        int nxt = 0;
        if (lane == 0) nxt = atomicAdd(p.cursor, 1) + active;
        w = __shfl_sync(0xffffffffu, nxt, 0);
        if (w < n_items) u = __ldg(p.unit_info + w / p.Hq);  // before the ring slot frees up
      }
      if (!pok && lane == 0) fail();
      __syncwarp();
      // the last copy into each stage and slot has landed before the CTA can wind down, however
      // the consumers fare (on the normal path these phases completed long ago)
      for (int j = (issued_k > S ? issued_k - S : 0); j < issued_k; ++j)
        tc::mbar_wait(bar(PB_KFULL + stg(j)), phs(j), 200000000LL);
      for (int j = (issued_v > S ? issued_v - S : 0); j < issued_v; ++j)
        tc::mbar_wait(bar(PB_VFULL + stg(j)), phs(j), 200000000LL);
      if (nq0 > 0) tc::mbar_wait(bar(PB_Q + 0), (nq0 - 1) & 1, 200000000LL);
      if (nq1 > 0) tc::mbar_wait(bar(PB_Q + 1), (nq1 - 1) & 1, 200000000LL);
    } else if (warp == kMmaWarp) {
      // ======================= MMA issuer =======================
      constexpr uint32_t idesc_s = tc::idesc_bf16(128, kCtxTileN, 0);
      constexpr uint32_t idesc_o = tc::idesc_bf16(128, D, 1);
      const uint64_t dq0 = tc::sdesc_sw128(sQ, 16, 1024);
      const uint64_t dq1 = tc::sdesc_sw128(sQ + L::kTile, 16, 1024);
      const uint64_t dk0 = tc::sdesc_sw128(sK(0), 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(sV(0), L::kHalf, 1024);
      auto stage_off = [](int st) { return static_cast<uint64_t>(st) * (L::kTile / 16); };
      int G = 0;               // K / V stream tiles of earlier items
      int sc0 = 0, sc1 = 0;    // S / P tiles of earlier items, per Q tile
      int nq0 = 0, nq1 = 0;    // Q loads consumed per slot
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int w = -1;
        int4 u;
        if (!take_item(k, w, u)) { ok = false; break; }
        if (w < 0) break;
        const Item it = item_of(w, u);
        if (!it.ok) continue;
        auto uses = [&](int j, int x) { return j < (x ? it.nkt1 : it.nkt0); };
        auto frees = [&](int j, int x) { return x == ((it.hasB && j < it.nkt1) ? 1 : 0); };
        auto issue_s = [&](int j, int x) {
          const int st = stg(G + j);
          const uint64_t a0 = x == 0 ? dq0 : dq1;
          const uint64_t b0 = dk0 + stage_off(st);
          if (tc::elect_one()) {
            if constexpr (D == 128) {
              tc::mma_bf16_ss_x8<0, 2, 4, 6, L::kHalf / 16, L::kHalf / 16 + 2, L::kHalf / 16 + 4, L::kHalf / 16 + 6>(
                  tmem + 128 * x, a0, b0, idesc_s, 0u);
            } else {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4);
                tc::mma_bf16_ss(tmem + 128 * x, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u);
              }
            }
            tc::mma_commit(bar(PB_SFULL + x));
            if (frees(j, x)) tc::mma_commit(bar(PB_KEMPTY + st));
            if (j == (x ? it.nkt1 : it.nkt0) - 1) tc::mma_commit(bar(PB_QFREE + x));  // the slot's last S
          }
          __syncwarp();
        };
        // first S of each Q tile: its Q tile and the item's first K tile
        ok = warp_wait(bar(PB_Q + 0), nq0 & 1) && warp_wait(bar(PB_KFULL + stg(G)), phs(G));
        ++nq0;
        if (ok) {
          tc::fence_after_sync();
          issue_s(0, 0);
          if (it.hasB) {
            ok = warp_wait(bar(PB_Q + 1), nq1 & 1);
            ++nq1;
            if (ok) {
              tc::fence_after_sync();
              issue_s(0, 1);
            }
          }
        }
        for (int j = 0; ok && j < it.nT; ++j) {
          bool v_ready = false, k_ready = false;  // B reuses the tiles A waited for
          const int g = G + j;
          for (int x = 0; x < 2 && ok; ++x) {
            if (!uses(j, x)) continue;
            if (!warp_wait(bar(PB_PFULL + x), ((x ? sc1 : sc0) + j) & 1)) { ok = false; break; }
            if (!v_ready) {
              if (!warp_wait(bar(PB_VFULL + stg(g)), phs(g))) { ok = false; break; }
              v_ready = true;
            }
            tc::fence_after_sync();
            const uint64_t v0 = dv0 + stage_off(stg(g));
            if (tc::elect_one()) {
              static_assert(kCtxTileN == 128, "eight K=16 steps per KV tile");
              tc::mma_bf16_ts_x8<16 * 128 / 16>(tmem + 256 + 128 * x, tmem + 128 * x, v0, idesc_o, j > 0 ? 1u : 0u);
              if (frees(j, x)) tc::mma_commit(bar(PB_VEMPTY + stg(g)));
              if (j == (x ? it.nkt1 : it.nkt0) - 1) tc::mma_commit(bar(PB_ODONE + x));
            }
            __syncwarp();
            if (uses(j + 1, x)) {
              if (!k_ready && !warp_wait(bar(PB_KFULL + stg(g + 1)), phs(g + 1))) { ok = false; break; }
              k_ready = true;
              tc::fence_after_sync();
              issue_s(j + 1, x);
            }
          }
        }
        G += it.nT;
        sc0 += it.nkt0;
        if (it.hasB) sc1 += it.nkt1;
      }
      if (!ok && lane == 0) fail();
      if (tc::elect_one()) {
        tc::mma_commit(bar(PB_MMADONE));
        tc::mbar_wait(bar(PB_MMADONE), 0, 200000000LL);  // nothing of ours still runs on TMEM
      }
      __syncwarp();
    }
  } else {
    // ======================= softmax warpgroups =======================
    tc::regs_inc<kRegsSoftmax>();
    const int x = warp >> 2;                 // Q tile A (0) or B (1)
    const int row = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128 * x + lane_off;
    const uint32_t tO = tmem + 256 + 128 * x + lane_off;
    const float sl2 = p.scale_log2;
    int G = 0, sc = 0, n_epi = 0;  // stream tiles, this tile's S / P tiles and epilogues so far
    int n_stg = 0, n_own = 0;      // staging-tile uses so far (both Q tiles), and this tile's own
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int w = -1;
      int4 u;
      if (!take_item(k, w, u)) { ok = false; break; }
      if (w < 0) break;
      const Item it = item_of(w, u);
      if (!it.ok) continue;
      const int nvx = x ? it.nv1 : it.nv0, nk = x ? it.nkt1 : it.nkt0;
      const int stg_idx = n_stg + (x ? (it.fullA ? 1 : 0) : 0);  // A's store goes first
      const bool full = x ? it.fullB : it.fullA;
      const int zero_x = (it.nkt0 == it.nT) ? 0 : 1;  // first user of the last V tile zeroes its tail
      const int q_pos = it.past + 128 * x + min(row, max(nvx, 1) - 1);  // padding rows mirror the last row
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; ok && j < nk; ++j) {
        if (!warp_wait(bar(PB_SFULL + x), (sc + j) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        uint32_t v0[32], v1[32], v2[32], v3[32];
        tc::tmem_ld32_async(tS + 0, v0);
        tc::tmem_ld32_async(tS + 32, v1);
        tc::tmem_ld32_async(tS + 64, v2);
        tc::tmem_ld32_async(tS + 96, v3);
        tc::tmem_wait_ld_dep(v0);
        tc::reg_dep(v1);
        tc::reg_dep(v2);
        tc::reg_dep(v3);
        const int lim = q_pos - j * kCtxTileN;  // key column c is visible iff c <= lim
        if (__any_sync(0xffffffffu, lim < kCtxTileN - 1)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            v0[e] = e <= lim ? v0[e] : __float_as_uint(-INFINITY);
            v1[e] = 32 + e <= lim ? v1[e] : __float_as_uint(-INFINITY);
            v2[e] = 64 + e <= lim ? v2[e] : __float_as_uint(-INFINITY);
            v3[e] = 96 + e <= lim ? v3[e] : __float_as_uint(-INFINITY);
          }
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          mx[0] = max3f(mx[0], __uint_as_float(v0[e]), __uint_as_float(v0[e + 1]));
          mx[1] = max3f(mx[1], __uint_as_float(v1[e]), __uint_as_float(v1[e + 1]));
          mx[2] = max3f(mx[2], __uint_as_float(v2[e]), __uint_as_float(v2[e + 1]));
          mx[3] = max3f(mx[3], __uint_as_float(v3[e]), __uint_as_float(v3[e + 1]));
        }
        const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2);
        float m_use = m_run;
        if (j == 0) {
          m_use = m_new;  // O is still empty
        } else if (__any_sync(0xffffffffu, m_new > m_run + kRescaleThreshold)) {
          const float f = ex2_approx(m_run - m_new);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tc::tmem_ld32(tO + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tc::tmem_st32(tO + cc * 32, o);
          }
          l_run *= f;
          m_use = m_new;
        }
        m_run = m_use;
        float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float m_base = m_use == -INFINITY ? 0.f : m_use;
        const float2 sl2x2 = make_float2(sl2, sl2), negm = make_float2(-m_base, -m_base);
        auto emit = [&](uint32_t(&v)[32], int c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 xa = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl2x2, negm);
            const float2 pv = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
            ls[c] = fadd2(ls[c], pv);
            pk[e >> 1] = pack_bf16x2(pv.x, pv.y);
          }
          tc::tmem_st16(tS + 16 * c, pk);
        };
        emit(v0, 0);
        emit(v1, 1);
        emit(v2, 2);
        emit(v3, 3);
        const float2 lsum = fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3]));
        l_run += lsum.x + lsum.y;
        tc::tmem_wait_st();
        if (j == it.nT - 1 && x == zero_x) {
          // zero V rows past the end of the sequence (stale or unloaded slots) before any PV
          const int g = G + it.nT - 1;
          if (!warp_wait(bar(PB_VFULL + stg(g)), phs(g))) { ok = false; break; }
          if (j * kCtxTileN + row >= it.L_r) {
            uint8_t* vrow = base + (sV(stg(g)) - base_s) + row * 128;
#pragma unroll
            for (int dh = 0; dh < D / 64; ++dh)
#pragma unroll
              for (int kq = 0; kq < 8; ++kq)
                reinterpret_cast<uint4*>(vrow + dh * L::kHalf)[kq] = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(PB_PFULL + x));
      }
      if (!ok) break;
      if (nk > 0) {
        // ---- epilogue: O / l -> bf16 row ----
        if (!warp_wait(bar(PB_ODONE + x), n_epi & 1)) { ok = false; break; }
        ++n_epi;
        tc::fence_after_sync();
        const float inv_l = p.out_scale / l_run;
        // (the next item's first PV on this tile comes after this warp's next P-ready arrive,
        // which follows these TMEM loads in program order)
        if (full) {
          // the staging tile, once the previous store from it has been read out
          if (stg_idx > 0 && !warp_wait(bar(PB_OSTG), (stg_idx - 1) & 1)) { ok = false; break; }
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t v[32];
            tc::tmem_ld32(tO + cc * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              pk[e >> 1] = pack_bf16x2(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
            // 128-byte swizzle of the TMA box: 16-byte chunk c of row r sits at chunk c ^ (r % 8)
            const uint32_t rbase = sO + (cc >> 1) * L::kHalf + row * 128;
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
              const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + kq) ^ static_cast<uint32_t>(row & 7);
              st_shared_v4(rbase + chunk * 16, pk[4 * kq], pk[4 * kq + 1], pk[4 * kq + 2], pk[4 * kq + 3]);
            }
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(PB_OWRITTEN + x));
          if ((warp & 3) == 0) {
            // one thread stores the tile once its four warps have written it, waits for the
            // read-out and hands the staging tile on
            if (!warp_wait(bar(PB_OWRITTEN + x), n_own & 1)) { ok = false; break; }
            if (lane == 0) {
              for (int dh = 0; dh < D / 64; ++dh)
                tc::tma_store_4d(&out_map, sO + dh * L::kHalf, 0, dh, it.hq, it.q_row + 128 * x);
              tc::bulk_commit();
              tc::bulk_wait_read0();
              tc::mbar_arrive(bar(PB_OSTG));
            }
            __syncwarp();
          }
          ++n_own;
        } else {
          // a partial tile (the end of a request, whose next rows belong to another request):
          // per-row stores
          const int grow = it.q_row + 128 * x + row;
          const bool store = row < nvx && grow < p.T;
          uint16_t* orow = p.out + static_cast<int64_t>(grow) * p.out_stride + static_cast<int64_t>(it.hq) * D;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t v[32];
            tc::tmem_ld32(tO + cc * 32, v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              pk[e >> 1] = pack_bf16x2(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l);
            if (store) {
#pragma unroll
              for (int kq = 0; kq < 4; ++kq)
                reinterpret_cast<uint4*>(orow + cc * 32)[kq] =
                    make_uint4(pk[4 * kq], pk[4 * kq + 1], pk[4 * kq + 2], pk[4 * kq + 3]);
            }
          }
        }
      }
      G += it.nT;
      sc += nk;
      n_stg += (it.fullA ? 1 : 0) + (it.fullB ? 1 : 0);
    }
    if (!ok) fail();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- 8-bit pools: stage the context requests' pages as bf16 (exact code values) ----
constexpr int kStageThreads = 256;

template <bool I8>  // false: E4M3 codes, true: int8 codes
__global__ void __launch_bounds__(kStageThreads) stage_q8_kernel(const StageParams p) {
  const int gp = blockIdx.x;  // staging page
  pdl_wait();
  if (gp >= __ldg(p.counts + kCntStagePages)) return;  // past this batch's pages (a bucket's spare CTA)
  int lo = 0, hi = p.C - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.stage_prefix + mid) <= gp) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo, lb = gp - __ldg(p.stage_prefix + r);
  const int n_pages = (__ldg(p.past + r) + __ldg(p.ctx_len + r) + p.B - 1) / p.B;
  if (lb < 0 || lb >= n_pages || lb >= p.max_blocks) {  // plan disagrees with the launch
    if (threadIdx.x == 0) flag_error(p.d_error, PKV_DEVERR_PLAN_MISMATCH);
    return;
  }
  int page = __ldg(p.tbl + static_cast<int64_t>(r) * p.max_blocks + lb);
  const bool ok = page >= 0 && page < p.NB;
  if (threadIdx.x == 0) {
    p.stage_tbl[static_cast<int64_t>(r) * p.max_blocks + lb] = gp;
    if (!ok) flag_error(p.d_error, PKV_DEVERR_BAD_PAGE);
  }
  const int64_t page_elems = static_cast<int64_t>(2) * p.B * p.Hkv * p.D;  // K and V of one page
  const uint4* src = reinterpret_cast<const uint4*>(p.pool + (ok ? page : 0) * page_elems);
  uint4* dst = reinterpret_cast<uint4*>(p.stage_pool + gp * page_elems);
  for (int64_t i = threadIdx.x; i < page_elems / 16; i += kStageThreads) {
    uint4 c = ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (I8) {  // exact: every int8 is a bf16 value (8 significant bits)
          const int c0 = static_cast<int8_t>(w[k] >> (16 * h)), c1 = static_cast<int8_t>(w[k] >> (16 * h + 8));
          o[2 * k + h] = pack_bf16x2(static_cast<float>(c0), static_cast<float>(c1));
        } else {
          const uint32_t h2 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[k] >> (16 * h)));
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          o[2 * k + h] = pack_bf16x2(f.x, f.y);  // exact: every E4M3 value is a bf16 value
        }
      }
    }
    dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_stage_q8(const StageParams& p, cudaStream_t s) {
  if (p.kv_dtype == PKV_INT8) return launch_pdl(stage_q8_kernel<true>, dim3(p.total_pages), dim3(kStageThreads), 0, s, p);
  return launch_pdl(stage_q8_kernel<false>, dim3(p.total_pages), dim3(kStageThreads), 0, s, p);
}

template <int D, int KV>
cudaError_t launch_gen_t(const ContextParams& p, const CUtensorMap& qm, const CUtensorMap& km, cudaStream_t s) {
  auto kern = p.half_rows ? gen_attn_kernel<D, KV, true> : gen_attn_kernel<D, KV, false>;
  constexpr int bytes = GenSmem<D, KV>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  // persistent: at most one CTA per SM, items = (generation CTA of the plan, KV head)
  const int64_t items = static_cast<int64_t>(p.num_titems) * p.Hkv;
  const int grid = static_cast<int>(std::min<int64_t>(items, std::max(p.num_ctas, 1)));
  return launch_pdl(kern, dim3(grid), dim3(kThreads), bytes, s, p, qm, km);
}

template <int D>
cudaError_t launch_context_t(const ContextParams& p, const CUtensorMap& qm, const CUtensorMap& km,
                             const CUtensorMap& om, cudaStream_t s) {
  auto kern = context_attn_kernel<D>;
  constexpr int bytes = CtxSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(p.num_tiles) * p.Hq;
  const int grid = static_cast<int>(std::min<int64_t>(items, std::max(p.num_ctas, 1)));
  return launch_pdl(kern, dim3(grid), dim3(kThreads), bytes, s, p, qm, km, om);
}

cudaError_t launch_context(const ContextParams& p, const void* q_map, const void* kv_map, const void* out_map,
                           cudaStream_t s) {
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(kv_map);
  const CUtensorMap& om = *static_cast<const CUtensorMap*>(out_map);
  return p.D == 128 ? launch_context_t<128>(p, qm, km, om, s) : launch_context_t<64>(p, qm, km, om, s);
}

cudaError_t launch_gen_tc(const ContextParams& p, const void* q_map, const void* kv_map, cudaStream_t s) {
  const CUtensorMap& qm = *static_cast<const CUtensorMap*>(q_map);
  const CUtensorMap& km = *static_cast<const CUtensorMap*>(kv_map);
  if (p.kv_dtype != PKV_BF16) {  // 8-bit codes, converted in shared memory (head_dim 128)
    if (p.D != 128) return cudaErrorInvalidValue;
    return p.kv_dtype == PKV_INT8 ? launch_gen_t<128, PKV_INT8>(p, qm, km, s) : launch_gen_t<128, PKV_FP8_E4M3>(p, qm, km, s);
  }
  return p.D == 128 ? launch_gen_t<128, 0>(p, qm, km, s) : launch_gen_t<64, 0>(p, qm, km, s);
}

}  // namespace pkv
