/*
 * paged_kv.h -- C ABI of the GB300 (sm_103a) paged-KV RoPE + attention library
 * (libpaged_kv.so).
 *
 * One inflight batch per call: requests are packed with no padding, context (prefill or
 * chunked-context) requests first, generation (decode) requests after.  For every new token
 * the library rotates Q and K (GPT-NeoX RoPE), appends K and V into a paged KV pool through
 * each request's block table, and then runs causal GQA self-attention over the pool.
 *
 * Sources (web pages on one LLM serving engine, cited by title and section):
 *   [ARCH]   "TensorRT-LLM 源码完全拆解(一):整体架构与模块全景" (pinghaoyang.com.cn)
 *   [NOTES]  "TensorRT-LLM 1.0 源码学习笔记" (openharmonycrossplatform.csdn.net)
 *   [REPORT] TensorRT-LLM source report at adg.csdn.net/69730cc6
 *
 * Conventions shared by every entry point
 *   - All pointers named d_* and all tensor pointers (q, k, v, q_out, out, pool, rope table,
 *     workspace, error word) are DEVICE pointers; h_* pointers are HOST pointers.
 *   - The caller owns every buffer.  The library allocates no device memory at run time and
 *     keeps no state between calls other than cached device attributes, one auxiliary stream
 *     with two events per device (created on first use, see paged_attention_forward) and --
 *     for paged_attention_forward_noalloc only -- one file-scope device scratch buffer of
 *     PKV_NOALLOC_SCRATCH_BYTES that exists on every GPU loading the library, with its address
 *     cached per device.  No call synchronises a stream: each call only enqueues kernels and
 *     returns, and its effects are ordered on `stream` like one kernel's (same-stream FIFO
 *     ordering as in [NOTES] 五 "完整的推理流程", 5.2 CPU/GPU Overlap).  The kernels are
 *     launched with programmatic stream serialisation; the append kernel signals its dependents
 *     early, so a caller's kernel launched right after it with that attribute may start before
 *     the append ends and must run griddepcontrol.wait before it reads q_out or the pool (an
 *     ordinary launch, an event or a stream wait still sees the call complete).
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* detected on the host before anything
 *     was enqueued.  Errors only the device can see (a page id outside [0, num_blocks), a
 *     bounded wait that ran out) are OR-ed as PKV_DEVERR_* bits into the caller's device int
 *     `d_error`; the offending access is skipped, no kernel traps.  The caller zeroes d_error
 *     and reads it back when it wants to know.
 *   - Tensors are bf16 unless stated otherwise; rows are 16-byte aligned (row strides are in
 *     elements and must be multiples of 8; base pointers 16-byte aligned).
 */
#ifndef PAGED_KV_H_
#define PAGED_KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* == cudaStream_t; NULL = legacy default stream */

/* ---- status codes ----------------------------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARGUMENT (-1) /* NULL pointer, negative or inconsistent count          */
#define PKV_ERR_UNSUPPORTED (-2)      /* head_dim not 64/128, tokens_per_block not 16..128,
                                         Hq not a multiple of Hkv, bad dtype                   */
#define PKV_ERR_BATCH_ORDER (-3)      /* a context request after a generation request, or a
                                         generation request with context_length outside
                                         1 .. PKV_MAX_GEN_TOKENS                               */
#define PKV_ERR_CAPACITY (-4)         /* past + new exceeds max_blocks_per_seq * tokens_per_block
                                         or the RoPE table's max_pos                           */
#define PKV_ERR_ALIGNMENT (-5)        /* pointer or row stride not 16-byte aligned            */
#define PKV_ERR_WORKSPACE (-6)        /* workspace NULL or smaller than the size query said     */
#define PKV_ERR_CUDA (-7)             /* a CUDA runtime/driver call failed (launch, tensor map) */

/* ---- device error bits (OR-ed into *d_error) ---------------------------------------------- */
#define PKV_DEVERR_BAD_PAGE 1u        /* block-table entry outside [0, num_blocks): skipped     */
#define PKV_DEVERR_TIMEOUT 2u         /* a bounded mbarrier / TMA wait gave up                   */
#define PKV_DEVERR_PLAN_MISMATCH 4u   /* device metadata disagrees with the host copies         */
#define PKV_DEVERR_BAD_OFFSET 8u      /* a draft-token position offset outside [0, context_length):
                                         that token is skipped by the append                   */
#define PKV_DEVERR_BUCKET 16u         /* bucket calls: the batch in the device arrays does not
                                         fit its bucket; nothing after the append runs          */

/* Most new tokens one generation request may bring in one step (draft tokens under
 * verification, [REPORT] 1.4 "推测解码技术": spec_decoding_max_generation_length). */
#define PKV_MAX_GEN_TOKENS 64

/* ---- KV-pool element type ([ARCH] "KVCacheManager 的三个对外接口": kv_cache_dtype; [NOTES] 6.4
 * "量化": FP8 and "INT8 KV Cache") ------------------------------------------------------------- */
typedef enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1, PKV_INT8 = 2 } pkv_dtype;

/* ---- request phase ([REPORT] 1.1 host_request_types) --------------------------------------- */
typedef enum { PKV_REQ_CONTEXT = 0, PKV_REQ_GENERATION = 1 } pkv_req_type;

/*
 * One layer's KV pool.  Layout [num_blocks, 2, tokens_per_block, num_kv_heads, head_dim],
 * row-major, K at index 0 and V at index 1 of dim 1 ([ARCH] "KVCacheManager 的三个对外接口",
 * get_buffers).  Element type bf16, or one byte per element (OCP FP8 E4M3 or int8 codes) with
 * one scale for the whole pool ([NOTES] 6.4 "量化": quantise on write with kv_scale_orig_quant,
 * dequantise on read with kv_scale_quant_orig).
 */
typedef struct pkv_pool {
  void* pool;                /* device, 16-byte aligned                                        */
  int32_t dtype;             /* pkv_dtype                                                      */
  int32_t num_blocks;        /* pages in the pool                                              */
  int32_t tokens_per_block;  /* 16, 32, 64 or 128                                               */
  int32_t num_kv_heads;      /* Hkv                                                            */
  int32_t head_dim;          /* D: 64 or 128                                                   */
  float kv_scale_quant_orig; /* 8-bit pools: dequantisation multiplier (value = code * this);
                                ignored for bf16                                               */
  float kv_scale_orig_quant; /* 8-bit pools: quantisation multiplier (code = enc(x * this)),
                                normally (float)(1 / kv_scale_quant_orig); ignored for bf16    */
} pkv_pool;

/*
 * One inflight batch ([ARCH] "AttentionMetadata 的字段与它的含义": seq_lens on host plus
 * seq_lens_cuda on device, context_lens, num_contexts; [REPORT] 1.2 KeyValueCacheParams:
 * host_past_key_value_lengths, kv_cache_block_offsets; [REPORT] 1.3: context requests first).
 * Request r owns packed rows cu_r .. cu_r + context_lengths[r] - 1, cu_r being the sum of
 * context_lengths over earlier requests.  Its KV sequence after this step's append has
 * L_r = past_kv_lengths[r] + context_lengths[r] tokens; token t of it lives in page
 * block_offsets[r * max_blocks_per_seq + t / tokens_per_block], slot t % tokens_per_block.
 * The host and device copies must hold the same values; the host copies plan the launch, the
 * device copies are what the kernels read (a disagreement is flagged PKV_DEVERR_PLAN_MISMATCH
 * where it is detectable).  Two requests may share a page read-only (prefix reuse).
 *
 * Draft tokens ([REPORT] 1.4 "推测解码技术": spec_decoding_generation_lengths, _position_offsets,
 * _packed_mask; [NOTES] 3.2 "Draft Token 裁剪": draft tokens verified by the large model in one
 * pass; [ARCH] "还有哪些值得一提的模块": the Medusa candidate tree): a generation request may bring
 * 1 .. PKV_MAX_GEN_TOKENS new tokens.  Its token i is stored at slot past + i like any new
 * token.  The two optional arrays below are indexed by a token's place among the generation
 * rows, k = packed row - (rows of the context requests):
 *   d_position_offsets[k]  the token is rotated for position past + offset instead of past + i
 *                          (its depth in the candidate tree); 0 <= offset < context_length,
 *                          otherwise PKV_DEVERR_BAD_OFFSET and the token is not written.
 *                          NULL: offset = i.  Context rows always use past + i.
 *   d_packed_mask[k * mask_words + j / 32] bit j % 32: the token sees new token j of its request.
 *                          It always sees itself and every cached token (t < past).  NULL:
 *                          plain causal order among the new tokens (token i sees j <= i).
 */
typedef struct pkv_batch {
  int32_t num_requests;       /* R = num_contexts + number of generation requests             */
  int32_t num_contexts;       /* C: requests 0 .. C-1 are context requests                    */
  int32_t num_tokens;         /* T = sum of context_lengths                                   */
  int32_t max_blocks_per_seq; /* row length of the block table                                */
  const int32_t* h_request_types;   /* host [R], pkv_req_type                                 */
  const int32_t* h_context_lengths; /* host [R], new tokens this step (1 for generation)      */
  const int32_t* h_past_kv_lengths; /* host [R], tokens already in the pool                   */
  const int32_t* d_context_lengths; /* device copy of h_context_lengths                       */
  const int32_t* d_past_kv_lengths; /* device copy of h_past_kv_lengths                       */
  const int32_t* d_block_offsets;   /* device [R, max_blocks_per_seq] page ids                */
  const int32_t* d_position_offsets; /* device [T_gen] or NULL (draft tokens, see above)      */
  const uint32_t* d_packed_mask;     /* device [T_gen, mask_words] or NULL (see above)         */
  int32_t mask_words;                /* words per mask row: >= ceil(longest generation
                                        request / 32) when d_packed_mask is set, else ignored  */
} pkv_batch;

/*
 * Bytes of the fp32 (cos, sin) RoPE table for positions 0 .. max_pos-1: max_pos * head_dim * 4.
 */
size_t paged_rope_table_bytes(int32_t head_dim, int32_t max_pos);

/*
 * Fill a HOST buffer with the GPT-NeoX RoPE table ([REPORT] 1.1: rotary_embedding, "GPT-NeoX"
 * variant): entry [p][j] = (cos(p * theta_j), sin(p * theta_j)) with theta_j = base^(-2j/D),
 * j < D/2, each computed in fp64 and rounded once to fp32.  The caller uploads it once per
 * (base, D, max_pos); paged_kv_append_rope reads it.  Returns PKV_OK or
 * PKV_ERR_INVALID_ARGUMENT.  Host-only set-up, not part of the per-step path.
 */
int paged_rope_table_build(double base, int32_t head_dim, int32_t max_pos, float* h_table);

/*
 * RoPE + append ([NOTES] 二.2 "KVCacheManager 详解": the attention op writes each new token's
 * K/V into the pages named by the block table; [ARCH] "AttentionMetadata 的字段与它的含义":
 * the backend may apply RoPE itself when position_ids is None; [NOTES] 6.4 "量化": quantise
 * on write).  For every packed row (request r, index i, slot position s = past_r + i, page
 * block_offsets[r][s / B], slot s % B; rotation position p = s, or past_r + offset for draft
 * tokens with d_position_offsets set):
 *   q_out[row, h*D:(h+1)*D] = bf16(rope(q[row, h*D:(h+1)*D], p))          for h < Hq
 *   pool[page, 0, slot, h, :] = bf16(rope(k[row, h*D:...], p))            for h < Hkv
 *   pool[page, 1, slot, h, :] = v[row, h*D:...]
 * (FP8 pool: e4m3(x * kv_scale_orig_quant) with round-to-nearest-even, saturating to +-448;
 * INT8 pool: the nearest integer to x * kv_scale_orig_quant, ties to even, saturated to
 * [-128, 127].)
 * rope(x, p): y_j = x_j c - x_{j+D/2} s, y_{j+D/2} = x_{j+D/2} c + x_j s, (c, s) = table[p][j],
 * evaluated in fp32 as fma(x_j, c, -(x_{j+D/2} * s)) and fma(x_{j+D/2}, c, x_j * s).
 *   q, k, v      device bf16 rows [T, Hq*D], [T, Hkv*D], [T, Hkv*D] with row strides in
 *                elements (a fused QKV tensor can be passed as three views)
 *   q_out        device bf16 [T, q_out_row_stride]; may equal q (in-place, same stride)
 *   rope_table   device fp32 table from paged_rope_table_build, max_pos rows
 *   d_error      device int32, PKV_DEVERR_* bits OR-ed in (bad page: that token's pool write
 *                is skipped, q_out is still written; bad draft offset: nothing of that token
 *                is written)
 * Every pool byte not addressed by a new token is left untouched.  T == 0 is a no-op.
 */
int paged_kv_append_rope(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads,
                         const void* q, int64_t q_row_stride, const void* k,
                         int64_t k_row_stride, const void* v, int64_t v_row_stride, void* q_out,
                         int64_t q_out_row_stride, const float* rope_table, int32_t max_pos,
                         int32_t* d_error, pkv_stream_t stream);

/*
 * Variants of the append (adg.csdn.net/69730cc6 section 1.1: RoPE variants and QK LayerNorm;
 * [ARCH] kernel list: fused QK-norm + RoPE).  Fields:
 *   rope_style     PKV_ROPE_NEOX (rotate-half pairs (x_j, x_{j+r/2})) or PKV_ROPE_GPTJ
 *                  (interleaved pairs (x_{2j}, x_{2j+1})), j < r/2
 *   rotary_dim     r: rotated dims per head, a multiple of 16 and <= head_dim (0 = head_dim);
 *                  dims >= r are copied unchanged; the RoPE table must then be built with
 *                  head_dim = r (r/2 (cos, sin) pairs per position, theta_j = base^(-2j/r))
 *   q_norm_weight  device fp32 [head_dim]: RMSNorm each query head before rotating it,
 *                  y = x / sqrt(mean(x^2) + norm_eps) * w; NULL = no norm
 *   k_norm_weight  the same for key heads (V is never normalised or rotated)
 *   norm_eps       epsilon of the norms
 * With a norm the sum of squares is an fp32 reduction across lanes, so results agree with an
 * exact computation to rounding (not bit for bit); without one they are the fixed fp32
 * recipe of paged_kv_append_rope.
 */
typedef enum { PKV_ROPE_NEOX = 0, PKV_ROPE_GPTJ = 1 } pkv_rope_style;
typedef struct pkv_append_opts {
  int32_t rope_style;
  int32_t rotary_dim;
  const float* q_norm_weight;
  const float* k_norm_weight;
  float norm_eps;
} pkv_append_opts;

/* paged_kv_append_rope with the variants above; opts == NULL is paged_kv_append_rope. */
int paged_kv_append_rope_ex(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads,
                            const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                            const void* v, int64_t v_row_stride, void* q_out, int64_t q_out_row_stride,
                            const float* rope_table, int32_t max_pos, const pkv_append_opts* opts,
                            int32_t* d_error, pkv_stream_t stream);

/*
 * Workspace bytes paged_attention_forward needs for this pool geometry, batch and head count
 * ([NOTES] 五 5.1: the runtime checks that the scratch workspace is large enough): the device
 * plan, fp32 split-KV partials, and for 8-bit pools with context requests a bf16 staging copy
 * of those requests' pages.  0 on invalid arguments.
 */
size_t paged_attention_workspace_size(const pkv_pool* pool, const pkv_batch* batch,
                                      int32_t num_q_heads);

/*
 * Causal GQA attention over the paged pool, after paged_kv_append_rope on the same stream
 * ([NOTES] 6.1 "两者分工": input length > 1 runs the context (flash-attention) path, length 1
 * the generation (paged attention) path; 6.2 "Flash Attention算法核心"; 6.3 "Paged Attention
 * Kernel 内部"; [ARCH] "AttentionMetadata 的字段与它的含义": flattened (num_tokens, heads*D)
 * tensors).  For packed row (r, i), query head h, KV head h / (Hq/Hkv), position p = past_r + i:
 *   out[row, h*D:(h+1)*D] = sum_{t in V(r,i)} softmax_t(softmax_scale * <q_rot[row,h], K_t>) V_t
 * with K_t, V_t read through the block table (8-bit pool: value = code * kv_scale_quant_orig),
 * fp32 accumulation, bf16 output.  The visible keys V(r, i) are t <= p (causal), except for
 * generation requests with d_packed_mask set: every t < past_r, plus past_r + j for the new
 * tokens j that the token's mask row selects, plus the token itself.  Generation requests of
 * several tokens use the decode kernel with (token, query head) pairs of one KV head as the
 * columns of its score tile, so the KV stream is still read once per KV head.
 *   q_rot        device bf16 [T, q_row_stride] rotated queries (q_out of the append)
 *   out          device bf16 [T, Hq*D] (row stride Hq*D)
 *   workspace    device, at least paged_attention_workspace_size bytes, 256-byte aligned;
 *                its contents need not be initialised and are scratch after the call
 *   d_error      device int32 error bits as above
 * Context rows use a tcgen05/TMEM tensor-core kernel (for 8-bit pools after staging the context
 * requests' pages as exact bf16 code values in the workspace), generation rows a split-KV decode
 * kernel plus a log-sum-exp combine.  Generation requests with more (token, query head) pairs
 * than the decode kernel's narrow columns run on the tensor-core generation kernel when
 * the query group divides 128 and the pool is bf16, or 8-bit at head_dim 128 (codes converted
 * to f16 in shared memory); otherwise on a wide split-KV decode kernel.  When the batch has both kinds of rows, the generation
 * kernels run on the library's auxiliary stream for this device (highest stream priority),
 * forked from `stream` by an event after the planning kernel and joined back into it before
 * the call returns, so that they share the GPU with the context kernel; every other launch goes
 * to `stream`.  The auxiliary stream is created by the first such call that is not made under
 * stream capture (calls made before that, and calls made while paged_kv_set_kernel_events is
 * set, run everything on `stream`); the fork and join are captured like any other stream work.
 * T == 0 is a no-op.
 */
int paged_attention_forward(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads,
                            const void* q_rot, int64_t q_row_stride, void* out,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            int32_t* d_error, pkv_stream_t stream);

/*
 * Padding buckets for CUDA-graph replay ([NOTES] 五 5.2 "CUDA graph": a captured graph is only
 * replayed when the batch has the shape it was captured with, so batch shapes are padded to a
 * few fixed buckets to raise the hit rate; [ARCH] "AttentionMetadata 的字段与它的含义":
 * create_cuda_graph_metadata allocates the metadata tensors once and never again after warm-up).
 *
 * The *_bucket entry points take every launch shape from the bucket and the pkv_batch's slot
 * counts, never from the lengths: the lengths are read on the device only.  So one capture of a
 * step serves every batch of the bucket -- the caller rewrites the device arrays (lengths, block
 * table, draft-token arrays) and the input rows between replays.  In the pkv_batch given to
 * them:
 *   num_requests        request slots R (fixed); num_contexts = C context slots 0 .. C-1,
 *                       slots C .. R-1 generation slots
 *   num_tokens          row capacity: the rows of q / k / v / q_out / out; a batch uses the
 *                       first sum(context_lengths) rows, packed in slot order
 *   max_blocks_per_seq  block-table row length (fixed)
 *   h_* arrays          ignored (may be NULL)
 *   d_context_lengths   per slot, the new tokens this step; 0 = an empty slot (no rows, no work)
 *   d_past_kv_lengths, d_block_offsets, d_position_offsets, d_packed_mask: as in pkv_batch (the
 *                       draft-token arrays indexed by generation row, with capacity for the
 *                       bucket's largest batch)
 * Each step's batch must fit the bucket: at most max_context_tokens rows in context slots,
 * past + new <= max_kv_len for every slot, at most max_gen_tokens new tokens per generation
 * slot, at most num_tokens rows.  The device checks this; a batch that does not fit sets
 * PKV_DEVERR_BUCKET and the attention writes nothing (the append may already have written its
 * tokens).  Grids are sized for the bucket's largest batch: the spare CTAs of a smaller batch
 * read the plan's counts and exit at once.
 */
typedef struct pkv_bucket {
  int32_t max_context_tokens; /* rows of the context slots together, at most (0: no contexts) */
  int32_t max_kv_len;         /* past + new of any slot, at most (<= max_blocks_per_seq * B)   */
  int32_t max_gen_tokens;     /* new tokens of a generation slot, 1 .. PKV_MAX_GEN_TOKENS      */
} pkv_bucket;

/* Workspace bytes of paged_attention_forward_bucket for this pool, slot layout and bucket
 * (enough for any batch of the bucket).  0 on invalid arguments. */
size_t paged_attention_bucket_workspace_size(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                             int32_t num_q_heads);

/* paged_kv_append_rope over a bucket (see above): the same arithmetic and layouts; the RoPE
 * table must hold max_kv_len positions.  Returns a host-detected PKV_ERR_* as the plain call
 * does; batch-dependent errors are the device's (PKV_DEVERR_*). */
int paged_kv_append_rope_bucket(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                int32_t num_q_heads, const void* q, int64_t q_row_stride, const void* k,
                                int64_t k_row_stride, const void* v, int64_t v_row_stride, void* q_out,
                                int64_t q_out_row_stride, const float* rope_table, int32_t max_pos,
                                const pkv_append_opts* opts, int32_t* d_error, pkv_stream_t stream);

/* paged_attention_forward over a bucket (see above); the workspace must hold
 * paged_attention_bucket_workspace_size bytes.  Output rows past the batch's rows are left
 * untouched. */
int paged_attention_forward_bucket(const pkv_pool* pool, const pkv_batch* batch, const pkv_bucket* bucket,
                                   int32_t num_q_heads, const void* q_rot, int64_t q_row_stride, void* out,
                                   float softmax_scale, void* workspace, size_t workspace_bytes, int32_t* d_error,
                                   pkv_stream_t stream);

/*
 * paged_attention_forward without a caller workspace.  The pages have no counterpart: this is
 * an addition for callers that cannot allocate device memory where they call attention (a
 * plugin whose host framework owns all device memory and offers no workspace hook, or a
 * latency-critical loop that forbids allocator calls).  Same arguments and results as
 * paged_attention_forward minus the workspace; the scratch comes from one file-scope device
 * buffer of PKV_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until exit.
 *   - A batch needing more scratch than that (paged_attention_workspace_size) returns
 *     PKV_ERR_WORKSPACE and launches nothing.  The call allocates nothing itself.
 *   - The first call on each device looks the buffer's device address up (cudaGetSymbolAddress
 *     with that device current) and caches it; make that first call before any stream capture.
 *   - All calls share the buffer and leave their data in it; nothing in it has to start at zero,
 *     but calls whose kernels overlap on the GPU (several streams or threads) race on it, so
 *     serialise them on one stream.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (64u << 20)
int paged_attention_forward_noalloc(const pkv_pool* pool, const pkv_batch* batch, int32_t num_q_heads,
                                    const void* q_rot, int64_t q_row_stride, void* out, float softmax_scale,
                                    int32_t* d_error, pkv_stream_t stream);

/* Number of kernels the last successful call of either entry point on this thread enqueued. */
int32_t paged_kv_last_launch_count(void);

/* Name of the i-th kernel the last call on this thread enqueued ("append_rope", "plan",
 * "stage_q8", "context_attn", "decode_splitkv", "decode_splitkv_wide", "decode_tc", "combine"),
 * or NULL
 * when i is out of range. */
const char* paged_kv_last_launch_name(int32_t i);

/*
 * Optional per-kernel timing for profiling harnesses.  `events` points to 2 * max_kernels
 * cudaEvent_t handles (created by the caller, host array owned by the caller and kept alive
 * while set).  Every later call on this thread records events[2i] on the stream just before
 * its i-th kernel and events[2i + 1] just after it, for i < max_kernels.  While events are
 * set, every kernel of a call goes to the caller's stream (no overlap of context and generation
 * kernels), so that each pair brackets one kernel alone.  NULL turns it off.
 * Returns PKV_OK or PKV_ERR_INVALID_ARGUMENT.
 */
int paged_kv_set_kernel_events(void* const* events, int32_t max_kernels);

/* Static string for a PKV_OK / PKV_ERR_* code. */
const char* paged_kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H_ */
