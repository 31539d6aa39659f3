/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV RoPE + attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
 * leg may load this library.  It shares no code, header, table or constant generator with the
 * CUDA library in paged_kv_cache_rope_gb300/csrc/, and neither includes the other.
 *
 * Sources (web pages on one serving engine; cited by page title and section):
 *   [ARCH]  "TensorRT-LLM 源码完全拆解(一):整体架构与模块全景" (pinghaoyang.com.cn),
 *           sections "KVCacheManager 的三个对外接口" (pool layout
 *           [num_blocks, 2, num_tokens_per_block, num_kv_heads, head_dim], K and V stacked on
 *           dim 1) and "AttentionMetadata 的字段与它的含义" (packed token stream, seq_lens,
 *           context_lens, position_ids).
 *   [NOTES] "TensorRT-LLM 1.0 源码学习笔记" (openharmonycrossplatform.csdn.net), sections
 *           二.2 "KVCacheManager 详解" (the kernel writes KV into blocks through the block
 *           table), 6.2 "Flash Attention算法核心" (softmax(QK^T)V), 6.3 "Paged Attention Kernel
 *           内部" (loop over a request's KV blocks through the block pointers) and 6.4 "量化"
 *           (quantise on write with kv_scale_orig_quant, dequantise on read with
 *           kv_scale_quant_orig).
 *   [REPORT] adg.csdn.net/69730cc6 (TensorRT-LLM source report), sections 1.1 (GPT-NeoX RoPE,
 *           GQA), 1.2 (KeyValueCacheParams: past lengths, kv_cache_block_offsets) and 1.3
 *           (context requests precede generation requests, no input padding).
 *
 * What the pages leave open is read as follows:
 *   - RoPE is the GPT-NeoX "rotate half" form over the whole head: pairs (x_j, x_{j+D/2}),
 *     theta_j = base^(-2j/D), angle = position * theta_j, position = past + i.
 *   - The rotation is done in fp32 from an fp32 (cos, sin) table that is computed in fp64 and
 *     rounded once:  y_j = fma(x_j, c, -(x_{j+D/2}*s)),  y_{j+D/2} = fma(x_{j+D/2}, c, x_j*s).
 *     This fixes every rounding, so the written pool bytes are a single exact value.
 *   - kv_kind selects the pool's element type: 0 bf16, 1 FP8 E4M3, 2 INT8.
 *   - FP8 is OCP E4M3 (bias 7, max normal 448, no infinities, NaN = S.1111.111), encoded
 *     round-to-nearest-even with saturation to +-448; code = e4m3(fp32(x * inv_scale)),
 *     value = code * scale, one scale per pool.
 *   - GQA: query head h reads KV head floor(h / (Hq/Hkv)).
 *   - Attention is causal over the request's logical KV sequence after the append:
 *     query i of request r (absolute position p = past_r + i) sees keys 0..p.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (see oracle/build.py).  The flag
 * -ffp-contract=off matters: the fp32 RoPE recipe above must not be re-fused by the compiler.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_BAD_PAGE (-1)
#define ORC_ERR_BAD_ARG (-2)

/* ------------------------------------------------------------------------------------------ */
/* bfloat16: the top 16 bits of an IEEE binary32.                                             */
/* ------------------------------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round an fp32 to the nearest bf16, ties to the even bf16 (IEEE round-to-nearest-even).
 * The two candidates are the truncation `lo` and the next bf16 up in magnitude `lo + 1`. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN (quiet) */
  }
  uint32_t lo = u >> 16;          /* truncated pattern (same sign) */
  uint32_t rest = u & 0xFFFFu;    /* discarded low half */
  if (rest > 0x8000u) return (uint16_t)(lo + 1);
  if (rest < 0x8000u) return (uint16_t)lo;
  return (uint16_t)((lo & 1u) ? lo + 1 : lo); /* exact tie: pick the even pattern */
}

/* ------------------------------------------------------------------------------------------ */
/* OCP FP8 E4M3 ("fn": finite, one NaN pattern per sign).                                     */
/* ------------------------------------------------------------------------------------------ */

/* Value of an E4M3 code from the format definition: sign s, exponent e (4 bits, bias 7),
 * mantissa m (3 bits).  e == 0 is subnormal: m/8 * 2^-6.  e == 15 && m == 7 is NaN. */
double orc_e4m3_to_f64(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even code, saturating finite and infinite overflow to the
 * largest finite magnitude 448 (code 0x7E).  The positive finite codes 0x00..0x7E are strictly
 * increasing in value, so a binary search finds the bracketing pair. */
uint8_t orc_f32_to_e4m3(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_to_f64((uint8_t)mid) <= a) lo = mid;
    else hi = mid;
  }
  double dlo = a - orc_e4m3_to_f64((uint8_t)lo);
  double dhi = orc_e4m3_to_f64((uint8_t)hi) - a;
  int pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo % 2 == 0) ? lo : hi;
  return (uint8_t)(sign | pick);
}

/* ------------------------------------------------------------------------------------------ */
/* INT8 ("INT8 KV Cache": the cache stored as 8-bit integers, quantised on write with            */
/* kv_scale_orig_quant and turned back into real values with kv_scale_quant_orig on read --     */
/* "TensorRT-LLM 1.0 源码学习笔记" 6.4 "量化").  Reading: the nearest integer, ties to the even    */
/* one, saturated to [-128, 127]; NaN encodes as 0.  value = code * scale.                       */
/* ------------------------------------------------------------------------------------------ */
int8_t orc_f32_to_int8(float x) {
  if (isnan(x)) return 0;
  double a = (double)x;
  if (a >= 127.0) return 127;
  if (a <= -128.0) return -128;
  double f = floor(a), diff = a - f;
  double n;
  if (diff > 0.5) n = f + 1.0;
  else if (diff < 0.5) n = f;
  else n = (fmod(f, 2.0) == 0.0) ? f : f + 1.0; /* exact tie: the even neighbour */
  return (int8_t)n;
}

/* ------------------------------------------------------------------------------------------ */
/* RoPE (GPT-NeoX rotate-half).                                                               */
/* ------------------------------------------------------------------------------------------ */

/* cs[(p * (D/2) + j) * 2 + {0,1}] = fp32(cos(p * theta_j)), fp32(sin(p * theta_j)),
 * theta_j = base^(-2j/D), all in fp64 and rounded once to fp32. */
void orc_rope_table(double base, int32_t head_dim, int32_t max_pos, float* cs) {
  int half = head_dim / 2;
  for (int p = 0; p < max_pos; ++p) {
    for (int j = 0; j < half; ++j) {
      double theta = pow(base, -(2.0 * (double)j) / (double)head_dim);
      double angle = (double)p * theta;
      cs[((size_t)p * half + j) * 2 + 0] = (float)cos(angle);
      cs[((size_t)p * half + j) * 2 + 1] = (float)sin(angle);
    }
  }
}

/* fp32 rotation of one head vector x[D] by the table row cs_row (D/2 (cos, sin) pairs). */
void orc_rope32(const float* x, int32_t head_dim, const float* cs_row, float* y) {
  int half = head_dim / 2;
  for (int j = 0; j < half; ++j) {
    float c = cs_row[2 * j], s = cs_row[2 * j + 1];
    float a = x[j], b = x[j + half];
    float bs = b * s; /* separate fp32 products: -ffp-contract=off keeps them unfused */
    float as = a * s;
    y[j] = fmaf(a, c, -bs);
    y[j + half] = fmaf(b, c, as);
  }
}

/* Exact-arithmetic reference rotation in fp64 (no table): used only to bound rope32's error. */
void orc_rope64(const double* x, int32_t head_dim, double base, int64_t pos, double* y) {
  int half = head_dim / 2;
  for (int j = 0; j < half; ++j) {
    double theta = pow(base, -(2.0 * (double)j) / (double)head_dim);
    double c = cos((double)pos * theta), s = sin((double)pos * theta);
    y[j] = x[j] * c - x[j + half] * s;
    y[j + half] = x[j + half] * c + x[j] * s;
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Pool addressing: pool[blk][kv][slot][h][d], kv 0 = K, 1 = V ([ARCH] get_buffers shape).     */
/* ------------------------------------------------------------------------------------------ */

static size_t pool_index(int blk, int kv, int slot, int h, int d, int B, int Hkv, int D) {
  return ((((size_t)blk * 2 + kv) * B + slot) * Hkv + h) * (size_t)D + d;
}

/* ------------------------------------------------------------------------------------------ */
/* O1: write image.  For every new token (request r, index i, position p = past_r + i):        */
/*   q_out row = bf16(rope32(q)), pool K slot = bf16(rope32(k)) or e4m3(rope32(k) * inv),       */
/*   pool V slot = v or e4m3(v * inv).  Every other pool byte is left untouched.               */
/* The packed stream holds request r's new tokens at rows cu_r .. cu_r + new_len[r] - 1 with    */
/* cu_r = sum of new_len over earlier requests ([ARCH] forward signature; [REPORT] 1.3).        */
/* Returns ORC_ERR_BAD_PAGE (and skips that token's pool write) when a page id is out of range. */
/* ------------------------------------------------------------------------------------------ */
int orc_append_rope(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                    const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                    int32_t num_blocks, int32_t kv_kind, float inv_scale, const uint16_t* q,
                    int64_t q_stride, const uint16_t* k, int64_t k_stride, const uint16_t* v,
                    int64_t v_stride, const float* cs, int32_t max_pos, uint16_t* q_out,
                    int64_t q_out_stride, void* pool) {
  int D = head_dim, B = tokens_per_block, Hkv = num_kv_heads, half = head_dim / 2;
  int status = ORC_OK;
  float* x = (float*)malloc(sizeof(float) * D);
  float* y = (float*)malloc(sizeof(float) * D);
  int64_t row = 0;
  for (int r = 0; r < num_requests; ++r) {
    for (int i = 0; i < new_len[r]; ++i, ++row) {
      int64_t pos = (int64_t)past[r] + i;
      if (pos >= max_pos) { status = ORC_ERR_BAD_ARG; continue; }
      const float* cs_row = cs + (size_t)pos * half * 2;
      for (int h = 0; h < num_q_heads; ++h) {
        for (int d = 0; d < D; ++d) x[d] = orc_bf16_to_f32(q[row * q_stride + (int64_t)h * D + d]);
        orc_rope32(x, D, cs_row, y);
        for (int d = 0; d < D; ++d) q_out[row * q_out_stride + (int64_t)h * D + d] = orc_f32_to_bf16(y[d]);
      }
      int logical_block = (int)(pos / B), slot = (int)(pos % B);
      int blk = logical_block < max_blocks_per_seq
                    ? block_table[(size_t)r * max_blocks_per_seq + logical_block] : -1;
      if (blk < 0 || blk >= num_blocks) {
        status = ORC_ERR_BAD_PAGE;
        continue;
      }
      for (int h = 0; h < Hkv; ++h) {
        for (int d = 0; d < D; ++d) x[d] = orc_bf16_to_f32(k[row * k_stride + (int64_t)h * D + d]);
        orc_rope32(x, D, cs_row, y);
        for (int d = 0; d < D; ++d) {
          uint16_t vb = v[row * v_stride + (int64_t)h * D + d];
          size_t ik = pool_index(blk, 0, slot, h, d, B, Hkv, D);
          size_t iv = pool_index(blk, 1, slot, h, d, B, Hkv, D);
          if (kv_kind == 1) {
            uint8_t* p8 = (uint8_t*)pool;
            p8[ik] = orc_f32_to_e4m3(y[d] * inv_scale);
            p8[iv] = orc_f32_to_e4m3(orc_bf16_to_f32(vb) * inv_scale);
          } else if (kv_kind == 2) {
            int8_t* p8 = (int8_t*)pool;
            p8[ik] = orc_f32_to_int8(y[d] * inv_scale);
            p8[iv] = orc_f32_to_int8(orc_bf16_to_f32(vb) * inv_scale);
          } else {
            uint16_t* p16 = (uint16_t*)pool;
            p16[ik] = orc_f32_to_bf16(y[d]);
            p16[iv] = vb;
          }
        }
      }
    }
  }
  free(x);
  free(y);
  return status;
}

/* ------------------------------------------------------------------------------------------ */
/* O2: attention in fp64 over the pool, per the definition                                    */
/*   out[row, h, :] = sum_t softmax_t(scale * <q[row, h, :], K_t>) V_t,  t = 0 .. past_r + i,  */
/* with K_t, V_t read through the block table (page tbl[r][t / B], slot t % B) and decoded     */
/* exactly (bf16 -> double; e4m3 or int8 code -> value * kv_scale).  q is fp64 [T, Hq, D].      */
/* rows == NULL computes every row; otherwise only the listed packed-row indices.              */
/* Returns ORC_ERR_BAD_PAGE if a needed page id is out of range (that row is left as NaN).     */
/* ------------------------------------------------------------------------------------------ */
static double pool_value(const void* pool, int kv_kind, double kv_scale, size_t idx) {
  if (kv_kind == 1) return orc_e4m3_to_f64(((const uint8_t*)pool)[idx]) * kv_scale;
  if (kv_kind == 2) return (double)((const int8_t*)pool)[idx] * kv_scale;
  return (double)orc_bf16_to_f32(((const uint16_t*)pool)[idx]);
}

/* Keys visible to query i of request r: every cached key t < past_r, and the new key
 * past_r + j (j < new_len[r]) when j <= i -- plain causal order.  A generation request of
 * several new tokens (draft tokens verified in one step: [REPORT] 1.4 "推测解码技术",
 * spec_decoding_generation_lengths / spec_decoding_packed_mask; [ARCH] "还有哪些值得一提的模块",
 * the Medusa candidate tree) may instead carry a packed mask row per token: bit j of word j / 32
 * set means "sees new token j"; the token always sees itself.  gen_mask is indexed by the
 * token's place among the generation rows (packed row - rows of the context requests). */
static int attention_core(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                          const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                          int32_t num_blocks, int32_t kv_kind, double kv_scale, const void* pool,
                          const double* q, double softmax_scale, const int64_t* rows, int64_t num_rows,
                          int32_t num_contexts, const uint32_t* gen_mask, int32_t mask_words,
                          double* out) {
  int D = head_dim, B = tokens_per_block, Hkv = num_kv_heads;
  int group = num_q_heads / num_kv_heads;
  if (group * num_kv_heads != num_q_heads) return ORC_ERR_BAD_ARG;
  int64_t T = 0, ctx_rows = 0;
  for (int r = 0; r < num_requests; ++r) {
    T += new_len[r];
    if (r < num_contexts) ctx_rows += new_len[r];
  }
  if (gen_mask) {
    for (int r = num_contexts; r < num_requests; ++r)
      if (new_len[r] > 32 * mask_words) return ORC_ERR_BAD_ARG;
  }
  /* request of each packed row, and its index inside the request */
  int32_t* row_req = (int32_t*)malloc(sizeof(int32_t) * (T > 0 ? T : 1));
  int32_t* row_idx = (int32_t*)malloc(sizeof(int32_t) * (T > 0 ? T : 1));
  {
    int64_t row = 0;
    for (int r = 0; r < num_requests; ++r)
      for (int i = 0; i < new_len[r]; ++i, ++row) { row_req[row] = r; row_idx[row] = i; }
  }
  int64_t n = rows ? num_rows : T;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t w = 0; w < n; ++w) {
    for (int h = 0; h < num_q_heads; ++h) {
      int64_t row = rows ? rows[w] : w;
      int r = row_req[row], i = row_idx[row];
      const uint32_t* mrow = (gen_mask && r >= num_contexts) ? gen_mask + (row - ctx_rows) * mask_words : NULL;
      /* keys 0 .. past + i (causal), or every key of the request when a mask row decides */
      int64_t L = mrow ? (int64_t)past[r] + new_len[r] : (int64_t)past[r] + i + 1;
      int hk = h / group;
      const double* qv = q + (row * num_q_heads + h) * (int64_t)D;
      double* o = out + (row * num_q_heads + h) * (int64_t)D;
      double* s = (double*)malloc(sizeof(double) * L);
      int bad = 0;
      for (int64_t t = 0; t < L && !bad; ++t) {
        if (mrow && t >= past[r]) {
          int j = (int)(t - past[r]);
          if (j != i && !((mrow[j / 32] >> (j % 32)) & 1u)) { s[t] = -INFINITY; continue; }
        }
        int lb = (int)(t / B);
        int blk = lb < max_blocks_per_seq ? block_table[(size_t)r * max_blocks_per_seq + lb] : -1;
        if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
          dot += qv[d] * pool_value(pool, kv_kind, kv_scale, pool_index(blk, 0, (int)(t % B), hk, d, B, Hkv, D));
        s[t] = softmax_scale * dot;
      }
      if (bad) {
        for (int d = 0; d < D; ++d) o[d] = NAN;
#pragma omp atomic write
        status = ORC_ERR_BAD_PAGE;
        free(s);
        continue;
      }
      double m = -INFINITY;
      for (int64_t t = 0; t < L; ++t) m = s[t] > m ? s[t] : m;
      double z = 0.0;
      for (int64_t t = 0; t < L; ++t) { s[t] = exp(s[t] - m); z += s[t]; }
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int64_t t = 0; t < L; ++t) {
        int blk = block_table[(size_t)r * max_blocks_per_seq + (int)(t / B)];
        double w_t = s[t] / z;
        for (int d = 0; d < D; ++d)
          o[d] += w_t * pool_value(pool, kv_kind, kv_scale, pool_index(blk, 1, (int)(t % B), hk, d, B, Hkv, D));
      }
      free(s);
    }
  }
  free(row_req);
  free(row_idx);
  return status;
}

int orc_attention(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                  const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                  int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                  int32_t num_blocks, int32_t kv_kind, double kv_scale, const void* pool,
                  const double* q, double softmax_scale, const int64_t* rows, int64_t num_rows,
                  double* out) {
  return attention_core(num_requests, new_len, past, block_table, max_blocks_per_seq, num_q_heads,
                        num_kv_heads, head_dim, tokens_per_block, num_blocks, kv_kind, kv_scale, pool,
                        q, softmax_scale, rows, num_rows, num_requests, NULL, 0, out);
}

/* O2 with packed masks for the generation requests (requests num_contexts .. R-1). */
int orc_attention_spec(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                       const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                       int32_t num_blocks, int32_t kv_kind, double kv_scale, const void* pool,
                       const double* q, double softmax_scale, const int64_t* rows, int64_t num_rows,
                       int32_t num_contexts, const uint32_t* gen_mask, int32_t mask_words,
                       double* out) {
  return attention_core(num_requests, new_len, past, block_table, max_blocks_per_seq, num_q_heads,
                        num_kv_heads, head_dim, tokens_per_block, num_blocks, kv_kind, kv_scale, pool,
                        q, softmax_scale, rows, num_rows, num_contexts, gen_mask, mask_words, out);
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Element-wise array forms of the two encoders (same per-element definitions as above). */
void orc_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

void orc_f32_to_e4m3_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(x[i]);
}

void orc_f32_to_int8_array(const float* x, int64_t n, int8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_int8(x[i]);
}

void orc_e4m3_to_f64_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f64(c[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* Variants of the append (adg.csdn.net/69730cc6 section 1.1: several RoPE variants, QK       */
/* LayerNorm; "TensorRT-LLM 源码完全拆解(一)" kernel list: fused QK-norm + RoPE).  Readings:     */
/*   style 0 = GPT-NeoX rotate-half: pairs (x_j, x_{j+r/2}), j < r/2;                          */
/*   style 1 = GPT-J interleaved:    pairs (x_{2j}, x_{2j+1}), j < r/2;                         */
/*   r = rotary dims (a multiple of 16, <= D), theta_j = base^(-2j/r); dims >= r pass through;  */
/*   QK-norm = RMSNorm over each q / k head before the rotation:                               */
/*     y_d = fp32(fp32(x_d * inv_rms) * w_d), inv_rms = fp32(1 / sqrt(mean(x^2) + eps)),        */
/*   the mean taken in fp64 (the reference value; the kernel sums in fp32, so outputs with      */
/*   QK-norm agree to rounding, not bit for bit).  V is never normalised or rotated.            */
/* ------------------------------------------------------------------------------------------ */
static void rotate_variant(const float* x, int32_t D, int32_t rot, int32_t style, const float* cs_row, float* y) {
  for (int d = 0; d < D; ++d) y[d] = x[d];
  int half = rot / 2;
  for (int j = 0; j < half; ++j) {
    int ia = style == 0 ? j : 2 * j;
    int ib = style == 0 ? j + half : 2 * j + 1;
    float c = cs_row[2 * j], s = cs_row[2 * j + 1];
    float a = x[ia], b = x[ib];
    float bs = b * s, as = a * s;
    y[ia] = fmaf(a, c, -bs);
    y[ib] = fmaf(b, c, as);
  }
}

static void rms_norm(float* x, int32_t D, const float* w, double eps) {
  double ss = 0.0;
  for (int d = 0; d < D; ++d) ss += (double)x[d] * (double)x[d];
  float inv = (float)(1.0 / sqrt(ss / D + eps));
  for (int d = 0; d < D; ++d) {
    float t = x[d] * inv;
    x[d] = t * w[d];
  }
}

static int append_core(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                       const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                       int32_t num_blocks, int32_t kv_kind, float inv_scale, const uint16_t* q,
                       int64_t q_stride, const uint16_t* k, int64_t k_stride, const uint16_t* v,
                       int64_t v_stride, const float* cs, int32_t max_pos, int32_t style,
                       int32_t rotary_dim, const float* q_norm_w, const float* k_norm_w,
                       double norm_eps, const int32_t* pos_offset, uint16_t* q_out,
                       int64_t q_out_stride, void* pool) {
  int D = head_dim, B = tokens_per_block, Hkv = num_kv_heads;
  int rot = rotary_dim > 0 ? rotary_dim : D;
  int status = ORC_OK;
  float* x = (float*)malloc(sizeof(float) * D);
  float* y = (float*)malloc(sizeof(float) * D);
  int64_t row = 0;
  for (int r = 0; r < num_requests; ++r) {
    for (int i = 0; i < new_len[r]; ++i, ++row) {
      int64_t pos = (int64_t)past[r] + i; /* where the token is stored */
      int64_t off = pos_offset ? pos_offset[row] : i;
      if (off < 0 || off >= new_len[r]) { status = ORC_ERR_BAD_ARG; continue; }
      int64_t rpos = (int64_t)past[r] + off; /* the position its rotation uses */
      if (pos >= max_pos || rpos >= max_pos) { status = ORC_ERR_BAD_ARG; continue; }
      const float* cs_row = cs + (size_t)rpos * (rot / 2) * 2;
      for (int h = 0; h < num_q_heads; ++h) {
        for (int d = 0; d < D; ++d) x[d] = orc_bf16_to_f32(q[row * q_stride + (int64_t)h * D + d]);
        if (q_norm_w) rms_norm(x, D, q_norm_w, norm_eps);
        rotate_variant(x, D, rot, style, cs_row, y);
        for (int d = 0; d < D; ++d) q_out[row * q_out_stride + (int64_t)h * D + d] = orc_f32_to_bf16(y[d]);
      }
      int logical_block = (int)(pos / B), slot = (int)(pos % B);
      int blk = logical_block < max_blocks_per_seq
                    ? block_table[(size_t)r * max_blocks_per_seq + logical_block] : -1;
      if (blk < 0 || blk >= num_blocks) { status = ORC_ERR_BAD_PAGE; continue; }
      for (int h = 0; h < Hkv; ++h) {
        for (int d = 0; d < D; ++d) x[d] = orc_bf16_to_f32(k[row * k_stride + (int64_t)h * D + d]);
        if (k_norm_w) rms_norm(x, D, k_norm_w, norm_eps);
        rotate_variant(x, D, rot, style, cs_row, y);
        for (int d = 0; d < D; ++d) {
          uint16_t vb = v[row * v_stride + (int64_t)h * D + d];
          size_t ik = pool_index(blk, 0, slot, h, d, B, Hkv, D);
          size_t iv = pool_index(blk, 1, slot, h, d, B, Hkv, D);
          if (kv_kind == 1) {
            uint8_t* p8 = (uint8_t*)pool;
            p8[ik] = orc_f32_to_e4m3(y[d] * inv_scale);
            p8[iv] = orc_f32_to_e4m3(orc_bf16_to_f32(vb) * inv_scale);
          } else if (kv_kind == 2) {
            int8_t* p8 = (int8_t*)pool;
            p8[ik] = orc_f32_to_int8(y[d] * inv_scale);
            p8[iv] = orc_f32_to_int8(orc_bf16_to_f32(vb) * inv_scale);
          } else {
            uint16_t* p16 = (uint16_t*)pool;
            p16[ik] = orc_f32_to_bf16(y[d]);
            p16[iv] = vb;
          }
        }
      }
    }
  }
  free(x);
  free(y);
  return status;
}

int orc_append_rope_ex(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                       const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                       int32_t num_blocks, int32_t kv_kind, float inv_scale, const uint16_t* q,
                       int64_t q_stride, const uint16_t* k, int64_t k_stride, const uint16_t* v,
                       int64_t v_stride, const float* cs, int32_t max_pos, int32_t style,
                       int32_t rotary_dim, const float* q_norm_w, const float* k_norm_w,
                       double norm_eps, uint16_t* q_out, int64_t q_out_stride, void* pool) {
  return append_core(num_requests, new_len, past, block_table, max_blocks_per_seq, num_q_heads,
                     num_kv_heads, head_dim, tokens_per_block, num_blocks, kv_kind, inv_scale, q,
                     q_stride, k, k_stride, v, v_stride, cs, max_pos, style, rotary_dim, q_norm_w,
                     k_norm_w, norm_eps, NULL, q_out, q_out_stride, pool);
}

/* ------------------------------------------------------------------------------------------ */
/* O1 for draft tokens ([REPORT] 1.4 "推测解码技术", spec_decoding_position_offsets): packed row  */
/* `row` (request r, index i) is still stored at slot past_r + i, but rotated for position      */
/* past_r + pos_offset[row] (its depth in the candidate tree); 0 <= pos_offset[row] < new_len[r] */
/* or the token is skipped with ORC_ERR_BAD_ARG.  pos_offset holds one entry per packed row.     */
/* ------------------------------------------------------------------------------------------ */
int orc_append_rope_spec(int32_t num_requests, const int32_t* new_len, const int32_t* past,
                         const int32_t* block_table, int32_t max_blocks_per_seq, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t tokens_per_block,
                         int32_t num_blocks, int32_t kv_kind, float inv_scale, const uint16_t* q,
                         int64_t q_stride, const uint16_t* k, int64_t k_stride, const uint16_t* v,
                         int64_t v_stride, const float* cs, int32_t max_pos, int32_t style,
                         int32_t rotary_dim, const float* q_norm_w, const float* k_norm_w,
                         double norm_eps, const int32_t* pos_offset, uint16_t* q_out,
                         int64_t q_out_stride, void* pool) {
  return append_core(num_requests, new_len, past, block_table, max_blocks_per_seq, num_q_heads,
                     num_kv_heads, head_dim, tokens_per_block, num_blocks, kv_kind, inv_scale, q,
                     q_stride, k, k_stride, v, v_stride, cs, max_pos, style, rotary_dim, q_norm_w,
                     k_norm_w, norm_eps, pos_offset, q_out, q_out_stride, pool);
}
