/*
 * kvattn_oracle.c -- plain, slow, float64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg and reference arm may load this file's library.  It shares no
 * code, header, table or constant with the CUDA library: it is written from
 * the definitions on the pages, in the pages' notation, and nothing here is
 * blocked, fused or reordered beyond what those definitions state.
 *
 * Sources (page title, then section):
 *   [P1] "MHA -> MQA -> GQA -> MLA" (mlinterviewnotes, Inference §3.5)
 *   [P2] "Multi-Head Latent Attention (MLA): Mathematical Foundations,
 *         Low-Rank KV Compression, Decoupled Rotary Positional Embeddings,
 *         and Inference Matrix Absorption" (llms.blog)
 *   [P3] "The KV cache size formula" (mlinterviewnotes, Inference §2.1)
 *   [P4] "MLA：为什么一份 Latent 可以代替多头 KV Cache" (charlestar.github.io)
 *
 * Inputs are the stored values: bf16 bit patterns are widened exactly; FP8
 * codes are decoded from the E4M3 format definition and multiplied by their
 * per-tensor scale.  All arithmetic is double.  Natural exp/log throughout;
 * lse is the natural log-sum-exp of the scaled scores.
 *
 * Every function is pinned by tests/test_oracle.py against something other
 * than itself (page figures, closed forms, brute force, a library routine, or
 * the explicit-vs-absorbed MLA identity).  Parity unpinned: none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KVO_FMT_BF16 0   /* uint16 bfloat16 bit patterns            */
#define KVO_FMT_E4M3 1   /* uint8 E4M3 codes, value = decode * scale */
#define KVO_FMT_F64  2   /* double                                   */

int kvo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Element formats                                                           */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the top half of an IEEE binary32; widening is exact. */
double kvo_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* FP8-E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits.  Exponent field 0 is subnormal: (-1)^s * 2^-6 * m/8.  Otherwise
 * (-1)^s * 2^(e-7) * (1 + m/8).  There is no infinity; S.1111.111 is NaN,
 * so the largest finite magnitude is 2^8 * 1.75 = 448.  The pages name the
 * format and the per-tensor scale = amax/448 recipe ([P2] "High-Throughput
 * Serving Kernels: FlashMLA and SGLang"; [P4] "MLA 与 KV Cache 量化可以叠加";
 * [P3] "--kv-cache-dtype fp8 doubles the token count"). */
double kvo_e4m3_decode(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  double mag;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Encode a binary32 value to E4M3: round to the nearest representable value,
 * ties to the code with an even mantissa, and saturate magnitudes above 448 to
 * 448 (the format has no infinity).  The non-negative finite codes 0x00..0x7E
 * decode to strictly increasing magnitudes, so the nearest one is found by a
 * binary search for the first code whose magnitude is >= |x| and a comparison
 * with the code below it. */
uint8_t kvo_e4m3_encode(float x) {
  double a = fabs((double)x);
  uint8_t sign = (x < 0.0f || (x == 0.0f && signbit(x))) ? 0x80 : 0x00;
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E;              /* first code with magnitude >= a */
  while (lo < hi) {
    int mid = (lo + hi) / 2;
    if (kvo_e4m3_decode((uint8_t)mid) >= a)
      hi = mid;
    else
      lo = mid + 1;
  }
  int best = lo;
  if (lo > 0) {
    double up = kvo_e4m3_decode((uint8_t)lo) - a, down = a - kvo_e4m3_decode((uint8_t)(lo - 1));
    if (down < up || (down == up && ((lo - 1) & 1) == 0)) best = lo - 1;
  }
  return (uint8_t)(sign | best);
}

/* Quantise stored bf16 values to E4M3 codes with a per-tensor scale:
 * code = e4m3(x / scale).  The division is done in binary32, the precision
 * the device writer divides in, so that both sides take the same integer
 * decision. */
void kvo_quantize_e4m3(const uint16_t* x, int64_t n, float scale, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)kvo_bf16_to_double(x[i]);
    float q = v / scale;
    codes[i] = kvo_e4m3_encode(q);
  }
}

static double elem(const void* p, int fmt, double scale, int64_t i) {
  switch (fmt) {
    case KVO_FMT_BF16: return kvo_bf16_to_double(((const uint16_t*)p)[i]);
    case KVO_FMT_E4M3: return kvo_e4m3_decode(((const uint8_t*)p)[i]) * scale;
    default: return ((const double*)p)[i];
  }
}

/* ------------------------------------------------------------------------ */
/* Cache sizing                                                              */
/* ------------------------------------------------------------------------ */

/* Cell size (bytes per token, whole model).  GQA/MQA/MHA: every layer stores
 * one K and one V vector per KV head, L * h_kv * (d_k + d_v) * b, i.e.
 * 2 * L * h_kv * d_h * b when d_k = d_v = d_h ([P3] "The KV cache size
 * formula" and "SGLang: one cell size, one division").  MLA: one latent row of
 * d_c + d_rope elements per layer, with neither a factor 2 nor a head count,
 * L * (d_c + d_rope) * b ([P3] "Where MLA breaks the formula"). */
int64_t kvo_cell_bytes_gqa(int64_t L, int64_t h_kv, int64_t d_k, int64_t d_v, int64_t b) {
  return L * h_kv * (d_k + d_v) * b;
}
int64_t kvo_cell_bytes_mla(int64_t L, int64_t d_c, int64_t d_rope, int64_t b) {
  return L * (d_c + d_rope) * b;
}

/* vLLM's per-layer page: num_heads * block_size * (head_size + head_size_v)
 * * dtype bytes; MLA pins num_heads = 1, head_size = 576, head_size_v = 0
 * ([P3] "vLLM: a per-layer page, then integer division"). */
int64_t kvo_page_bytes(int64_t num_heads, int64_t block_size, int64_t head_size,
                       int64_t head_size_v, int64_t b) {
  return num_heads * block_size * (head_size + head_size_v) * b;
}

/* Whole blocks per request: cdiv(len, block_size) ([P3] "a 17-token request
 * occupies 32 slots at block_size=16"). */
int64_t kvo_blocks_for(int64_t len, int64_t block_size) {
  return (len + block_size - 1) / block_size;
}

/* Decode arithmetic intensity in FLOP/byte.  GQA: 2g/b ([P1] "Context length s
 * cancelled ... What survives is g and the dtype").  MLA at h local query
 * heads: 2h(2 r_kv + d_rope) / (b (r_kv + d_rope)) ([P1] "the query heads
 * shard and the latent does not, so per-rank intensity is ..."). */
double kvo_intensity_gqa(double g, double b) { return 2.0 * g / b; }
double kvo_intensity_mla(double h, double r_kv, double d_rope, double b) {
  return 2.0 * h * (2.0 * r_kv + d_rope) / (b * (r_kv + d_rope));
}

/* ------------------------------------------------------------------------ */
/* Paged placement                                                           */
/* ------------------------------------------------------------------------ */

/* Logical token t of sequence b lives in block block_table[b][t / bs] at
 * offset t % bs ([P4] "Paged KV Cache 的 Block 里放什么": the cache writer,
 * the block table and the attention kernel must agree on one layout; [P3]
 * "vLLM allocates whole blocks").  Returns -1 if the table entry is missing. */
int64_t kvo_slot_block(const int32_t* block_table, int max_blocks, int bs, int b, int64_t t) {
  int64_t j = t / bs;
  if (j >= max_blocks) return -1;
  return block_table[(int64_t)b * max_blocks + j];
}

/* Element offset of K[t][kvh][0] (or V) of sequence b in a GQA pool laid out
 * [num_blocks][h_kv][bs][d]: one buffer per K and per V, indexed by KV head
 * ([P3] "MHA takes two buffers per layer indexed by KV head"). */
int64_t kvo_gqa_pool_offset(const int32_t* block_table, int max_blocks, int bs, int h_kv, int d,
                            int b, int64_t t, int kvh) {
  int64_t blk = kvo_slot_block(block_table, max_blocks, bs, b, t);
  if (blk < 0) return -1;
  return ((blk * h_kv + kvh) * bs + (t % bs)) * (int64_t)d;
}

/* Element offset of row t of sequence b in an MLA pool [num_blocks][bs][width];
 * each row is [c_KV | k_R] ([P4] "page / token i: [c_KV | k_R]"; [P3] "MLA one
 * with a head axis pinned to 1"). */
int64_t kvo_mla_pool_offset(const int32_t* block_table, int max_blocks, int bs, int width,
                            int b, int64_t t) {
  int64_t blk = kvo_slot_block(block_table, max_blocks, bs, b, t);
  if (blk < 0) return -1;
  return (blk * bs + (t % bs)) * (int64_t)width;
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

/* Single-token decode attention for one sequence with grouped KV heads.
 *
 *   o_i = softmax_t( scale * q_i . K_t[kvh(i)] ) V[kvh(i)],  kvh(i) = i / g,
 *
 * over all s cached positions t = 0..s-1, g = h / h_kv query heads per KV
 * head ([P3] "Attention computes softmax(qK^T/sqrt(d_h))V against all previous
 * positions"; [P1] "Query heads are broadcast against whatever KV heads exist",
 * "MHA, MQA and GQA are all the same code path with a different integer").
 * lse_i = m + log(sum_t exp(s_t - m)), the log-sum-exp the pages ask kernels
 * to be compared on ([P4] "正确性验证应该从两种实现互证", step 5).
 *
 * q: [h][d] bf16 bits.  k, v: [s][h_kv][d] contiguous (a gathered, unpaged
 * cache) in format fmt.  out: [h][d], lse: [h].  s == 0 gives out = 0 and
 * lse = -inf.  Returns 0, or -1 on a bad shape. */
int kvo_gqa_decode(const uint16_t* q, const void* k, const void* v, int fmt,
                   double k_scale, double v_scale, int64_t s, int h, int h_kv, int d,
                   double scale, double* out, double* lse) {
  if (h <= 0 || h_kv <= 0 || d <= 0 || h % h_kv != 0 || s < 0) return -1;
  int g = h / h_kv;
  int i;
#pragma omp parallel for schedule(dynamic, 1)
  for (i = 0; i < h; ++i) {
    int kvh = i / g;
    double* o = out + (int64_t)i * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (s == 0) {
      lse[i] = -INFINITY;
      continue;
    }
    double* sc = (double*)malloc(sizeof(double) * (size_t)s);
    double m = -INFINITY;
    for (int64_t t = 0; t < s; ++t) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c)
        acc += kvo_bf16_to_double(q[(int64_t)i * d + c]) *
               elem(k, fmt, k_scale, (t * h_kv + kvh) * d + c);
      sc[t] = scale * acc;
      if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < s; ++t) {
      double p = exp(sc[t] - m);
      l += p;
      for (int c = 0; c < d; ++c) o[c] += p * elem(v, fmt, v_scale, (t * h_kv + kvh) * d + c);
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
    lse[i] = m + log(l);
    free(sc);
  }
  return 0;
}

/* MLA decode in absorbed ("MQA mode") form for one sequence.
 *
 * Each cached row is [c_KV (d_c) | k_R (d_rope)].  With the absorbed query
 * q~_i = [W_UK,i^T q^C_i | q^R_i] the score is
 *     Score_i,t = q~^C_i . c_t + q^R_i . k^R_t = q~_i . row_t,
 * A_i = softmax_t(scale * Score_i,t) and the output is the latent weighted sum
 *     u~_i = sum_t A_i,t c_t          (d_c wide; k^R enters the scores only)
 * ([P2] "Attention Logit Matrix Absorption", "Value Output Matrix Absorption";
 * [P4] "第一次矩阵吸收" and "第二次矩阵吸收").  The scale is the caller's
 * (1/sqrt(d_h^C + d_r) on the pages, not 1/sqrt of the row width).
 *
 * q: [h][d_c + d_rope], rows: [s][d_c + d_rope], both in format fmt (bf16 bits
 * or double).  out: [h][d_c], lse: [h]. */
int kvo_mla_decode(const void* q, const void* rows, int fmt, int64_t s, int h, int d_c,
                   int d_rope, double scale, double* out, double* lse) {
  if (h <= 0 || d_c <= 0 || d_rope < 0 || s < 0) return -1;
  int w = d_c + d_rope;
  int i;
#pragma omp parallel for schedule(dynamic, 1)
  for (i = 0; i < h; ++i) {
    double* o = out + (int64_t)i * d_c;
    for (int c = 0; c < d_c; ++c) o[c] = 0.0;
    if (s == 0) {
      lse[i] = -INFINITY;
      continue;
    }
    double* sc = (double*)malloc(sizeof(double) * (size_t)s);
    double m = -INFINITY;
    for (int64_t t = 0; t < s; ++t) {
      double acc = 0.0;
      for (int c = 0; c < w; ++c)
        acc += elem(q, fmt, 1.0, (int64_t)i * w + c) * elem(rows, fmt, 1.0, t * w + c);
      sc[t] = scale * acc;
      if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < s; ++t) {
      double p = exp(sc[t] - m);
      l += p;
      for (int c = 0; c < d_c; ++c) o[c] += p * elem(rows, fmt, 1.0, t * w + c);
    }
    for (int c = 0; c < d_c; ++c) o[c] /= l;
    lse[i] = m + log(l);
    free(sc);
  }
  return 0;
}

/* MLA absorbed decode over an FP8-E4M3 latent cache.  Each cached row is
 * stored as E4M3 codes: the c_KV part decodes to e4m3(code) * c_scale and the
 * k_R part to e4m3(code) * r_scale, one per-tensor scale each (the pages
 * store the MLA latent in FP8 with scaling factors: [P2] "High-Throughput
 * Serving Kernels: FlashMLA and SGLang"; [P4] "MLA 与 KV Cache 量化可以叠加").
 * The rows are decoded to double and the attention is kvo_mla_decode's on
 * those values.  q: bf16 [h][d_c + d_rope]; codes: [s][d_c + d_rope]. */
int kvo_mla_decode_e4m3(const uint16_t* q, const uint8_t* codes, int64_t s, int h, int d_c,
                        int d_rope, double c_scale, double r_scale, double scale, double* out,
                        double* lse) {
  if (h <= 0 || d_c <= 0 || d_rope < 0 || s < 0) return -1;
  int w = d_c + d_rope;
  double* qd = (double*)malloc(sizeof(double) * (size_t)h * (size_t)w);
  double* rows = (double*)malloc(sizeof(double) * ((size_t)s * (size_t)w + 1));
  if (!qd || !rows) {
    free(qd);
    free(rows);
    return -1;
  }
  for (int64_t i = 0; i < (int64_t)h * w; ++i) qd[i] = kvo_bf16_to_double(q[i]);
  for (int64_t t = 0; t < s; ++t)
    for (int c = 0; c < w; ++c)
      rows[t * w + c] = kvo_e4m3_decode(codes[t * w + c]) * (c < d_c ? c_scale : r_scale);
  int rc = kvo_mla_decode(qd, rows, KVO_FMT_F64, s, h, d_c, d_rope, scale, out, lse);
  free(qd);
  free(rows);
  return rc;
}

/* Query-side absorption q~^C_i = W_UK,i^T q^C_i, W_UK viewed (h, d_hc, d_c)
 * ([P2] "Let us define the absorbed query vector"; the reference module's
 * w_uk.view(n_heads, d_head, d_c_kv)).  q_c: [h][d_hc]; w_uk: [h][d_hc][d_c];
 * q_tilde: [h][d_c]. */
void kvo_mla_absorb_query(const double* q_c, const double* w_uk, int h, int d_hc, int d_c,
                          double* q_tilde) {
  for (int i = 0; i < h; ++i)
    for (int c = 0; c < d_c; ++c) {
      double acc = 0.0;
      for (int j = 0; j < d_hc; ++j)
        acc += w_uk[((int64_t)i * d_hc + j) * d_c + c] * q_c[(int64_t)i * d_hc + j];
      q_tilde[(int64_t)i * d_c + c] = acc;
    }
}

/* Deferred value up-projection u_i = W_UV,i u~_i ([P2] "By linearity, the
 * matrix W_UV,i can be factored outside the summation").  u_tilde: [h][d_c];
 * w_uv: [h][d_v][d_c]; u: [h][d_v]. */
void kvo_mla_apply_wuv(const double* u_tilde, const double* w_uv, int h, int d_v, int d_c,
                       double* u) {
  for (int i = 0; i < h; ++i)
    for (int j = 0; j < d_v; ++j) {
      double acc = 0.0;
      for (int c = 0; c < d_c; ++c)
        acc += w_uv[((int64_t)i * d_v + j) * d_c + c] * u_tilde[(int64_t)i * d_c + c];
      u[(int64_t)i * d_v + j] = acc;
    }
}

/* MLA explicit form ("MHA mode"): expand per-head content keys and values
 * k^C_t,i = W_UK,i c_t, v^C_t,i = W_UV,i c_t, form
 * Score_i,t = q^C_i . k^C_t,i + q^R_i . k^R_t, A = softmax(scale * Score) and
 * u_i = sum_t A_i,t v^C_t,i ([P2] "Low-Rank Joint Key-Value Compression",
 * "The Decoupled RoPE Solution", "Value Output Matrix Absorption"; [P4]
 * "MHA Mode").  Used only to pin the absorbed form on tiny inputs.
 * q_c [h][d_hc], q_r [h][d_r], c [s][d_c], k_r [s][d_r], w_uk [h][d_hc][d_c],
 * w_uv [h][d_v][d_c]; u [h][d_v], lse [h]. */
int kvo_mla_explicit(const double* q_c, const double* q_r, const double* c, const double* k_r,
                     const double* w_uk, const double* w_uv, int64_t s, int h, int d_c,
                     int d_r, int d_hc, int d_v, double scale, double* u, double* lse) {
  if (s <= 0) return -1;
  double* kc = (double*)malloc(sizeof(double) * (size_t)(s * d_hc));
  double* vc = (double*)malloc(sizeof(double) * (size_t)(s * d_v));
  double* sc = (double*)malloc(sizeof(double) * (size_t)s);
  for (int i = 0; i < h; ++i) {
    for (int64_t t = 0; t < s; ++t) {
      for (int j = 0; j < d_hc; ++j) {
        double acc = 0.0;
        for (int x = 0; x < d_c; ++x) acc += w_uk[((int64_t)i * d_hc + j) * d_c + x] * c[t * d_c + x];
        kc[t * d_hc + j] = acc;
      }
      for (int j = 0; j < d_v; ++j) {
        double acc = 0.0;
        for (int x = 0; x < d_c; ++x) acc += w_uv[((int64_t)i * d_v + j) * d_c + x] * c[t * d_c + x];
        vc[t * d_v + j] = acc;
      }
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < s; ++t) {
      double a = 0.0;
      for (int j = 0; j < d_hc; ++j) a += q_c[(int64_t)i * d_hc + j] * kc[t * d_hc + j];
      for (int j = 0; j < d_r; ++j) a += q_r[(int64_t)i * d_r + j] * k_r[t * d_r + j];
      sc[t] = scale * a;
      if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int j = 0; j < d_v; ++j) u[(int64_t)i * d_v + j] = 0.0;
    for (int64_t t = 0; t < s; ++t) {
      double p = exp(sc[t] - m);
      l += p;
      for (int j = 0; j < d_v; ++j) u[(int64_t)i * d_v + j] += p * vc[t * d_v + j];
    }
    for (int j = 0; j < d_v; ++j) u[(int64_t)i * d_v + j] /= l;
    lse[i] = m + log(l);
  }
  free(kc);
  free(vc);
  free(sc);
  return 0;
}

/* Explicit-form ("MHA mode") MLA over a chunk of q_len new tokens, causal
 * among them: the sequence's cached rows are t = 0 .. s-1 and the new tokens
 * are its last q_len rows, so token j sits at position s - q_len + j and, for
 * each head i, attends to the rows t <= s - q_len + j with
 *   k_t,i = [W_UK,i c_t | k_R,t],  q_j,i = [q^C_j,i | q^R_j,i],
 *   score_t = scale * q_j,i . k_t,i,  out_j,i = sum_t softmax(score)_t W_UV,i c_t
 * ([P2] "Low-Rank Joint Key-Value Compression", "The Decoupled RoPE
 * Solution"; [P4] "MHA Mode", "Prefill 为什么未必使用与 Decode 相同的吸收方式":
 * prefill expands k and v per head from the latent instead of absorbing).
 * A token whose position is negative (s < q_len) sees nothing: out 0, lse -inf.
 * q_c [q_len][h][d_hc], q_r [q_len][h][d_r], c [s][d_c], k_r [s][d_r],
 * w_uk [h][d_hc][d_c], w_uv [h][d_v][d_c]; out [q_len][h][d_v], lse [q_len][h]. */
int kvo_mla_prefill(const double* q_c, const double* q_r, const double* c, const double* k_r,
                    const double* w_uk, const double* w_uv, int64_t s, int q_len, int h,
                    int d_c, int d_r, int d_hc, int d_v, double scale, double* out, double* lse) {
  if (s < 0 || q_len <= 0 || h <= 0 || d_c <= 0 || d_r < 0 || d_hc <= 0 || d_v <= 0) return -1;
  int rc = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < h; ++i) {
    /* this head's keys and values for every cached row */
    double* kc = (double*)malloc(sizeof(double) * (size_t)((s > 0 ? s : 1) * d_hc));
    double* vc = (double*)malloc(sizeof(double) * (size_t)((s > 0 ? s : 1) * d_v));
    double* sc = (double*)malloc(sizeof(double) * (size_t)(s > 0 ? s : 1));
    if (!kc || !vc || !sc) {
      rc = -1;
      free(kc);
      free(vc);
      free(sc);
      continue;
    }
    for (int64_t t = 0; t < s; ++t) {
      for (int j = 0; j < d_hc; ++j) {
        double acc = 0.0;
        for (int x = 0; x < d_c; ++x) acc += w_uk[((int64_t)i * d_hc + j) * d_c + x] * c[t * d_c + x];
        kc[t * d_hc + j] = acc;
      }
      for (int j = 0; j < d_v; ++j) {
        double acc = 0.0;
        for (int x = 0; x < d_c; ++x) acc += w_uv[((int64_t)i * d_v + j) * d_c + x] * c[t * d_c + x];
        vc[t * d_v + j] = acc;
      }
    }
    for (int jt = 0; jt < q_len; ++jt) {
      const int64_t n = s - q_len + jt + 1;   /* rows this token sees */
      const double* qc = q_c + ((int64_t)jt * h + i) * d_hc;
      const double* qr = q_r + ((int64_t)jt * h + i) * d_r;
      double* o = out + ((int64_t)jt * h + i) * d_v;
      for (int j = 0; j < d_v; ++j) o[j] = 0.0;
      if (n <= 0) {
        lse[(int64_t)jt * h + i] = -INFINITY;
        continue;
      }
      double m = -INFINITY;
      for (int64_t t = 0; t < n; ++t) {
        double a = 0.0;
        for (int j = 0; j < d_hc; ++j) a += qc[j] * kc[t * d_hc + j];
        for (int j = 0; j < d_r; ++j) a += qr[j] * k_r[t * d_r + j];
        sc[t] = scale * a;
        if (sc[t] > m) m = sc[t];
      }
      double l = 0.0;
      for (int64_t t = 0; t < n; ++t) {
        const double p = exp(sc[t] - m);
        l += p;
        for (int j = 0; j < d_v; ++j) o[j] += p * vc[t * d_v + j];
      }
      for (int j = 0; j < d_v; ++j) o[j] /= l;
      lse[(int64_t)jt * h + i] = m + log(l);
    }
    free(kc);
    free(vc);
    free(sc);
  }
  return rc;
}

/* Stable merge of split-KV partial results.  Split w covered a disjoint token
 * range and produced its own normalised output o_w and log-sum-exp lse_w.
 * With M = max_w lse_w:  o = sum_w e^(lse_w - M) o_w / sum_w e^(lse_w - M),
 * lse = M + log sum_w e^(lse_w - M)  ([P4] "FlashMLA 解决的不是模型公式本身":
 * each KV tile yields a local max, normaliser and output, merged stably
 * without changing the exact semantics).  part_o: [W][n][dv], part_lse: [W][n];
 * out: [n][dv], lse: [n].  Splits with lse = -inf (empty) carry no weight. */
void kvo_lse_combine(const double* part_o, const double* part_lse, int W, int n, int dv,
                     double* out, double* lse) {
  for (int r = 0; r < n; ++r) {
    double M = -INFINITY;
    for (int w = 0; w < W; ++w)
      if (part_lse[(int64_t)w * n + r] > M) M = part_lse[(int64_t)w * n + r];
    for (int c = 0; c < dv; ++c) out[(int64_t)r * dv + c] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double den = 0.0;
    for (int w = 0; w < W; ++w) {
      double lw = part_lse[(int64_t)w * n + r];
      if (lw == -INFINITY) continue;
      double e = exp(lw - M);
      den += e;
      for (int c = 0; c < dv; ++c)
        out[(int64_t)r * dv + c] += e * part_o[((int64_t)w * n + r) * dv + c];
    }
    for (int c = 0; c < dv; ++c) out[(int64_t)r * dv + c] /= den;
    lse[r] = M + log(den);
  }
}
