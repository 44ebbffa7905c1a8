/*
 * kvattn.h -- C ABI of libkvattn.so: single-token decode attention over a
 * paged KV cache on NVIDIA GB300 (sm_103a).
 *
 * The operation (sources are named by page title and section):
 *   For each sequence b and query head i, with s_b cached positions
 *   (the current token included, appended before attending),
 *       o_i = softmax_t(scale * q_i . k_t) V,   lse_i = log sum_t exp(scale * q_i . k_t)
 *   - GQA/MQA/MHA: query head i reads KV head i / g, g = h / h_kv ("MHA -> MQA
 *     -> GQA -> MLA", mlinterviewnotes §3.5: "Query heads are broadcast against
 *     whatever KV heads exist"; "The KV cache size formula", §2.1: "Attention
 *     computes softmax(qK^T/sqrt(d_h))V against all previous positions").
 *   - MLA absorbed ("MQA mode"): each cached row is [c_KV (d_c) | k_R (d_rope)],
 *     the score is q~_i . row_t over the whole row and the output is the
 *     weighted latent sum sum_t p_t c_t, d_c wide ("Multi-Head Latent Attention
 *     (MLA): Mathematical Foundations, ...", sections "Attention Logit Matrix
 *     Absorption" and "Value Output Matrix Absorption").
 *   The cache is paged: token t of sequence b lives in block
 *   block_table[b][t / block_size] at slot t % block_size ("MLA：为什么一份
 *   Latent 可以代替多头 KV Cache", section "Paged KV Cache 的 Block 里放什么";
 *   "The KV cache size formula", section "vLLM: a per-layer page").
 *
 * Conventions for every call:
 *   - Ownership: the caller allocates and owns every buffer.  No call
 *     allocates device memory; scratch space comes from the caller's
 *     workspace (kvattn_decode_gqa_noalloc instead uses a fixed array that
 *     the library holds, described with it).  Pointers marked "device" must
 *     be device-accessible; a call only reads the host struct `kvattn_cache`
 *     during the call.
 *   - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Work is enqueued asynchronously; results are valid after the stream
 *     reaches that point.
 *   - CUDA graphs: the first call of an entry point on a device does one-time
 *     host set-up (kernel attributes, occupancy queries, the tensor-map
 *     encoder's address); make it outside any stream capture.  After it,
 *     kvattn_append, kvattn_decode_gqa, kvattn_decode_gqa_multi,
 *     kvattn_decode_mla, kvattn_mla_absorb_q, kvattn_mla_up_v and
 *     kvattn_mla_prefill only enqueue kernels on `stream`, so they can be
 *     captured in a CUDA graph and replayed.  Replays read the buffers the
 *     captured call was given, whatever they hold at replay time; the host
 *     struct and scalars are fixed at capture.
 *   - Errors: invalid arguments are rejected before any launch with
 *     KVATTN_ERR_INVALID_ARG or KVATTN_ERR_UNSUPPORTED and nothing is
 *     enqueued.  KVATTN_ERR_CUDA means a CUDA call or launch failed.
 *     Data-dependent faults found on the device (a block id outside the pool,
 *     a length longer than the block table row, a wait inside a kernel that
 *     gave up after its time limit of 0.2 s) never trap: the kernel skips or
 *     zero-fills the access, or stops and drains its copies, and ORs a
 *     KVATTN_DEVERR_* bit into *err (a device int32 the caller zeroes; err may
 *     be NULL).  Outputs touched by such a fault are unspecified but finite.
 *   - Layouts are row-major and densely packed unless stated.
 *   - Lengths of 0 are valid: that sequence's output rows are 0 and its lse
 *     rows are -inf.
 */
#ifndef KVATTN_H_
#define KVATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVATTN_ABI_VERSION 3

#if defined(__GNUC__)
#define KVATTN_API __attribute__((visibility("default")))
#else
#define KVATTN_API
#endif

typedef enum kvattn_status {
  KVATTN_OK = 0,
  KVATTN_ERR_INVALID_ARG = 1,   /* null pointer, bad count, inconsistent shape */
  KVATTN_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. head dim 96)     */
  KVATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed          */
  KVATTN_ERR_WORKSPACE = 4      /* workspace missing, misaligned or too small */
} kvattn_status;

/* Device-side error bits ORed into *err. */
#define KVATTN_DEVERR_BLOCK_ID 1  /* block_table entry outside [0, num_blocks)        */
#define KVATTN_DEVERR_SEQ_LEN 2   /* seq_len < 0 or > max_blocks_per_seq * block_size  */
#define KVATTN_DEVERR_POSITION 4  /* append: seq_idx or pos outside the table          */
#define KVATTN_DEVERR_TIMEOUT 8   /* a bounded barrier wait gave up                    */

typedef enum kvattn_kind { KVATTN_GQA = 0, KVATTN_MLA = 1 } kvattn_kind;
typedef enum kvattn_dtype { KVATTN_BF16 = 0, KVATTN_FP8_E4M3 = 1 } kvattn_dtype;

/* Non-owning view of one layer's paged cache.
 *   GQA: two pools, K and V, each [num_blocks][h_kv][block_size][d_h]
 *        (one contiguous block_size x d_h chunk per (block, KV head); "MHA
 *        takes two buffers per layer indexed by KV head", "The KV cache size
 *        formula", section "SGLang: one cell size, one division").
 *   MLA: one pool [num_blocks][block_size][d_c + d_rope], each row
 *        [c_KV | k_R] ("page / token i: [c_KV | k_R]", "MLA：为什么一份
 *        Latent ...", section "Paged KV Cache 的 Block 里放什么").
 *   Element type: bf16, or FP8-E4M3 codes with one scale per tensor: GQA
 *   code * k_scale (K) or code * v_scale (V); MLA code * k_scale for the c_KV
 *   part of a row and code * v_scale for its k_R part (c_KV and k_R are
 *   quantised separately: "MLA：为什么一份 Latent ...", section "MLA 与 KV Cache
 *   量化可以叠加").
 * Pools must be 16-byte aligned; 256-byte alignment is recommended. */
typedef struct kvattn_cache {
  int32_t kind;        /* kvattn_kind                                   */
  int32_t dtype;       /* kvattn_dtype                                  */
  int64_t num_blocks;  /* blocks in the pool                            */
  int32_t block_size;  /* tokens per block                              */
  int32_t h_kv;        /* GQA: KV heads (MLA: 1)                        */
  int32_t d_h;         /* GQA: head dim (MLA: ignored)                  */
  int32_t d_c;         /* MLA: latent width c_KV (512)                  */
  int32_t d_rope;      /* MLA: decoupled RoPE key width (64)            */
  float k_scale;       /* FP8 dequant scale of K / MLA c_KV (1.0 bf16)  */
  float v_scale;       /* FP8 dequant scale of V / MLA k_R (1.0 bf16)   */
  int32_t reserved;    /* must be 0                                     */
  void* k;             /* GQA K pool (device)                           */
  void* v;             /* GQA V pool (device)                           */
  void* latent;        /* MLA latent pool (device)                      */
} kvattn_cache;

/* Human-readable name of a status code; never NULL. */
KVATTN_API const char* kvattn_status_string(int status);

/* KVATTN_ABI_VERSION of the loaded library. */
KVATTN_API int kvattn_abi_version(void);

/* Bytes of one block of one layer: GQA 2 * h_kv * block_size * d_h * b,
 * MLA block_size * (d_c + d_rope) * b, b = 2 (bf16) or 1 (FP8) -- vLLM's
 * page_size_bytes with head_size_v = 0 for MLA ("The KV cache size formula",
 * section "vLLM: a per-layer page, then integer division").  Returns -1 on an
 * invalid descriptor. */
KVATTN_API int64_t kvattn_page_bytes(const kvattn_cache* cache);

/* Cell size, bytes per token over num_layers layers: GQA
 * 2 * L * h_kv * d_h * elem_bytes, MLA L * (d_c + d_rope) * elem_bytes (no
 * factor 2, no head count; "The KV cache size formula", sections on the
 * formula and "Where MLA breaks the formula").  Returns -1 on bad input. */
KVATTN_API int64_t kvattn_cell_bytes(int kind, int num_layers, int h_kv, int d_h, int d_c, int d_rope,
                          int elem_bytes);

/* Paged append: write n_tokens new tokens into their slots.
 *   Token n goes to sequence seq_idx[n] at position pos[n]:
 *   block = block_table[seq_idx[n] * max_blocks_per_seq + pos[n] / block_size],
 *   slot  = pos[n] % block_size.
 *   GQA: k_or_ckv = K [n_tokens][h_kv][d_h] bf16, v_or_kr = V, same shape.
 *        FP8 pools store e4m3(x / scale), x / scale in binary32, rounded to
 *        nearest even and saturated to +-448.
 *   MLA: k_or_ckv = c_KV [n_tokens][d_c] bf16, v_or_kr = k_R [n_tokens][d_rope]
 *        bf16 (already rotated by the caller); the row becomes [c_KV | k_R]
 *        ("MLA：为什么一份 Latent ...": "cache_j = [c_j^KV ; k_j^R]").  An
 *        FP8 pool stores c_KV as e4m3(x / k_scale) and k_R as
 *        e4m3(x / v_scale), rounded as for GQA.
 *   All pointers except cache are device pointers.  Tokens whose (seq, pos)
 *   falls outside the table or whose block id is outside the pool are skipped
 *   and flagged in *err.  Two tokens with the same slot race. */
KVATTN_API kvattn_status kvattn_append(const kvattn_cache* cache, const void* k_or_ckv, const void* v_or_kr,
                            int64_t n_tokens, const int32_t* seq_idx, const int32_t* pos,
                            const int32_t* block_table, int batch, int max_blocks_per_seq,
                            int32_t* err, void* stream);

/* Workspace bytes a decode call needs: the split plan ("tile scheduler
 * metadata and split info", "MLA：为什么一份 Latent ...", section "FlashMLA
 * 解决的不是模型公式本身") and the per-split partial outputs.  kind selects GQA
 * (dv = d_h) or MLA (dv = d_c).  num_ctas = 0 means the library's default for
 * the current device (this queries the device; it fails with 0 if there is
 * none).  Returns 0 on invalid input. */
KVATTN_API size_t kvattn_decode_workspace_bytes(int kind, int batch, int h, int h_kv, int dv, int num_ctas);

/* Default CTA count of a decode launch on the current device (SMs times
 * resident CTAs per SM for that kernel), or -1 without a device. */
KVATTN_API int kvattn_default_num_ctas(int kind, int dtype, int h, int h_kv, int d_h);

/* GQA / MQA / MHA decode.
 *   q:           device, [batch][h][d_h] bf16.
 *   cache:       host struct; kind GQA, h_kv and d_h must match the arguments.
 *   block_table: device, [batch][max_blocks_per_seq] int32.
 *   seq_lens:    device, [batch] int32, tokens cached per sequence (the
 *                current token included).
 *   h % h_kv == 0, g = h / h_kv <= 128 for d_h 128 (<= 64 for d_h 64);
 *   d_h in {64, 128} (FP8: 128);
 *   block_size a multiple of 16, at most 256 (vLLM's 16 up to one block of
 *   a short sequence).
 *   scale:       softmax scale (1/sqrt(d_h) in the pages' formula).
 *   out:         device, [batch][h][d_h] float32.
 *   lse:         device, [batch][h] float32, natural log; -inf for empty rows.
 *   workspace:   device, >= kvattn_decode_workspace_bytes(KVATTN_GQA, batch,
 *                h, h_kv, d_h, num_ctas) bytes, 256-byte aligned.
 *   num_ctas:    0 = default; otherwise the number of CTAs the page range is
 *                split over (tests use this to force split counts).
 * Launches three kernels on `stream`: the split planner, the decode kernel
 * and the split-KV combine.  Units of more than 32 rows (g, or q_len * g for
 * kvattn_decode_gqa_multi) with bf16, and of more than 16 with FP8, run on
 * the tensor cores' tcgen05 MMAs, the others on warp-level MMAs.  Results
 * depend on num_ctas only through rounding (the softmax weights enter P.V in
 * bf16, or as f16 or two E4M3 terms for FP8 caches). */
KVATTN_API kvattn_status kvattn_decode_gqa(const void* q, const kvattn_cache* cache,
                                const int32_t* block_table, const int32_t* seq_lens, int batch,
                                int max_blocks_per_seq, int h, int h_kv, int d_h, float scale,
                                float* out, float* lse, void* workspace, size_t workspace_bytes,
                                int num_ctas, int32_t* err, void* stream);

/* Multi-token GQA decode: q_len new tokens per sequence, all already in the
 * cache (speculative decoding verifies several draft tokens in one pass: "MLA：
 * 为什么一份 Latent 可以代替多头 KV Cache", section "Prefill 为什么未必使用与
 * Decode 相同的吸收方式" lists the tokens one verification checks among the
 * inputs of kernel selection, and section "正确性验证应该从两种实现互证" item 5
 * asks the kernel to be checked with speculative tokens).  Token j of sequence
 * b sits at position s_b - q_len + j and attends causally to positions
 * [0, s_b - q_len + j]; a token whose position would be negative (s_b < q_len)
 * sees nothing: out 0, lse -inf.  One K/V read serves all q_len * g rows of a
 * KV head.
 *   q:    device, [batch][q_len][h][d_h] bf16.
 *   out:  device, [batch][q_len][h][d_h] float32;  lse: [batch][q_len][h].
 *   q_len >= 1 (KVATTN_ERR_INVALID_ARG otherwise), q_len * g <= 128 for
 *   d_h 128, <= 64 for d_h 64 (KVATTN_ERR_UNSUPPORTED otherwise).
 *   workspace: >= kvattn_decode_workspace_bytes(KVATTN_GQA, batch, h * q_len,
 *   h_kv, d_h, num_ctas) bytes.
 * Other arguments, and the three launches, as for kvattn_decode_gqa, which is
 * this call with q_len = 1. */
KVATTN_API kvattn_status kvattn_decode_gqa_multi(const void* q, const kvattn_cache* cache,
                                const int32_t* block_table, const int32_t* seq_lens, int batch,
                                int max_blocks_per_seq, int q_len, int h, int h_kv, int d_h,
                                float scale, float* out, float* lse, void* workspace,
                                size_t workspace_bytes, int num_ctas, int32_t* err, void* stream);

/* MLA absorbed decode.
 *   q_absorbed:  device, [batch][h][d_c + d_rope] bf16: [W_UK^T q^C | q^R] per
 *                head ("Let us define the absorbed query vector").
 *   cache:       host struct; kind MLA, bf16 or FP8-E4M3 (k_scale, v_scale >
 *                0), block_size 64, d_c = 512, d_rope = 64; other shapes
 *                return KVATTN_ERR_UNSUPPORTED.
 *   h:           query heads, 1..128.
 *   scale:       softmax scale (1/sqrt(d_h^C + d_r) = 1/sqrt(192) for
 *                DeepSeek-V3 -- not 1/sqrt of the row width).
 *   out:         device, [batch][h][d_c] float32 (the latent sum u~).
 *   lse:         device, [batch][h] float32.
 *   workspace:   >= kvattn_decode_workspace_bytes(KVATTN_MLA, batch, h, 1, d_c,
 *                num_ctas) bytes.
 * Launches two kernels on `stream`: the split planner and the decode kernel,
 * which also merges the partials of sequences it split over several CTA
 * pairs.  Other arguments as for kvattn_decode_gqa. */
KVATTN_API kvattn_status kvattn_decode_mla(const void* q_absorbed, const kvattn_cache* cache,
                                const int32_t* block_table, const int32_t* seq_lens, int batch,
                                int max_blocks_per_seq, int h, int d_c, int d_rope, float scale,
                                float* out, float* lse, void* workspace, size_t workspace_bytes,
                                int num_ctas, int32_t* err, void* stream);

/* MLA query-side absorption ("MLA：为什么一份 Latent 可以代替多头 KV Cache" and
 * "Multi-Head Latent Attention (MLA) ...", the absorbed query vector): for every
 * batch row b and head i,
 *   q_absorbed[b][i] = [ W_UK,i^T q^C[b][i]  |  q^R[b][i] ],
 * the row kvattn_decode_mla takes.  W_UK,i maps a latent to head i's key
 * (k^C = W_UK,i c), so its transpose takes the head's query into latent space.
 *   q_nope:      device, [batch][h][d_hc] bf16 (q^C).
 *   q_rope:      device, [batch][h][d_rope] bf16 (q^R, already rotated; may
 *                be null when d_rope = 0).
 *   w_uk:        device, [h][d_hc][d_c] bf16 (W_UK,i row-major, d_c fastest).
 *   q_absorbed:  device, [batch][h][d_c + d_rope] bf16; the product is
 *                accumulated in float32 and rounded to nearest even.
 * Built for d_hc = 128, d_c a multiple of 256, d_rope a multiple of 8 with
 * d_c + d_rope <= 4096, ceil(batch / 128) and h at most 65535
 * (KVATTN_ERR_UNSUPPORTED otherwise).  All pointers 16-byte aligned
 * (KVATTN_ERR_INVALID_ARG otherwise).  One kernel on `stream` (tcgen05
 * tensor cores, one CTA per head, 128 batch rows and 256 latent columns);
 * a bounded wait that gives up sets KVATTN_DEVERR_TIMEOUT in *err and leaves
 * that CTA's rows unwritten. */
KVATTN_API kvattn_status kvattn_mla_absorb_q(const void* q_nope, const void* q_rope,
                                             const void* w_uk, int batch, int h, int d_hc,
                                             int d_c, int d_rope, void* q_absorbed, int32_t* err,
                                             void* stream);

/* MLA deferred value up-projection (same pages: W_UV,i moves outside the
 * probability-weighted sum over cached latents):
 *   v[b][i] = W_UV,i u~[b][i]
 * for the decode output u~ of kvattn_decode_mla.  W_O, which maps the
 * concatenated heads to the model width, is a plain GEMM over all heads and
 * is not part of this library.
 *   u_tilde:  device, [batch][h][d_c] float32.
 *   w_uv:     device, [h][d_v][d_c] bf16 (W_UV,i row-major, d_c fastest).
 *   v:        device, [batch][h][d_v] float32.
 * u~ is rounded to bf16 (nearest even) for the tensor cores; products are
 * accumulated in float32.  Built for d_v = 128 and d_c a multiple of 128 up
 * to 65536, ceil(batch / 128) and h at most 65535 (KVATTN_ERR_UNSUPPORTED
 * otherwise); pointers 16-byte aligned (KVATTN_ERR_INVALID_ARG otherwise).
 * One kernel on `stream`; error behaviour as for kvattn_mla_absorb_q. */
KVATTN_API kvattn_status kvattn_mla_up_v(const float* u_tilde, const void* w_uv, int batch, int h,
                                         int d_c, int d_v, float* v, int32_t* err, void* stream);

/* Explicit-form ("MHA mode") MLA prefill over the paged latent: q_len new
 * tokens per sequence, already appended (token j of sequence b sits at
 * position s_b - q_len + j), attend causally to the cached rows with keys and
 * values expanded per head from the latent,
 *   k_t,i = [W_UK,i c_t | k_R,t],  v_t,i = W_UV,i c_t,
 *   out_j,i = sum_{t <= s_b - q_len + j} softmax_t(scale * [q^C_j,i | q^R_j,i] . k_t,i) v_t,i
 * ("MLA：为什么一份 Latent 可以代替多头 KV Cache", sections "MHA Mode" and "Prefill
 * 为什么未必使用与 Decode 相同的吸收方式": prefill expands keys and values per
 * head, decode absorbs W_UK into the query; the last new token's result equals
 * the absorbed decode's followed by W_UV).  A token whose position would be
 * negative (s_b < q_len) sees nothing: out 0, lse -inf.
 *   q_nope:     device, [batch][q_len][h][d_hc] bf16 (q^C).
 *   q_rope:     device, [batch][q_len][h][64] bf16 (q^R, already rotated).
 *   cache:      host struct; kind MLA, bf16, d_c = 512, d_rope = 64, block 64.
 *   block_table, seq_lens: as for kvattn_decode_mla (seq_lens include the new
 *               tokens).
 *   w_uk, w_uv: device, [h][d_hc][d_c] and [h][d_v][d_c] bf16 (row-major, d_c
 *               fastest; the layouts of kvattn_mla_absorb_q and kvattn_mla_up_v).
 *   scale:      softmax scale (1/sqrt(d_hc + d_rope)).
 *   out:        device, [batch][q_len][h][d_v] float32;  lse: [batch][q_len][h].
 * Built for d_hc = d_v = 128, h and batch at most 65535 (KVATTN_ERR_UNSUPPORTED
 * otherwise).  Needs no workspace: the expanded keys and values of each tile
 * of 128 cached rows live only in the SM that uses them (tensor memory, then
 * shared memory).  One kernel on `stream`, one CTA per (128 new tokens, head,
 * sequence); device errors as for kvattn_decode_mla. */
KVATTN_API kvattn_status kvattn_mla_prefill(const void* q_nope, const void* q_rope,
                                            const kvattn_cache* cache, const int32_t* block_table,
                                            const int32_t* seq_lens, int batch,
                                            int max_blocks_per_seq, int q_len, int h, int d_hc,
                                            int d_v, const void* w_uk, const void* w_uv,
                                            float scale, float* out, float* lse, int32_t* err,
                                            void* stream);

/* Split-KV log-sum-exp combine.
 *   Unit u owns split_count[u] consecutive partial slots starting at
 *   split_first[u]; each slot holds rows_per_unit rows of a normalised partial
 *   output (part_out [slot][rows_per_unit][dv] float32) and its natural
 *   log-sum-exp (part_lse [slot][rows_per_unit]).  For every row:
 *     M = max_w lse_w,  out = sum_w e^(lse_w - M) o_w / sum_w e^(lse_w - M),
 *     lse = M + log sum_w e^(lse_w - M)
 *   ("MLA：为什么一份 Latent ...", section "FlashMLA 解决的不是模型公式本身":
 *   local max, normaliser and output per KV tile, merged stably).  Units with
 *   split_count 0 get zeros and -inf; splits whose lse is -inf carry no
 *   weight.  out [n_units][rows_per_unit][dv], lse [n_units][rows_per_unit].
 *   All pointers are device pointers; dv must be a multiple of 4 and
 *   part_out / out 16-byte aligned (KVATTN_ERR_INVALID_ARG otherwise);
 *   n_units * rows_per_unit must stay below 2^31 and dv at most 512
 *   (KVATTN_ERR_UNSUPPORTED otherwise). */
KVATTN_API kvattn_status kvattn_combine(const float* part_out, const float* part_lse,
                             const int32_t* split_first, const int32_t* split_count, int n_units,
                             int rows_per_unit, int dv, float* out, float* lse, void* stream);

/* Size of the scratch array built into the library for
 * kvattn_decode_gqa_noalloc: 8 MiB of device memory on every GPU that loads
 * the library, held until the process exits. */
#define KVATTN_NOALLOC_SCRATCH_BYTES (8u << 20)

/* GQA / MQA / MHA decode that allocates nothing and takes no workspace.
 *   The pages have no counterpart: this exists for callers that cannot give
 *   the library device memory -- a plugin or custom-op interface that passes
 *   only the op's inputs and outputs, a runtime whose memory all belongs to
 *   its own pool, or a path where cudaMalloc (which may synchronise the
 *   device) is not allowed.
 *   Arguments and results are those of kvattn_decode_gqa without `workspace`
 *   and `workspace_bytes`; the plan and the partial outputs go to a fixed
 *   scratch array inside the library (KVATTN_NOALLOC_SCRATCH_BYTES).
 *   - A problem whose kvattn_decode_workspace_bytes(KVATTN_GQA, batch, h, h_kv,
 *     d_h, num_ctas) exceeds KVATTN_NOALLOC_SCRATCH_BYTES is rejected with
 *     KVATTN_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before capturing any stream.
 *   - All calls on a device share the one array and it keeps what the last
 *     call left there; nothing in it needs to start at zero.  Calls whose work
 *     overlaps on the GPU (different streams, or different host threads without
 *     ordering) race on the array and corrupt each other's results: order them
 *     on one stream.
 *   - No cudaMalloc, cudaFree or other allocating call is made. */
KVATTN_API kvattn_status kvattn_decode_gqa_noalloc(const void* q, const kvattn_cache* cache,
                                                   const int32_t* block_table,
                                                   const int32_t* seq_lens, int batch,
                                                   int max_blocks_per_seq, int h, int h_kv,
                                                   int d_h, float scale, float* out, float* lse,
                                                   int num_ctas, int32_t* err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVATTN_H_ */
