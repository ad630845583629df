/*
 * mla.h -- C ABI of the absorbed-latent MLA decode library (GB300, sm_103a).
 *
 * The library implements DeepSeek Multi-head Latent Attention decode in its
 * weight-absorbed form over a cache that stores one 576-element bf16 row per
 * token: the shared 512-dim KV latent c_kv followed by the shared 64-dim
 * decoupled RoPE key ("DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界"
 * §2.2-§2.4 and §4; "80 行 PyTorch 从零写 DeepSeek 的 MLA" §4-§5).
 *
 * Fixed dimensions: d_nope = 128, d_rope = 64, d_c = 512, d_v = 128, row = 576.
 * Variable: heads H (16, 32, 64 or 128), query tokens per sequence Hq, batch B.
 * Hq * H must be 16, 32 or 64, or a multiple of 64 up to 2^20: one decode
 * token (Hq = 1), a multi-token step (Hq = 2), or a prefill chunk of Hq query
 * tokens per sequence (up to 2^20 / H: 65,536 at H = 16, 8,192 at H = 128).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers the caller allocated and owns; the
 *    library allocates nothing in these calls. bf16 tensors are passed as
 *    `void*` (IEEE bfloat16 bit patterns), rows dense and 16-byte aligned.
 *  - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t,
 *    NULL = the legacy default stream). Device-side argument faults (an index
 *    out of range, a bad length) do not trap: they set bits in the context's
 *    device status word, read with mla_get_device_status().
 *  - Every call returns MLA_OK or an error code; mla_last_error() gives text.
 *    No C++ exception crosses the ABI. Calls on one context are not
 *    thread-safe with respect to each other.
 *  - The GPU must be compute capability 10.3 (sm_103a, GB300).
 *  - Consecutive calls on a stream overlap (programmatic dependent launch): a
 *    call may read its weights and some inputs before the previous MLA call on
 *    the stream has finished, so those must not be outputs of that previous
 *    call. Read early: c_kv, k_rope, seq_idx, pos and the block table
 *    (mla_append_latent); w_uk, q_nope, q_rope, q_pos (mla_absorb_q); seq_lens and
 *    the block table (mla_decode_attn); w_uv (mla_expand_v); w_o (mla_out_proj);
 *    w_kv_a (mla_project_latent). Everything else, and every write, waits for
 *    the previous call: the cache after an append, q_abs, o_lat, o, h.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or shape */
  MLA_ERR_UNSUPPORTED = 2, /* a shape the library does not handle, or not an sm_103 GPU */
  MLA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
  MLA_ERR_TIMEOUT = 4,     /* device status: a bounded wait inside a kernel ran out */
  MLA_ERR_BOUNDS = 5       /* device status: an index or length was out of range */
} mla_status_t;

/* Device status bits returned by mla_get_device_status(). */
#define MLA_DEVICE_BOUNDS 1  /* cache slot, block id or position out of range */
#define MLA_DEVICE_TIMEOUT 2 /* a kernel gave up waiting (its outputs are invalid) */
#define MLA_DEVICE_LENGTH 4  /* a sequence shorter than Hq tokens (output zeroed) */

typedef struct mla_ctx mla_ctx_t;

/*
 * Latent cache descriptor. Rows are [c_kv (512) | RoPE'd k_rope (64)] bf16,
 * 1,152 bytes each.
 *  contiguous (paged = 0): base is [num_seqs, capacity, 576]; token t of
 *    sequence s lives in row s * capacity + t.
 *  paged (paged = 1): base is a pool [num_blocks, 64, 576]; token t of sequence
 *    s lives in row block_table[s * max_blocks + t / 64] * 64 + t % 64.
 *    block_table is a device int32 array [num_seqs, max_blocks].
 * A paged cache with 64-token blocks is named in "DeepSeek-V2-Lite 真实权重执行审计"
 * §3.3; the block size and layout are this library's.
 */
typedef struct {
  void* base;
  int32_t paged;
  int32_t num_seqs;
  int32_t capacity;            /* contiguous: rows per sequence */
  int32_t num_blocks;          /* paged: blocks in the pool */
  const int32_t* block_table;  /* paged: device [num_seqs, max_blocks] */
  int32_t max_blocks;          /* paged: columns of block_table */
} mla_cache_t;

/*
 * Create a context on CUDA device `device`. Builds the RoPE table for positions
 * [0, max_pos): for pair i < 32, theta_i = 1 / rope_base^(2i/64), and
 * cos/sin(pos * theta_i) computed in double precision on the host and rounded
 * to float (interleaved-pair RoPE of "80 行 PyTorch 从零写 DeepSeek 的 MLA",
 * Appendix A). This call allocates the table and a status word on the device,
 * and looks up the device address of the static split-KV scratch used by
 * mla_decode_attn_static_scratch (16 MiB, committed once per device).
 * Errors: MLA_ERR_INVALID_ARG (null out, max_pos <= 0, rope_base <= 0),
 * MLA_ERR_UNSUPPORTED (device is not sm_103), MLA_ERR_CUDA.
 */
mla_status_t mla_create(mla_ctx_t** out, int32_t device, int32_t max_pos, double rope_base);

/* Free the context and its device allocations (synchronizes the device). */
mla_status_t mla_destroy(mla_ctx_t* ctx);

/* Text of the last error on this context ("" if none). Owned by the context. */
const char* mla_last_error(const mla_ctx_t* ctx);

/* Number of SMs of the context's device. */
int32_t mla_num_sms(const mla_ctx_t* ctx);

/*
 * Append n tokens to the cache (the cache-concat step, "80 行 PyTorch 从零写
 * DeepSeek 的 MLA" §2; the 576-element per-token contract, "DeepSeek MLA
 * 吸收式缓存" §2.4). For token k:
 *   row(seq_idx[k], pos[k])[0:512]   = c_kv[k, :]            (bytes copied)
 *   row(seq_idx[k], pos[k])[512:576] = RoPE_pos[k](k_rope[k, :])
 * RoPE pair i maps (a, b) -> (a*c - b*s, b*c + a*s) with c, s the context's
 * float table at pos[k]; each product and sum is a separately rounded float
 * operation (no FMA), and the result is rounded to bf16 (nearest even), so the
 * stored bytes are exactly reproducible.
 *  c_kv   : device bf16 [n, 512];  k_rope: device bf16 [n, 64] (before RoPE)
 *  seq_idx: device int32 [n];      pos   : device int32 [n]
 * A token whose slot is out of range (seq_idx, pos >= max_pos, capacity or
 * block table bounds) is skipped and sets MLA_DEVICE_BOUNDS.
 * Errors: MLA_ERR_INVALID_ARG (null/misaligned pointers, n < 0, bad descriptor).
 */
mla_status_t mla_append_latent(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv,
                               const void* k_rope, const int32_t* seq_idx, const int32_t* pos,
                               int32_t n, void* stream);

/*
 * Absorb the query into latent space (key absorption, "DeepSeek MLA 吸收式缓存"
 * §2.2; "80 行 PyTorch 从零写 DeepSeek 的 MLA" §4 path B) and rotate its RoPE
 * part. For row r = b*Hq + j and head h:
 *   q_abs[r, h, 0:512]   = bf16( W_UK[h]^T q_nope[r, h, :] )   (fp32 accumulation)
 *   q_abs[r, h, 512:576] = RoPE_{q_pos[r]}(q_rope[r, h, :])    (as in append)
 *  w_uk  : device bf16 [H, 128, 512] (nn.Linear(512 -> H*128) weight, per head)
 *  q_nope: device bf16 [B, Hq, H, 128]; q_rope: device bf16 [B, Hq, H, 64]
 *  q_pos : device int32 [B, Hq], the absolute position of each query token
 *  q_abs : device bf16 [B, Hq, H, 576] (output)
 * The softmax scale is not folded in; mla_decode_attn applies it in fp32.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H), MLA_ERR_CUDA.
 */
mla_status_t mla_absorb_q(mla_ctx_t* ctx, int32_t H, const void* w_uk, const void* q_nope,
                          const void* q_rope, const int32_t* q_pos, int32_t B, int32_t Hq,
                          void* q_abs, void* stream);

/*
 * mla_append_latent and mla_absorb_q in one launch (the two calls' work is
 * independent: the new cache rows and the absorbed queries), so that a decode
 * step pays for one kernel boundary less; when absorb_q alone needs more CTAs
 * than the GPU has SMs (H * 4 * ceil(B*Hq/128) > SMs) the two kernels are
 * launched one after the other instead, which is faster there. Arguments,
 * results, inputs read early and errors are those of the two calls; n = 0
 * appends nothing.
 * mla_append_fp8_absorb_q writes FP8 cache rows (as mla_append_latent_fp8).
 */
mla_status_t mla_append_absorb_q(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv,
                                 const void* k_rope, const int32_t* seq_idx, const int32_t* pos,
                                 int32_t n, int32_t H, const void* w_uk, const void* q_nope,
                                 const void* q_rope, const int32_t* q_pos, int32_t B, int32_t Hq,
                                 void* q_abs, void* stream);
mla_status_t mla_append_fp8_absorb_q(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv,
                                     const void* k_rope, const int32_t* seq_idx, const int32_t* pos,
                                     int32_t n, int32_t H, const void* w_uk, const void* q_nope,
                                     const void* q_rope, const int32_t* q_pos, int32_t B, int32_t Hq,
                                     void* q_abs, void* stream);

/*
 * Bytes of device workspace mla_decode_attn needs for (H, B, Hq): split-KV
 * partial outputs and their log-sum-exp. 0 on invalid arguments.
 */
size_t mla_decode_workspace_size(mla_ctx_t* ctx, int32_t H, int32_t B, int32_t Hq);

/*
 * Attention over the latent cache (the absorbed single pass, "DeepSeek MLA
 * 吸收式缓存" §2.2-§2.3; "80 行 PyTorch 从零写 DeepSeek 的 MLA" §5). Sequence b
 * holds seq_lens[b] tokens (the new ones included); its query j sits at
 * position seq_lens[b] - Hq + j and attends tokens t <= that position. For
 * query row g = j*H + h:
 *   s_t   = scale * (q_abs[b, g, :] . row_t)
 *   o_lat[b, g, :] = sum_t softmax(s)_t * row_t[0:512]      (fp32)
 *   lse[b, g]      = log sum_t exp(s_t)                      (natural log)
 *  q_abs   : device bf16 [B, Hq, H, 576] (from mla_absorb_q)
 *  B       : at most 1024 sequences per call (MLA_ERR_UNSUPPORTED above)
 *  seq_lens: device int32 [B] (read early, see the conventions above); a
 *            length below Hq sets MLA_DEVICE_LENGTH and
 *            zeroes that sequence's output (lse = -inf).
 *  scale   : softmax scale, e.g. 1/sqrt(d_nope + d_rope) = 1/sqrt(192)
 *  workspace, ws_bytes: device memory of at least mla_decode_workspace_size()
 *  o_lat   : device float [B, Hq, H, 512]; lse: device float [B, Hq, H]
 * Long or ragged batches are split across SMs (split-KV) and merged with a
 * log-sum-exp combine inside this call. A call whose Hq * H rows per sequence
 * need more CTAs (64 rows each) than the GPU has SMs (a long prompt chunk:
 * Hq * H > 64 * SMs) is not split: its CTAs run in waves, each over every
 * sequence up to the last tile its query tokens attend, and the workspace it
 * needs is 256 bytes.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA.
 */
mla_status_t mla_decode_attn(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache,
                             const void* q_abs, const int32_t* seq_lens, int32_t B, int32_t Hq,
                             float scale, void* workspace, size_t ws_bytes, float* o_lat,
                             float* lse, void* stream);

/*
 * mla_decode_attn for callers that cannot allocate device memory. (Not from the
 * pages: they have no counterpart of this call.)
 *
 * Some callers have no way to obtain a workspace: a serving runtime that hands
 * every byte of device memory to its own pool and forbids other allocations, an
 * embedded or real-time host thread that must not call cudaMalloc/cudaFree
 * (they can block and synchronize the device), or a plugin whose host offers no
 * allocator. This entry point computes exactly what mla_decode_attn computes,
 * with the same arguments minus the workspace: the split-KV partials go to a
 * scratch array that the library keeps in device memory
 * (mla_static_scratch_bytes() bytes = 16 MiB per GPU). It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *  - The array is part of the library's device image. mla_create looks up its
 *    device address on the context's device (cudaGetSymbolAddress, with that
 *    device current), which loads the image there, so the 16 MiB are committed
 *    when the context is created and stay until the process exits; no call of
 *    this entry point allocates or loads anything. A context does not outlive
 *    a reset of its device (cudaDeviceReset): create a new one after a reset.
 *  - Limit: shapes whose mla_decode_workspace_size() exceeds the scratch are
 *    rejected with MLA_ERR_UNSUPPORTED (the message gives both sizes); use
 *    mla_decode_attn for them. Arguments are checked first, exactly as
 *    mla_decode_attn checks them, with the same codes and messages.
 *  - All calls share the one scratch array, which keeps the previous call's
 *    contents (nothing in it needs to start at zero). Calls whose kernels
 *    overlap on the GPU (other streams, other threads, other contexts on the
 *    same device) race on it: order them.
 * Errors: as mla_decode_attn, plus MLA_ERR_UNSUPPORTED above the limit.
 */
mla_status_t mla_decode_attn_static_scratch(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache,
                                            const void* q_abs, const int32_t* seq_lens, int32_t B,
                                            int32_t Hq, float scale, float* o_lat, float* lse,
                                            void* stream);

/* Size in bytes of the scratch array used by mla_decode_attn_static_scratch. */
size_t mla_static_scratch_bytes(void);

/*
 * FP8 latent cache (FlashMLA's decoding with an FP8 KV cache in MQA mode,
 * "DeepSeek MLA 吸收式缓存" §6.1; the pages name the variant only, the row format
 * is this library's). Same descriptor and addressing as the bf16 cache, but a
 * row is 656 bytes (a page of 64 rows 41,984 bytes):
 *   bytes   0..511  e4m3 codes of c_kv / sigma (OCP E4M3, nearest, ties to even)
 *   bytes 512..639  the RoPE'd key, bf16: the bits mla_append_latent stores
 *   bytes 640..643  sigma, float32: the smallest power of two (at least 2^-64)
 *                   with max|c_kv| / sigma <= 448
 *   bytes 644..655  zero
 * The latent then costs 512 bytes per token instead of 1,024; c_kv is stored to
 * within 2^-4 of each value (relative), the RoPE key exactly as in bf16.
 *
 * mla_append_latent_fp8: as mla_append_latent (same arguments, inputs read
 * early alike), writing FP8 rows.
 * mla_decode_attn_fp8: as mla_decode_attn (same arguments, outputs and
 * workspace size) over FP8 rows: the latent row is codes * sigma. Scores and the
 * value aggregation run on e4m3 tensor-core products with the query and the
 * softmax weights each split into two e4m3 terms (hi + remainder), about bf16
 * precision; the RoPE part of the score stays bf16. The weights enter the
 * tensor-core product as p_t * sigma_t (the softmax weight times the token's
 * scale) relative to the running maximum of that product over the tokens seen
 * so far: they are carried to within 2^-22 of it (absolute) and smaller ones
 * are dropped when Hq * H <= 32; when Hq * H >= 64 the bound is 2^-18. A long
 * tail of weights near that bound can therefore shift the output by up to
 * (tokens x bound) relative to the exact attention over the rows.
 */
mla_status_t mla_append_latent_fp8(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv,
                                   const void* k_rope, const int32_t* seq_idx, const int32_t* pos,
                                   int32_t n, void* stream);
mla_status_t mla_decode_attn_fp8(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache,
                                 const void* q_abs, const int32_t* seq_lens, int32_t B, int32_t Hq,
                                 float scale, void* workspace, size_t ws_bytes, float* o_lat,
                                 float* lse, void* stream);

/*
 * A whole decode step for short sequences in one launch: mla_append_latent of
 * each sequence's new token, mla_absorb_q, mla_decode_attn and mla_expand_v
 * (the absorbed single pass of "DeepSeek MLA 吸收式缓存" §2.2-§2.4 and "80 行
 * PyTorch 从零写 DeepSeek 的 MLA" §4-§5), for one query token per sequence
 * (Hq = 1). Meant for the latency-bound case (few sequences of up to a few
 * hundred tokens, such as a single V2-Lite step), where the general path's four
 * dependent launches dominate; each (sequence, head) re-reads its sequence's
 * cache, so for long or many sequences the four calls are faster. Per
 * (sequence b, head h), with L = seq_lens[b] (the new token included):
 *   row(b, L-1)   = [c_kv[b] | RoPE_{L-1}(k_rope[b])]      (as mla_append_latent)
 *   q_lat         = W_UK[h]^T q_nope[b, h]                  (fp32, not rounded)
 *   s_t           = scale (q_lat . c_t + RoPE_{L-1}(q_rope[b, h]) . k_rope_t), t < L
 *   o_lat[b, h]   = sum_t softmax(s)_t c_t;  lse[b, h] = log sum_t exp(s_t)
 *   out[b, h]     = bf16(W_UV[h] o_lat[b, h])
 * all in fp32 on CUDA cores; the RoPE'd query and key are the bf16 values the
 * other calls use.
 *  c_kv, k_rope : device bf16 [B, 512], [B, 64] (pre-RoPE): the new tokens
 *  w_uk, w_uv   : device bf16 [H, 128, 512]
 *  q_nope, q_rope: device bf16 [B, H, 128], [B, H, 64] (pre-RoPE)
 *  seq_lens     : device int32 [B], at most mla_small_step_max_len() (4096):
 *                 a length of 0 or above it sets MLA_DEVICE_LENGTH and zeroes
 *                 that sequence's outputs (lse = -inf)
 *  out          : device bf16 [B, H, 128]; o_lat: device float [B, H, 512];
 *                 lse: device float [B, H]
 * Inputs read early: c_kv, k_rope, w_uk, w_uv, q_nope, q_rope, seq_lens and the
 * block table. The kernel needs no workspace.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H, B), MLA_ERR_CUDA.
 */
size_t mla_small_step_max_len(void);
mla_status_t mla_decode_step_small(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* c_kv,
                                   const void* k_rope, const void* w_uk, const void* w_uv, const void* q_nope,
                                   const void* q_rope, const int32_t* seq_lens, int32_t B, float scale, void* out,
                                   float* o_lat, float* lse, void* stream);

/*
 * Expand the latent result per head (value absorption applied after the
 * aggregation, "DeepSeek MLA 吸收式缓存" §2.3):
 *   out[r, h, :] = bf16( W_UV[h] o_lat[r, h, :] )   (128 <- 512, fp32 accumulation)
 *  w_uv : device bf16 [H, 128, 512]; o_lat: device float [B, Hq, H, 512]
 *  out  : bf16 [B, Hq, H, 128] in device memory, or in pinned host memory the
 *         device addresses directly (unified addressing): the kernel writes it
 *         with plain stores, so on a coherent host link the result reaches the
 *         host without a separate copy
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA.
 */
mla_status_t mla_expand_v(mla_ctx_t* ctx, int32_t H, const void* w_uv, const float* o_lat,
                          int32_t B, int32_t Hq, void* out, void* stream);

/*
 * Latent producer: the new tokens' cache rows from their hidden states
 * ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §2, Wdkv / Wkr; "DeepSeek-V2-Lite 真实权重
 * 执行审计" §3.3, kv_a_proj_with_mqa and kv_a_layernorm; "DeepSeek MLA 吸收式缓存"
 * §2.4, the 576-element cached row). For token k:
 *   y = W_KV_A h[k]                         (576 <- d_model, fp32 accumulation)
 *   c = y[0:512]; with kv_norm: c = c / sqrt(mean(c^2) + eps) * kv_norm (fp32)
 *   row(seq_idx[k], pos[k]) = [ bf16(c) | RoPE_pos[k](bf16(y[512:576])) ]
 * the RoPE part rotated exactly as mla_append_latent does.
 *  w_kv_a : device bf16 [576, d_model] (latent rows 0..511, RoPE-key rows 512..575)
 *  d_model: hidden width, a multiple of 64
 *  kv_norm: device bf16 [512] RMSNorm weight, or NULL for no normalisation
 *  h      : device bf16 [n, d_model]; seq_idx, pos: device int32 [n]
 *  workspace, ws_bytes: device memory of at least
 *           mla_project_latent_workspace_size(n) bytes (fp32 partial sums of
 *           the split contraction: up to 16 x n x 576 values)
 * One cooperative launch when the n tokens' row blocks (256 tokens each) fit
 * on the GPU five times over (n <= 7,680 on 152 SMs): the contraction is split
 * over the SMs into per-split partial slots, a grid-wide barrier follows, and
 * each token's partials are added in a fixed order before the norm, RoPE and
 * row write (deterministic results). Larger n: a split-K GEMM adding into the
 * workspace in L2 (low bits may vary from call to call), then the finish.
 * Calls on one context must not overlap on the GPU (the barrier uses the
 * context's words); a barrier that gives up sets MLA_DEVICE_TIMEOUT, and the
 * next mla_get_device_status() resets it.
 * Rows outside the cache set MLA_DEVICE_BOUNDS and are skipped, as in append.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (d_model), MLA_ERR_CUDA.
 */
size_t mla_project_latent_workspace_size(int32_t n);
mla_status_t mla_project_latent(mla_ctx_t* ctx, const mla_cache_t* cache, const void* w_kv_a, int32_t d_model,
                                const void* kv_norm, float eps, const void* h, const int32_t* seq_idx,
                                const int32_t* pos, int32_t n, void* workspace, size_t ws_bytes, void* stream);

/*
 * Prefill of a long prompt chunk in the expanded (MHA) form, for chunks long
 * enough that the naive form's arithmetic beats the absorbed one (FlashMLA's
 * "dense prefill, MHA mode", "DeepSeek MLA 吸收式缓存" §6.1; the expanded keys
 * and values of "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2-§3 and "DeepSeek MLA
 * 吸收式缓存" §2.1). For every sequence b < B the cache holds L_b = seq_lens[b]
 * tokens, the chunk's T new ones last (append them first, e.g. with
 * mla_append_latent); query j (0 <= j < T) sits at position L_b - T + j and
 * attends tokens 0 .. L_b - T + j:
 *   k_t = [W_UK[h] c_t ; k_rope_t]  (192),   v_t = W_UV[h] c_t  (128)
 *   q   = [q_nope ; RoPE_{q_pos}(q_rope)]
 *   out[b, j, h, :] = sum_t softmax_t(scale * q.k_t) v_t
 * the same quantity mla_absorb_q + mla_decode_attn + mla_expand_v compute with
 * Hq = T. Work per call: 2*H*256*512 flops per cached token (the expansion)
 * plus 2*H*320 per (query, key) pair, against 2*H*1088 per pair in the
 * absorbed form, so this form is the faster one for chunks of a few hundred
 * tokens and more.
 *  cache      : bf16 latent cache (the FP8 row format is not accepted)
 *  w_uk, w_uv : device bf16 [H, 128, 512]
 *  q_nope     : device bf16 [B, T, H, 128]
 *  q_rope     : device bf16 [B, T, H, 64] (before RoPE; rotated inside with the
 *               cache writer's float32 contract at q_pos)
 *  q_pos      : device int32 [B*T] RoPE positions of the queries
 *  seq_lens   : device int32 [B]; T <= seq_lens[b] <= max_len
 *  max_len    : host bound on seq_lens (sizes the workspace and the grid)
 *  workspace  : device memory of mla_prefill_mha_workspace_size(H, B, T,
 *               max_len) bytes (the expanded keys and values in bf16, then the
 *               rotated queries); nothing in it needs to start at zero
 *  out        : device bf16 [B, T, H, 128] (output)
 * Two launches: the expansion (a tcgen05 GEMM over the cached latent rows,
 * fp32 accumulation, bf16 out; it also rotates the queries) and a causal
 * attention kernel (fp32 online softmax, P in bf16, fp32 accumulation of P.V,
 * output rounded to bf16). K and V are rounded to bf16 after the expansion:
 * the rounding the absorbed form applies to q_abs falls on them here instead.
 * Inputs read early: w_uk, w_uv, seq_lens, the block table. Device-side:
 * seq_lens outside [T, max_len] set MLA_DEVICE_LENGTH (that sequence is
 * skipped, its output rows are not written); rows outside the cache or q_pos
 * outside the RoPE table set MLA_DEVICE_BOUNDS.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H, sizes), MLA_ERR_CUDA.
 */
size_t mla_prefill_mha_workspace_size(int32_t H, int32_t B, int32_t T, int32_t max_len);
mla_status_t mla_prefill_mha(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* w_uk, const void* w_uv,
                             const void* q_nope, const void* q_rope, const int32_t* q_pos, const int32_t* seq_lens,
                             int32_t B, int32_t T, int32_t max_len, float scale, void* workspace, size_t ws_bytes,
                             void* out, void* stream);

/*
 * Which form of a prefill chunk is the faster one: absorbed (mla_absorb_q +
 * mla_decode_attn + mla_expand_v with Hq = T) or expanded (mla_prefill_mha).
 * The choice between computing attention over the compressed latent and
 * decompressing K and V first ("DeepSeek MLA 吸收式缓存" §6.1 names FlashMLA's
 * MHA-mode prefill beside its absorbed decode) comes down to how many queries
 * see each cached key: the expansion costs 2*H*256*512 flops per cached token
 * and saves 2*H*(1088 - 320) per (query, key) pair. Host-only: no GPU, no
 * context. The estimate counts the work units of both forms (attended
 * triples, the split-KV units' key pages and query rows for the absorbed
 * form; expansion tiles, the attention's critical path in key tiles and its
 * items for the MHA form) with rates measured on a GB300; on 34 measured
 * chunks (H = 16 to 128, 16 to 1,024 new tokens, 11 of them not used in the
 * fit) it picks the faster form on all but one, where the two are within 1 %.
 *  H         : heads (16, 32, 64 or 128)
 *  B, T      : sequences and new tokens per sequence (T queries each)
 *  seq_lens  : HOST int32 [B]: tokens each sequence will hold, the chunk's
 *              included (T <= seq_lens[b])
 *  fp8_cache : nonzero for an FP8 cache (the MHA form reads bf16 caches only)
 *  ws_limit  : largest workspace the caller can give mla_prefill_mha, bytes
 *              (0: no limit)
 *  form      : out: MLA_PREFILL_ABSORBED or MLA_PREFILL_MHA. A form the
 *              library cannot run for this shape (the absorbed form's
 *              Hq * H rule, FP8, the workspace limit) is never chosen.
 *  est_us    : out, may be NULL: [2] estimated µs per step (append included)
 *              of the absorbed and the MHA form
 * Errors: MLA_ERR_INVALID_ARG (null seq_lens / form, B or T <= 0, a
 * seq_lens[b] < T), MLA_ERR_UNSUPPORTED (H, or neither form runs the shape).
 */
enum { MLA_PREFILL_ABSORBED = 0, MLA_PREFILL_MHA = 1 };
mla_status_t mla_prefill_choose_form(int32_t H, int32_t B, int32_t T, const int32_t* seq_lens, int32_t fp8_cache,
                                     size_t ws_limit, int32_t* form, double* est_us);

/*
 * Output projection of the attention block (the step after mla_expand_v, "80 行
 * PyTorch 从零写 DeepSeek 的 MLA" §2, the module's last line; "DeepSeek-V2-Lite
 * 真实权重执行审计" §3.3, o_proj / wo):
 *   y[r, :] = W_O concat_h(o[r, h, :])          (fp32 accumulation)
 * the heads concatenated head-major (row r of o viewed as H*128 values).
 *  w_o    : device bf16 [d_model, H*128] (nn.Linear(H*128 -> d_model) weight)
 *  d_model: output width, a multiple of 128 (2048 for V2-Lite, 7168 for V3)
 *  o      : device bf16 [M, H, 128] (from mla_expand_v, M = B*Hq rows)
 *  y      : device float [M, d_model] (output; the call overwrites it)
 * The contraction is split over many SMs and their fp32 partials are added
 * into y in L2, so the low bits of y may differ from call to call. y needs no
 * zero-fill: the first split of each output tile to start zeroes the tile and
 * raises a flag that the others check before adding. The flags are the
 * context's per-tile words, so calls on one context must not overlap on the
 * GPU; a wait that gives up sets MLA_DEVICE_TIMEOUT, and the next
 * mla_get_device_status() resets the words.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H, d_model), MLA_ERR_CUDA.
 */
mla_status_t mla_out_proj(mla_ctx_t* ctx, int32_t H, const void* w_o, int32_t d_model, const void* o,
                          int32_t M, float* y, void* stream);

/*
 * The value up-projection folded into the output projection: one weight for
 * both steps after the attention (the value absorption of "DeepSeek MLA
 * 吸收式缓存" §2.3, sum_t p_t W_UV c_t = W_UV sum_t p_t c_t, carried one matrix
 * further into the module's last line, "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2;
 * the pages themselves apply W_UV, then W_O).
 *   w_ov[f, h*512 + c] = bf16( sum_v w_o[f, h*128 + v] w_uv[h][v][c] )   (fp32 accumulation)
 * A one-time weight transform (run it when the weights are loaded).
 *  w_o : device bf16 [d_model, H*128]; w_uv: device bf16 [H, 128, 512]
 *  w_ov: device bf16 [d_model, H*512] (output; 4x the bytes of w_o)
 *  d_model: a multiple of 128
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H, d_model), MLA_ERR_CUDA.
 */
mla_status_t mla_absorb_w_o(mla_ctx_t* ctx, int32_t H, const void* w_o, int32_t d_model, const void* w_uv,
                            void* w_ov, void* stream);

/*
 * mla_expand_v followed by mla_out_proj as one projection of the attention's
 * latent output (the same y up to rounding):
 *   y[r, :] = W_OV concat_h(o_lat[r, h, :])            (fp32 accumulation)
 * with o_lat rounded to bf16 (nearest even) inside the kernel, where the
 * two-call path rounds the expanded o. One GEMM launch instead of two, over a
 * weight 4x as large as w_o: faster where the two calls are latency bound
 * (small d_model x H, e.g. V2-Lite), slower where they stream their weights at
 * bandwidth (e.g. V3 width).
 *  w_ov : device bf16 [d_model, H*512] from mla_absorb_w_o
 *  o_lat: device float [M, H, 512] (mla_decode_attn's output, M = B*Hq rows)
 *  y    : device float [M, d_model] (output; the call overwrites it)
 * The contraction is split over many SMs whose fp32 partials are added in L2
 * (into y, zero-filled first by the call), so the low bits of y may differ
 * from call to call. Inputs read early: w_ov.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H, d_model), MLA_ERR_CUDA.
 */
mla_status_t mla_out_proj_latent(mla_ctx_t* ctx, int32_t H, const void* w_ov, int32_t d_model, const float* o_lat,
                                 int32_t M, float* y, void* stream);

/*
 * Copy `bytes` bytes from src to dst on `stream` with a kernel (no copy-engine
 * transfer). Either side may be device memory or pinned host memory that the
 * device addresses directly (unified addressing): this is how a decode step's
 * inputs come from a pinned host buffer inside a CUDA graph, where a
 * copy-engine node between kernels cost ~12 us per step on GB300 against a few
 * microseconds for the kernel.
 * The kernel starts after the previous work in the stream has completed and
 * releases the next kernel only when every byte has landed, so the following
 * calls (including those that read their inputs before waiting on the kernel
 * in front of them) see the copied data.
 *  dst, src: 16-byte aligned, non-overlapping; bytes: a multiple of 16 (0: no-op)
 * Errors: MLA_ERR_INVALID_ARG (null, misaligned, bytes not a multiple of 16,
 * overlapping ranges), MLA_ERR_CUDA.
 */
mla_status_t mla_copy_async(mla_ctx_t* ctx, void* dst, const void* src, size_t bytes, void* stream);

/*
 * Synchronize `stream`, return the device status bits (MLA_DEVICE_*) set since
 * the last call in *status_out, and clear them.
 */
mla_status_t mla_get_device_status(mla_ctx_t* ctx, void* stream, int32_t* status_out);

/*
 * Tuning / test knob: number of split-KV units mla_decode_attn cuts the
 * flattened (sequence, 128-token tile) list into. 0 (default) = as many units
 * as fit on the GPU at once. Values above that are clamped. Affects
 * mla_decode_workspace_size().
 */
mla_status_t mla_set_decode_units(mla_ctx_t* ctx, int32_t units);

/*
 * Test hook for the kernels' bounded waits: launches one kernel that waits on a
 * barrier nothing completes, for limit_ns nanoseconds, then sets
 * MLA_DEVICE_TIMEOUT in the status word and returns. Faults nothing.
 */
mla_status_t mla_debug_wait_timeout(mla_ctx_t* ctx, uint64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
