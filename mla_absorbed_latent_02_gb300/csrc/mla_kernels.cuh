// Parameter blocks and launchers shared between the kernel translation units
// and the C-ABI layer (mla_api.cu). Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mla {

constexpr int D_NOPE = 128;
constexpr int D_ROPE = 64;
constexpr int D_C = 512;
constexpr int D_V = 128;
constexpr int ROW = D_C + D_ROPE;  // 576 bf16 per cached token
constexpr int PAGE = 64;           // paged-cache block size (tokens)
constexpr int TILE = 128;          // tokens per attention tile (MMA M)
constexpr int MAX_SEQS = 1024;     // sequences per mla_decode_attn call

// ----------------------------------------------------------------- append
struct AppendParams {
  uint16_t* cache;
  int paged, num_seqs, capacity, num_blocks, max_blocks;
  const int32_t* block_table;
  const uint16_t* c_kv;    // [n, 512]
  const uint16_t* k_rope;  // [n, 64] before RoPE
  const int32_t* seq_idx;  // [n]
  const int32_t* pos;      // [n]
  int n;
  const float2* rope;      // [max_pos, 32] (cos, sin)
  int max_pos;
  int* status;
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);

// Latent producer: y = W_KV_A h (fp32, [n, 576]) -> optional RMSNorm of the
// latent, RoPE of the key, bf16 cache row (the append addressing in `a`).
struct LatentFinishParams {
  AppendParams a;          // cache, indices, RoPE table, n, status (c_kv / k_rope unused)
  const float* y;          // [n, 576]
  const uint16_t* kv_norm; // [512] bf16 RMSNorm weight, or null for no norm
  float eps;
};
cudaError_t launch_latent_finish(const LatentFinishParams& q, cudaStream_t s);

// Latent producer in one cooperative launch (split-K GEMM into per-split
// partial slots, grid barrier, per-token finish). Grid (LP_FEATURE_TILES, S,
// token blocks); ws holds S x n x 576 fp32 partials; sync: two zeroed words of
// the context (the grid barrier's arrival count).
constexpr int LP_FEATURE_TILES = 5;   // 128-feature tiles over the 576 outputs
#ifndef MLA_LP_MAX_SPLITS
#define MLA_LP_MAX_SPLITS 16
#endif
constexpr int LP_MAX_SPLITS = MLA_LP_MAX_SPLITS;   // partial slots per token at most
constexpr int LP_SYNC_WORDS = 32;     // grid-barrier word (a 128-byte line of its own)
struct LatentProjParams {
  LatentFinishParams fin;  // cache, indices, RoPE table, n, status, kv_norm, eps
  float* ws;               // [S, n, 576] fp32
  int KB;                  // 64-column blocks of the contraction (d_model / 64)
  int S;                   // K splits
  int rows_box;            // h TMA box height (token rows of a block, rounded up to 8)
  unsigned* sync;          // [LP_SYNC_WORDS]: word 0 counts arrivals
};
// K splits for n tokens (0 when the token blocks do not fit on the GPU at once).
int latent_proj_splits(int n, int KB, int num_sms);
// tm_w: W_KV_A as {d_model, 576} bf16, box {64, 128}; tm_x: h as {d_model, n},
// box {64, rows_box}; both 128-byte swizzle.
cudaError_t launch_latent_proj(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const LatentProjParams& q,
                               cudaStream_t s);

// ----------------------------------------------------------------- fused short-sequence step
// append + absorb_q + attention + expand_v for one new token per sequence
// (Hq = 1), sequences of at most SMALL_MAX_LEN tokens; a cluster of four CTAs
// per (sequence, head). a: the cache, the new tokens' c_kv [B, 512] and k_rope
// [B, 64] (row b goes to position seq_lens[b] - 1), RoPE table, status.
constexpr int SMALL_MAX_LEN = 4096;
struct SmallStepParams {
  AppendParams a;
  const uint16_t* w_uk;    // [H, 128, 512]
  const uint16_t* w_uv;    // [H, 128, 512]
  const uint16_t* q_nope;  // [B, H, 128]
  const uint16_t* q_rope;  // [B, H, 64] before RoPE
  const int32_t* seq_lens; // [B], the new token included
  int H;
  float scale;
  uint16_t* out;           // [B, H, 128] bf16
  float* o_lat;            // [B, H, 512]
  float* lse;              // [B, H]
};
size_t small_step_smem_bytes();
cudaError_t launch_small_step(const SmallStepParams& p, int B, cudaStream_t s);

// ----------------------------------------------------------------- absorb_q
// TMA box height for the rows of an activation operand: the valid rows, rounded
// up to a whole 8-row swizzle atom, at most one 128-row MMA tile. Rows past it in
// shared memory hold stale values that only reach output rows that are not stored.
inline int rows_box_for(long long M) { return M >= 128 ? 128 : static_cast<int>((M + 7) / 8 * 8); }

struct AbsorbParams {
  int H, M;                // M = B*Hq query rows
  int rows_box;            // q_nope TMA box height (rows_box_for(M))
  const int32_t* q_pos;    // [M]
  const uint16_t* q_rope;  // [M, H, 64] before RoPE
  uint16_t* q_abs;         // [M, H, 576]
  const float2* rope;
  int max_pos;
  int* status;
};
cudaError_t launch_absorb_q(const CUtensorMap& tm_qnope, const CUtensorMap& tm_wuk,
                            const AbsorbParams& p, cudaStream_t s);
// absorb_q and the cache append (bf16 or FP8 rows) in one launch (two when
// absorb_q alone needs more than num_sms CTAs)
cudaError_t launch_append_absorb_q(const CUtensorMap& tm_qnope, const CUtensorMap& tm_wuk, const AbsorbParams& p,
                                   const AppendParams& a, bool fp8, int num_sms, cudaStream_t s);

// ----------------------------------------------------------------- expand_v
struct ExpandParams {
  int H, M;
  int rows_box;            // o_lat TMA box height (rows_box_for(M))
  const float* o_lat;      // [M, H, 512]
  uint16_t* out;           // [M, H, 128]
  int* status;
};
constexpr int EXPAND_KS = 4;   // CTAs of the cluster variant that split the 512-wide contraction
// tm_wuv: W_UV as {512, 128, H} bf16, box {64, 128, 1};
// tm_olat: o_lat as {512, H, M} fp32, box {32, 1, 128}; both 128-byte swizzle.
cudaError_t launch_expand_v(const CUtensorMap& tm_wuv, const CUtensorMap& tm_olat, const ExpandParams& p,
                            int num_sms, cudaStream_t s);

// ----------------------------------------------------------------- output projection
constexpr int OP_SYNC_TILES = 1024;   // output tiles a split-K out_proj launch may have
struct OutProjParams {
  int d_model, M;          // output features, rows
  int KB;                  // 64-column blocks of the contraction (H*128/64)
  int rows_box;            // x TMA box height: rows of a block, rounded up to 8
  float* y;                // [M, d_model] fp32, fully written by the launch
  unsigned* sync;          // [3 * OP_SYNC_TILES] per output tile: ticket, zeroed flag, done count (zero between calls)
  int* status;
};
int out_proj_nb(int M);    // rows per block (the MMA's N): 32, 64, 128 or 256
// tm_w: W_O as {H*128, d_model} bf16, box {64, 128}; tm_x: o as {H*128, M} bf16,
// box {64, rows_box}; both 128-byte swizzle.
cudaError_t launch_out_proj(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p, int num_sms,
                            cudaStream_t s);

// W_OV [d_model, H*512] bf16 = W_O (per head) x W_UV[h] (a one-time weight
// transform; d_model a multiple of 64).
cudaError_t launch_absorb_w_o(const uint16_t* w_o, const uint16_t* w_uv, uint16_t* w_ov, int H, int d_model,
                              cudaStream_t s);
// y += W_OV x over x = o_lat [M, H*512] fp32 (y zero-filled before the launch);
// p.KB = H*512/64. tm_w: W_OV as {H*512, d_model} bf16, box {64, 128}, 128-byte
// swizzle; tm_x: o_lat as {H*512, M} fp32, box {32, rows_box}, 128-byte swizzle.
cudaError_t launch_out_proj_latent(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p,
                                   int num_sms, cudaStream_t s);

// ----------------------------------------------------------------- decode attention
struct AttnParams {
  int B, H, Hq, G;         // G = Hq*H query rows per sequence
  int N, C, U;             // rows per CTA, CTAs per unit, units
  int paged, capacity, num_seqs, num_blocks, max_blocks;
  int slots;               // pair kernel, one unit: CTA pairs launched (each walks several row-group pairs); 0: one each
  const int32_t* block_table;
  const int32_t* seq_lens;
  const uint8_t* cache;    // cache storage: row r at cache + r * ROW * 2 (L2 prefetch hints)
  const uint16_t* q_abs;   // [B*G, 576] bf16 (the FP8 kernel reads the latent queries directly)
  float scale_log2;        // softmax scale * log2(e)
  float* o_lat;            // [B, G, 512]
  float* lse;              // [B, G]
  float* ws_o;             // [(B+U), G, 512]
  float* ws_lse;           // [(B+U), G]
  int* status;
};
// Rows per CTA and CTAs per unit for G query rows per sequence: G = 16..64 in
// steps of 16 on one CTA, larger G (several query tokens per sequence: a
// multi-token decode step or a prefill chunk) in groups of 64 rows, up to
// MAX_ROWS_PER_SEQ. When the C CTAs of a unit outnumber the SMs the call runs as
// one unit (no split, CTAs in waves) and each CTA stops at the last tile its
// query tokens can see.
constexpr int MAX_ROWS_PER_SEQ = 1 << 20;
inline bool attn_split(int G, int& N, int& C) {
  if (G <= 0 || G % 16) return false;
  if (G <= 64) { N = G; C = 1; return true; }
  if (G % 64 || G > MAX_ROWS_PER_SEQ) return false;
  N = 64; C = G / 64;
  return true;
}
size_t attn_smem_bytes(int N);
cudaError_t attn_prepare(int N);  // sets the dynamic shared-memory attribute
cudaError_t launch_decode_attn(const CUtensorMap& tm_cache, const CUtensorMap& tm_q,
                               const AttnParams& p, cudaStream_t s);
cudaError_t launch_combine(const AttnParams& p, cudaStream_t s);
// The same attention for N = 64 and an even C on CTA pairs (clusters of two,
// tcgen05 .cta_group::2): each pair owns 128 query rows. prepare() sets the
// shared-memory attribute and returns how many pairs fit on the GPU at once.
size_t attn_pair_smem_bytes();
cudaError_t attn_pair_prepare(int* max_pairs);
cudaError_t launch_decode_attn_pair(const CUtensorMap& tm_cache, const CUtensorMap& tm_q, const AttnParams& p,
                                    cudaStream_t s);

// ----------------------------------------------------------------- FP8 latent cache
// Row of the FP8 cache (656 bytes): e4m3 codes of c_kv / sigma (512 bytes) |
// RoPE'd key, bf16, the bits the bf16 cache stores (128 bytes) | sigma, float32,
// a power of two (4 bytes) | 12 zero bytes.
constexpr int ROW8 = 656;
constexpr int ROW8_ROPE = 512;
constexpr int ROW8_SCALE = 640;
constexpr int FP8_SCALE_EXP_MIN = -64;  // sigma >= 2^-64
// Append into the FP8 cache; p.cache points at its rows (ROW8 bytes apart).
cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s);
size_t attn8_smem_bytes(int N);
cudaError_t attn8_prepare(int N);
// tm_c8: the cache rows as bytes {656, rows}, box {128, 64}, 128-byte swizzle
// (latent column groups and the RoPE key); tm_sc: the same bytes, box {16, 64},
// no swizzle (the scales); tm_qr: q_abs as bf16 {576, B*G}, box {64, N},
// 128-byte swizzle (the RoPE query block).
cudaError_t launch_decode_attn_fp8(const CUtensorMap& tm_c8, const CUtensorMap& tm_sc, const CUtensorMap& tm_qr,
                                   const AttnParams& p, cudaStream_t s);

// ----------------------------------------------------------------- launch
// Launch with programmatic stream serialization (the kernel overlaps its
// set-up with the previous kernel's tail; it waits before touching memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------- misc
cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t s);
// bytes (a multiple of 16) from src to dst by a kernel; 16-byte aligned pointers,
// device or device-addressable pinned host memory
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t s);

}  // namespace mla
