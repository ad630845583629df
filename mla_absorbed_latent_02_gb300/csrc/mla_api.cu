// C-ABI layer: context, host-side argument checks, TMA descriptors, launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "mla.h"
#include "mla_kernels.cuh"
#include "prefill_mha.cuh"

struct mla_ctx {
  int device = 0;
  int num_sms = 0;
  int max_pos = 0;
  double rope_base = 10000.0;
  float2* d_rope = nullptr;  // [max_pos, 32]
  int* d_status = nullptr;
  unsigned* d_sync = nullptr;  // grid-barrier words of the one-launch latent producer
  unsigned* d_op_sync = nullptr;  // per-tile words of the split-K output projection
  int units_override = 0;
  bool attn_ready[65] = {};
  bool attn8_ready[65] = {};
  bool pair_ready = false;
  int attn_pairs = 0;        // CTA pairs of the 2-SM attention kernel that fit on the GPU at once
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  void* static_scratch = nullptr;  // device address of g_decode_scratch on `device`
  char err[512] = {0};
};

namespace {

mla_status_t fail(mla_ctx_t* ctx, mla_status_t code, const char* fmt, ...) {
  if (ctx) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(ctx->err, sizeof(ctx->err), fmt, ap);
    va_end(ap);
  }
  return code;
}

mla_status_t cuda_fail(mla_ctx_t* ctx, cudaError_t e, const char* what) {
  return fail(ctx, MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MLA_CUDA(ctx, call)                                \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool heads_ok(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }

// RAII device guard: make ctx->device current for the call.
struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

mla_status_t encode_map(mla_ctx_t* ctx, CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box, const char* what,
                        CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  uint32_t estr[3] = {1, 1, 1};
  const CUresult r = ctx->encode(map, dtype, rank, const_cast<void*>(base), dims, strides_bytes, box, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ctx, MLA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return MLA_OK;
}

mla_status_t check_cache(mla_ctx_t* ctx, const mla_cache_t* c) {
  if (!c || !c->base) return fail(ctx, MLA_ERR_INVALID_ARG, "cache descriptor or base is null");
  if (!aligned16(c->base)) return fail(ctx, MLA_ERR_INVALID_ARG, "cache base must be 16-byte aligned");
  if (c->num_seqs <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "cache num_seqs must be positive");
  if (c->paged) {
    if (c->num_blocks <= 0 || c->max_blocks <= 0 || !c->block_table)
      return fail(ctx, MLA_ERR_INVALID_ARG, "paged cache needs num_blocks, max_blocks and block_table");
    if ((long long)c->num_blocks * mla::PAGE >= (1ll << 31))
      return fail(ctx, MLA_ERR_UNSUPPORTED, "paged pool too large (rows must fit int32)");
  } else {
    if (c->capacity <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "contiguous cache capacity must be positive");
    if ((long long)c->num_seqs * c->capacity >= (1ll << 31))
      return fail(ctx, MLA_ERR_UNSUPPORTED, "contiguous cache too large (rows must fit int32)");
  }
  return MLA_OK;
}

// Split-KV scratch of mla_decode_attn_static_scratch, for callers that cannot
// allocate device memory: one file-scope device array instead of a
// caller-provided workspace. It is part of this library's device image, so a
// GPU holds its kStaticScratchBytes once the image is loaded there (mla_create
// loads it by looking up the array's address) until the process exits. On the
// host, `g_decode_scratch` names a stand-in object, never a device address.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

int decode_units(mla_ctx_t* ctx, int C) {
  const int max_units = ctx->num_sms / C;
  int u = ctx->units_override > 0 ? ctx->units_override : max_units;
  if (u > max_units) u = max_units;
  if (u < 1) u = 1;
  return u;
}

// Units of the 2-SM attention kernel: as many as its CTA pairs fit on the GPU
// at once (a pair needs two SMs of one cluster-capable group).
int pair_units(mla_ctx_t* ctx, int C) {
  int u = decode_units(ctx, C);
  const int fit = (2 * ctx->attn_pairs) / C;
  if (u > fit) u = fit;
  if (u < 1) u = 1;
  return u;
}

}  // namespace

extern "C" {

mla_status_t mla_create(mla_ctx_t** out, int32_t device, int32_t max_pos, double rope_base) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_pos <= 0 || !(rope_base > 0.0)) return MLA_ERR_INVALID_ARG;
  mla_ctx_t* ctx = new (std::nothrow) mla_ctx;
  if (!ctx) return MLA_ERR_CUDA;
  ctx->device = device;
  ctx->max_pos = max_pos;
  ctx->rope_base = rope_base;
  auto bail = [&](mla_status_t s) {
    if (ctx->d_rope) cudaFree(ctx->d_rope);
    if (ctx->d_status) cudaFree(ctx->d_status);
    if (ctx->d_sync) cudaFree(ctx->d_sync);
    if (ctx->d_op_sync) cudaFree(ctx->d_op_sync);
    delete ctx;
    return s;
  };
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (prop.major != 10 || prop.minor != 3) return bail(MLA_ERR_UNSUPPORTED);
  DeviceGuard g(device);
  ctx->num_sms = prop.multiProcessorCount;

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return bail(MLA_ERR_CUDA);
  ctx->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);

  // RoPE table: theta_i = 1 / base^(2i/64), angle pos * theta_i in double,
  // cos / sin in double, each rounded once to float.
  std::vector<float2> tab(static_cast<size_t>(max_pos) * 32);
  double inv[32];
  for (int i = 0; i < 32; ++i) inv[i] = 1.0 / std::pow(rope_base, (2.0 * i) / 64.0);
  for (int p = 0; p < max_pos; ++p)
    for (int i = 0; i < 32; ++i) {
      const double phi = static_cast<double>(p) * inv[i];
      tab[static_cast<size_t>(p) * 32 + i] = make_float2(static_cast<float>(std::cos(phi)),
                                                         static_cast<float>(std::sin(phi)));
    }
  if (cudaMalloc(&ctx->d_rope, tab.size() * sizeof(float2)) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (cudaMemcpy(ctx->d_rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
    return bail(MLA_ERR_CUDA);
  if (cudaMalloc(&ctx->d_status, sizeof(int)) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (cudaMemset(ctx->d_status, 0, sizeof(int)) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (cudaMalloc(&ctx->d_sync, mla::LP_SYNC_WORDS * sizeof(unsigned)) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (cudaMemset(ctx->d_sync, 0, mla::LP_SYNC_WORDS * sizeof(unsigned)) != cudaSuccess) return bail(MLA_ERR_CUDA);
  if (cudaMalloc(&ctx->d_op_sync, 3 * mla::OP_SYNC_TILES * sizeof(unsigned)) != cudaSuccess)
    return bail(MLA_ERR_CUDA);
  if (cudaMemset(ctx->d_op_sync, 0, 3 * mla::OP_SYNC_TILES * sizeof(unsigned)) != cudaSuccess)
    return bail(MLA_ERR_CUDA);
  // Device address of the static split-KV scratch on this device (which is
  // current). The lookup loads the module that holds the array, so its memory
  // is committed here, at set-up, and never inside a decode call.
  if (cudaGetSymbolAddress(&ctx->static_scratch, g_decode_scratch) != cudaSuccess || !ctx->static_scratch)
    return bail(MLA_ERR_CUDA);
  *out = ctx;
  return MLA_OK;
}

mla_status_t mla_destroy(mla_ctx_t* ctx) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  {
    DeviceGuard g(ctx->device);
    cudaDeviceSynchronize();
    if (ctx->d_rope) cudaFree(ctx->d_rope);
    if (ctx->d_status) cudaFree(ctx->d_status);
    if (ctx->d_sync) cudaFree(ctx->d_sync);
    if (ctx->d_op_sync) cudaFree(ctx->d_op_sync);
  }
  delete ctx;
  return MLA_OK;
}

const char* mla_last_error(const mla_ctx_t* ctx) { return ctx ? ctx->err : "null context"; }

int32_t mla_num_sms(const mla_ctx_t* ctx) { return ctx ? ctx->num_sms : 0; }

mla_status_t mla_set_decode_units(mla_ctx_t* ctx, int32_t units) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (units < 0) return fail(ctx, MLA_ERR_INVALID_ARG, "units must be >= 0");
  ctx->units_override = units;
  return MLA_OK;
}

}  // extern "C"

namespace {

// Checks the append arguments and fills p (p.n = 0: nothing to append).
mla_status_t build_append(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                          const int32_t* seq_idx, const int32_t* pos, int32_t n, mla::AppendParams& p) {
  if (mla_status_t s = check_cache(ctx, cache)) return s;
  if (n < 0) return fail(ctx, MLA_ERR_INVALID_ARG, "n must be >= 0");
  p = mla::AppendParams{};
  if (n == 0) return MLA_OK;
  if (!c_kv || !k_rope || !seq_idx || !pos) return fail(ctx, MLA_ERR_INVALID_ARG, "null input pointer");
  if (!aligned16(c_kv) || !aligned16(k_rope)) return fail(ctx, MLA_ERR_INVALID_ARG, "c_kv / k_rope must be 16-byte aligned");
  p.cache = static_cast<uint16_t*>(cache->base);
  p.paged = cache->paged;
  p.num_seqs = cache->num_seqs;
  p.capacity = cache->capacity;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = cache->max_blocks;
  p.block_table = cache->block_table;
  p.c_kv = static_cast<const uint16_t*>(c_kv);
  p.k_rope = static_cast<const uint16_t*>(k_rope);
  p.seq_idx = seq_idx;
  p.pos = pos;
  p.n = n;
  p.rope = ctx->d_rope;
  p.max_pos = ctx->max_pos;
  p.status = ctx->d_status;
  return MLA_OK;
}

mla_status_t append_impl(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                         const int32_t* seq_idx, const int32_t* pos, int32_t n, void* stream, bool fp8) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  mla::AppendParams p;
  if (mla_status_t st = build_append(ctx, cache, c_kv, k_rope, seq_idx, pos, n, p)) return st;
  if (p.n == 0) return MLA_OK;
  DeviceGuard g(ctx->device);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, fp8 ? mla::launch_append_fp8(p, s) : mla::launch_append(p, s));
  return MLA_OK;
}

// Checks the absorb_q arguments, encodes its tensor maps and fills p.
mla_status_t build_absorb(mla_ctx_t* ctx, int32_t H, const void* w_uk, const void* q_nope, const void* q_rope,
                          const int32_t* q_pos, int32_t B, int32_t Hq, void* q_abs, CUtensorMap& tq, CUtensorMap& tw,
                          mla::AbsorbParams& p) {
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (B <= 0 || Hq <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "B and Hq must be positive");
  if (!w_uk || !q_nope || !q_rope || !q_pos || !q_abs) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_uk) || !aligned16(q_nope) || !aligned16(q_rope) || !aligned16(q_abs))
    return fail(ctx, MLA_ERR_INVALID_ARG, "bf16 tensors must be 16-byte aligned");
  const long long M = (long long)B * Hq;
  if (M * H >= (1ll << 31)) return fail(ctx, MLA_ERR_UNSUPPORTED, "B*Hq*H too large");
  {
    const uint64_t dims[3] = {128, (uint64_t)H, (uint64_t)M};
    const uint64_t str[2] = {128 * 2, (uint64_t)H * 128 * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)mla::rows_box_for(M)};
    if (mla_status_t s = encode_map(ctx, &tq, q_nope, 3, dims, str, box, "q_nope")) return s;
  }
  {
    const uint64_t dims[3] = {512, 128, (uint64_t)H};
    const uint64_t str[2] = {512 * 2, 128 * 512 * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (mla_status_t s = encode_map(ctx, &tw, w_uk, 3, dims, str, box, "w_uk")) return s;
  }
  p = mla::AbsorbParams{};
  p.H = H;
  p.M = static_cast<int>(M);
  p.rows_box = mla::rows_box_for(M);
  p.q_pos = q_pos;
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.q_abs = static_cast<uint16_t*>(q_abs);
  p.rope = ctx->d_rope;
  p.max_pos = ctx->max_pos;
  p.status = ctx->d_status;
  return MLA_OK;
}

mla_status_t append_absorb_impl(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                                const int32_t* seq_idx, const int32_t* pos, int32_t n, int32_t H, const void* w_uk,
                                const void* q_nope, const void* q_rope, const int32_t* q_pos, int32_t B, int32_t Hq,
                                void* q_abs, void* stream, bool fp8) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  mla::AppendParams a;
  if (mla_status_t st = build_append(ctx, cache, c_kv, k_rope, seq_idx, pos, n, a)) return st;
  DeviceGuard g(ctx->device);
  CUtensorMap tq, tw;
  mla::AbsorbParams p;
  if (mla_status_t st = build_absorb(ctx, H, w_uk, q_nope, q_rope, q_pos, B, Hq, q_abs, tq, tw, p)) return st;
  MLA_CUDA(ctx, mla::launch_append_absorb_q(tq, tw, p, a, fp8, ctx->num_sms, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_append_latent(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                               const int32_t* seq_idx, const int32_t* pos, int32_t n, void* stream) {
  return append_impl(ctx, cache, c_kv, k_rope, seq_idx, pos, n, stream, false);
}

mla_status_t mla_append_latent_fp8(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                                   const int32_t* seq_idx, const int32_t* pos, int32_t n, void* stream) {
  return append_impl(ctx, cache, c_kv, k_rope, seq_idx, pos, n, stream, true);
}

mla_status_t mla_absorb_q(mla_ctx_t* ctx, int32_t H, const void* w_uk, const void* q_nope, const void* q_rope,
                          const int32_t* q_pos, int32_t B, int32_t Hq, void* q_abs, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  CUtensorMap tq, tw;
  mla::AbsorbParams p;
  if (mla_status_t st = build_absorb(ctx, H, w_uk, q_nope, q_rope, q_pos, B, Hq, q_abs, tq, tw, p)) return st;
  MLA_CUDA(ctx, mla::launch_absorb_q(tq, tw, p, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

mla_status_t mla_append_absorb_q(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                                 const int32_t* seq_idx, const int32_t* pos, int32_t n, int32_t H, const void* w_uk,
                                 const void* q_nope, const void* q_rope, const int32_t* q_pos, int32_t B, int32_t Hq,
                                 void* q_abs, void* stream) {
  return append_absorb_impl(ctx, cache, c_kv, k_rope, seq_idx, pos, n, H, w_uk, q_nope, q_rope, q_pos, B, Hq, q_abs,
                            stream, false);
}

mla_status_t mla_append_fp8_absorb_q(mla_ctx_t* ctx, const mla_cache_t* cache, const void* c_kv, const void* k_rope,
                                     const int32_t* seq_idx, const int32_t* pos, int32_t n, int32_t H,
                                     const void* w_uk, const void* q_nope, const void* q_rope, const int32_t* q_pos,
                                     int32_t B, int32_t Hq, void* q_abs, void* stream) {
  return append_absorb_impl(ctx, cache, c_kv, k_rope, seq_idx, pos, n, H, w_uk, q_nope, q_rope, q_pos, B, Hq, q_abs,
                            stream, true);
}

size_t mla_decode_workspace_size(mla_ctx_t* ctx, int32_t H, int32_t B, int32_t Hq) {
  if (!ctx || !heads_ok(H) || B <= 0 || Hq <= 0) return 0;
  int N, C;
  if (!mla::attn_split(Hq * H, N, C) || (N != 16 && N != 32 && N != 64)) return 0;
  const int U = decode_units(ctx, C);
  // one unit: no sequence is ever split, no partial is written
  const size_t rows = U == 1 ? 0 : (size_t)(B + U) * (size_t)(Hq * H);
  return rows * mla::D_C * sizeof(float) + rows * sizeof(float) + 256;
}

}  // extern "C"

namespace {

// Argument and shape checks shared by every decode-attention entry point (the
// workspace is checked by the caller of this helper). Fills the CTA split.
mla_status_t check_decode_args(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* q_abs,
                               const int32_t* seq_lens, int32_t B, int32_t Hq, float scale, const float* o_lat,
                               const float* lse, int& N, int& C) {
  if (mla_status_t s = check_cache(ctx, cache)) return s;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (B <= 0 || Hq <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "B and Hq must be positive");
  if (B > cache->num_seqs) return fail(ctx, MLA_ERR_INVALID_ARG, "B exceeds the cache's num_seqs");
  if (B > mla::MAX_SEQS) return fail(ctx, MLA_ERR_UNSUPPORTED, "B=%d above %d sequences per call", B, mla::MAX_SEQS);
  if (!q_abs || !seq_lens || !o_lat || !lse) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q_abs) || !aligned16(o_lat)) return fail(ctx, MLA_ERR_INVALID_ARG, "q_abs / o_lat must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(ctx, MLA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!mla::attn_split(Hq * H, N, C))
    return fail(ctx, MLA_ERR_UNSUPPORTED, "Hq*H=%d unsupported (16, 32 or 64, then multiples of 64 up to %d)",
                Hq * H, mla::MAX_ROWS_PER_SEQ);
  if (N != 16 && N != 32 && N != 64) return fail(ctx, MLA_ERR_UNSUPPORTED, "Hq*H=%d unsupported", Hq * H);
  if ((long long)B * Hq * H >= (1ll << 31)) return fail(ctx, MLA_ERR_UNSUPPORTED, "B*Hq*H too large");
  return MLA_OK;
}

mla_status_t decode_impl(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* q_abs,
                         const int32_t* seq_lens, int32_t B, int32_t Hq, float scale, void* workspace,
                         size_t ws_bytes, float* o_lat, float* lse, void* stream, bool fp8) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  int N, C;
  if (mla_status_t s = check_decode_args(ctx, H, cache, q_abs, seq_lens, B, Hq, scale, o_lat, lse, N, C)) return s;
  const size_t need = mla_decode_workspace_size(ctx, H, B, Hq);
  if (!workspace || ws_bytes < need)
    return fail(ctx, MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  if (!aligned16(workspace)) return fail(ctx, MLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  DeviceGuard g(ctx->device);
  const int G = Hq * H;
  // 128-row groups of a bf16 cache run on CTA pairs (the 2-SM tensor-core path)
  const bool pair = !fp8 && N == 64 && C % 2 == 0;
  if (pair) {
    if (!ctx->pair_ready) {
      MLA_CUDA(ctx, mla::attn_pair_prepare(&ctx->attn_pairs));
      ctx->pair_ready = true;
    }
  } else {
    bool& ready = fp8 ? ctx->attn8_ready[N] : ctx->attn_ready[N];
    if (!ready) {
      MLA_CUDA(ctx, fp8 ? mla::attn8_prepare(N) : mla::attn_prepare(N));
      ready = true;
    }
  }
  const int U = pair ? pair_units(ctx, C) : decode_units(ctx, C);
  const uint64_t cache_rows = cache->paged ? (uint64_t)cache->num_blocks * mla::PAGE
                                           : (uint64_t)cache->num_seqs * cache->capacity;
  CUtensorMap tc, tq, tsc;
  if (fp8) {
    const uint64_t dims[2] = {(uint64_t)mla::ROW8, cache_rows};
    const uint64_t str[1] = {(uint64_t)mla::ROW8};
    const uint32_t box[2] = {128, 64};
    if (mla_status_t s = encode_map(ctx, &tc, cache->base, 2, dims, str, box, "fp8 cache", CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return s;
    const uint32_t sbox[2] = {16, 64};
    if (mla_status_t s = encode_map(ctx, &tsc, cache->base, 2, dims, str, sbox, "fp8 cache scales",
                                    CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE))
      return s;
  } else {
    const uint64_t dims[2] = {(uint64_t)mla::ROW, cache_rows};
    const uint64_t str[1] = {(uint64_t)mla::ROW * 2};
    const uint32_t box[2] = {64, 64};
    if (mla_status_t s = encode_map(ctx, &tc, cache->base, 2, dims, str, box, "cache")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)mla::ROW, (uint64_t)B * G};
    const uint64_t str[1] = {(uint64_t)mla::ROW * 2};
    const uint32_t box[2] = {64, (uint32_t)N};
    if (mla_status_t s = encode_map(ctx, &tq, q_abs, 2, dims, str, box, "q_abs")) return s;
  }
  mla::AttnParams p{};
  p.B = B;
  p.H = H;
  p.Hq = Hq;
  p.G = G;
  p.N = N;
  p.C = C;
  p.U = U;
  // one unit with more row-group pairs than fit at once: launch the pairs that
  // fit, each walking several row-group pairs
  p.slots = (pair && U == 1 && C / 2 > ctx->attn_pairs) ? ctx->attn_pairs : 0;
  p.paged = cache->paged;
  p.capacity = cache->capacity;
  p.num_seqs = cache->num_seqs;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = cache->max_blocks;
  p.block_table = cache->block_table;
  p.seq_lens = seq_lens;
  p.cache = static_cast<const uint8_t*>(cache->base);
  p.q_abs = static_cast<const uint16_t*>(q_abs);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_lat = o_lat;
  p.lse = lse;
  const size_t rows = U == 1 ? 0 : (size_t)(B + U) * G;   // as mla_decode_workspace_size
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = p.ws_o + rows * mla::D_C;
  p.status = ctx->d_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, fp8    ? mla::launch_decode_attn_fp8(tc, tsc, tq, p, s)
                : pair ? mla::launch_decode_attn_pair(tc, tq, p, s)
                       : mla::launch_decode_attn(tc, tq, p, s));
  MLA_CUDA(ctx, mla::launch_combine(p, s));
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_attn(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* q_abs,
                             const int32_t* seq_lens, int32_t B, int32_t Hq, float scale, void* workspace,
                             size_t ws_bytes, float* o_lat, float* lse, void* stream) {
  return decode_impl(ctx, H, cache, q_abs, seq_lens, B, Hq, scale, workspace, ws_bytes, o_lat, lse, stream, false);
}

mla_status_t mla_decode_attn_fp8(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* q_abs,
                                 const int32_t* seq_lens, int32_t B, int32_t Hq, float scale, void* workspace,
                                 size_t ws_bytes, float* o_lat, float* lse, void* stream) {
  return decode_impl(ctx, H, cache, q_abs, seq_lens, B, Hq, scale, workspace, ws_bytes, o_lat, lse, stream, true);
}

size_t mla_small_step_max_len(void) { return mla::SMALL_MAX_LEN; }

mla_status_t mla_decode_step_small(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* c_kv,
                                   const void* k_rope, const void* w_uk, const void* w_uv, const void* q_nope,
                                   const void* q_rope, const int32_t* seq_lens, int32_t B, float scale, void* out,
                                   float* o_lat, float* lse, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (mla_status_t s = check_cache(ctx, cache)) return s;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (B <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "B must be positive");
  if (B > cache->num_seqs) return fail(ctx, MLA_ERR_INVALID_ARG, "B exceeds the cache's num_seqs");
  if (B > 65535) return fail(ctx, MLA_ERR_UNSUPPORTED, "B=%d above 65535 sequences per call", B);
  if (!c_kv || !k_rope || !w_uk || !w_uv || !q_nope || !q_rope || !seq_lens || !out || !o_lat || !lse)
    return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(c_kv) || !aligned16(k_rope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(q_nope) ||
      !aligned16(q_rope) || !aligned16(out) || !aligned16(o_lat))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(ctx, MLA_ERR_INVALID_ARG, "scale must be finite and > 0");
  DeviceGuard g(ctx->device);
  mla::SmallStepParams p{};
  p.a.cache = static_cast<uint16_t*>(cache->base);
  p.a.paged = cache->paged;
  p.a.num_seqs = cache->num_seqs;
  p.a.capacity = cache->capacity;
  p.a.num_blocks = cache->num_blocks;
  p.a.max_blocks = cache->max_blocks;
  p.a.block_table = cache->block_table;
  p.a.c_kv = static_cast<const uint16_t*>(c_kv);
  p.a.k_rope = static_cast<const uint16_t*>(k_rope);
  p.a.n = B;
  p.a.rope = ctx->d_rope;
  p.a.max_pos = ctx->max_pos;
  p.a.status = ctx->d_status;
  p.w_uk = static_cast<const uint16_t*>(w_uk);
  p.w_uv = static_cast<const uint16_t*>(w_uv);
  p.q_nope = static_cast<const uint16_t*>(q_nope);
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.seq_lens = seq_lens;
  p.H = H;
  p.scale = scale;
  p.out = static_cast<uint16_t*>(out);
  p.o_lat = o_lat;
  p.lse = lse;
  MLA_CUDA(ctx, mla::launch_small_step(p, B, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

mla_status_t mla_expand_v(mla_ctx_t* ctx, int32_t H, const void* w_uv, const float* o_lat, int32_t B, int32_t Hq,
                          void* out, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (B <= 0 || Hq <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "B and Hq must be positive");
  if (!w_uv || !o_lat || !out) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_uv) || !aligned16(o_lat) || !aligned16(out))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const long long M = (long long)B * Hq;
  if (M * H >= (1ll << 31)) return fail(ctx, MLA_ERR_UNSUPPORTED, "B*Hq*H too large");
  DeviceGuard g(ctx->device);
  CUtensorMap tw, to;
  {
    const uint64_t dims[3] = {512, 128, (uint64_t)H};
    const uint64_t str[2] = {512 * 2, 128 * 512 * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (mla_status_t s = encode_map(ctx, &tw, w_uv, 3, dims, str, box, "w_uv")) return s;
  }
  {
    const uint64_t dims[3] = {512, (uint64_t)H, (uint64_t)M};
    const uint64_t str[2] = {512 * 4, (uint64_t)H * 512 * 4};
    const uint32_t box[3] = {32, 1, (uint32_t)mla::rows_box_for(M)};
    if (mla_status_t s = encode_map(ctx, &to, o_lat, 3, dims, str, box, "o_lat", CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return s;
  }
  mla::ExpandParams p{};
  p.H = H;
  p.M = static_cast<int>(M);
  p.rows_box = mla::rows_box_for(M);
  p.o_lat = o_lat;
  p.out = static_cast<uint16_t*>(out);
  p.status = ctx->d_status;
  MLA_CUDA(ctx, mla::launch_expand_v(tw, to, p, ctx->num_sms, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

mla_status_t mla_out_proj(mla_ctx_t* ctx, int32_t H, const void* w_o, int32_t d_model, const void* o, int32_t M,
                          float* y, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (M <= 0 || d_model <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "M and d_model must be positive");
  if (d_model % 128) return fail(ctx, MLA_ERR_UNSUPPORTED, "d_model=%d is not a multiple of 128", d_model);
  if (!w_o || !o || !y) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_o) || !aligned16(o) || !aligned16(y))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((long long)M * d_model >= (1ll << 31)) return fail(ctx, MLA_ERR_UNSUPPORTED, "M*d_model too large");
  DeviceGuard g(ctx->device);
  const int K = H * mla::D_V;
  const int nb = mla::out_proj_nb(M);
  const int rows_box = M >= nb ? nb : ((M + 7) / 8) * 8;
  CUtensorMap tw, tx;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)d_model};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tw, w_o, 2, dims, str, box, "w_o")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, (uint32_t)rows_box};
    if (mla_status_t s = encode_map(ctx, &tx, o, 2, dims, str, box, "o")) return s;
  }
  mla::OutProjParams p{};
  p.d_model = d_model;
  p.M = M;
  p.KB = K / 64;
  p.rows_box = rows_box;
  p.y = y;
  p.sync = ctx->d_op_sync;
  p.status = ctx->d_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, mla::launch_out_proj(tw, tx, p, ctx->num_sms, s));
  return MLA_OK;
}

mla_status_t mla_absorb_w_o(mla_ctx_t* ctx, int32_t H, const void* w_o, int32_t d_model, const void* w_uv,
                            void* w_ov, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (d_model <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "d_model must be positive");
  if (d_model % 128) return fail(ctx, MLA_ERR_UNSUPPORTED, "d_model=%d is not a multiple of 128", d_model);
  if (!w_o || !w_uv || !w_ov) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_o) || !aligned16(w_uv) || !aligned16(w_ov))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  DeviceGuard g(ctx->device);
  MLA_CUDA(ctx, mla::launch_absorb_w_o(static_cast<const uint16_t*>(w_o), static_cast<const uint16_t*>(w_uv),
                                      static_cast<uint16_t*>(w_ov), H, d_model, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

mla_status_t mla_out_proj_latent(mla_ctx_t* ctx, int32_t H, const void* w_ov, int32_t d_model, const float* o_lat,
                                 int32_t M, float* y, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (M <= 0 || d_model <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "M and d_model must be positive");
  if (d_model % 128) return fail(ctx, MLA_ERR_UNSUPPORTED, "d_model=%d is not a multiple of 128", d_model);
  if (!w_ov || !o_lat || !y) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_ov) || !aligned16(o_lat) || !aligned16(y))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if ((long long)M * d_model >= (1ll << 31) || (long long)M * H * mla::D_C >= (1ll << 31))
    return fail(ctx, MLA_ERR_UNSUPPORTED, "M*d_model or M*H*512 too large");
  DeviceGuard g(ctx->device);
  const int K = H * mla::D_C;
  const int nb = mla::out_proj_nb(M);
  const int rows_box = M >= nb ? nb : ((M + 7) / 8) * 8;
  CUtensorMap tw, tx;
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)d_model};
    const uint64_t str[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tw, w_ov, 2, dims, str, box, "w_ov")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t str[1] = {(uint64_t)K * 4};
    const uint32_t box[2] = {32, (uint32_t)rows_box};
    if (mla_status_t s = encode_map(ctx, &tx, o_lat, 2, dims, str, box, "o_lat", CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
      return s;
  }
  mla::OutProjParams p{};
  p.d_model = d_model;
  p.M = M;
  p.KB = K / 64;
  p.rows_box = rows_box;
  p.y = y;
  p.status = ctx->d_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, cudaMemsetAsync(y, 0, (size_t)M * d_model * sizeof(float), s));
  MLA_CUDA(ctx, mla::launch_out_proj_latent(tw, tx, p, ctx->num_sms, s));
  return MLA_OK;
}

size_t mla_project_latent_workspace_size(int32_t n) {
  if (n <= 0) return 0;
  // the partial slots of the one-launch producer: at most LP_MAX_SPLITS per
  // token block, shared out among the blocks
  const int nb = mla::out_proj_nb(n);
  const int mblocks = (n + nb - 1) / nb;
  const int slots = mla::LP_MAX_SPLITS / mblocks > 1 ? mla::LP_MAX_SPLITS / mblocks : 1;
  return (size_t)slots * n * mla::ROW * sizeof(float);
}

mla_status_t mla_project_latent(mla_ctx_t* ctx, const mla_cache_t* cache, const void* w_kv_a, int32_t d_model,
                                const void* kv_norm, float eps, const void* h, const int32_t* seq_idx,
                                const int32_t* pos, int32_t n, void* workspace, size_t ws_bytes, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (mla_status_t s = check_cache(ctx, cache)) return s;
  if (n <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "n must be positive");
  if (d_model <= 0 || d_model % 64) return fail(ctx, MLA_ERR_UNSUPPORTED, "d_model=%d is not a multiple of 64", d_model);
  if (!w_kv_a || !h || !seq_idx || !pos || !workspace) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_kv_a) || !aligned16(h) || !aligned16(workspace) || (kv_norm && !aligned16(kv_norm)))
    return fail(ctx, MLA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (ws_bytes < mla_project_latent_workspace_size(n))
    return fail(ctx, MLA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", ws_bytes,
                mla_project_latent_workspace_size(n));
  if (!(eps >= 0.f)) return fail(ctx, MLA_ERR_INVALID_ARG, "eps must be non-negative");
  DeviceGuard g(ctx->device);
  const int nb = mla::out_proj_nb(n);
  const int rows_box = n >= nb ? nb : ((n + 7) / 8) * 8;
  CUtensorMap tw, tx;
  {
    const uint64_t dims[2] = {(uint64_t)d_model, (uint64_t)mla::ROW};
    const uint64_t str[1] = {(uint64_t)d_model * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tw, w_kv_a, 2, dims, str, box, "w_kv_a")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)d_model, (uint64_t)n};
    const uint64_t str[1] = {(uint64_t)d_model * 2};
    const uint32_t box[2] = {64, (uint32_t)rows_box};
    if (mla_status_t s = encode_map(ctx, &tx, h, 2, dims, str, box, "h")) return s;
  }
  float* y = static_cast<float*>(workspace);
  const int S = mla::latent_proj_splits(n, d_model / 64, ctx->num_sms);
  if (S > 0) {
    // one cooperative launch: split-K partials, grid barrier, per-token finish
    mla::LatentProjParams lp{};
    lp.fin.a.cache = static_cast<uint16_t*>(cache->base);
    lp.fin.a.paged = cache->paged;
    lp.fin.a.num_seqs = cache->num_seqs;
    lp.fin.a.capacity = cache->capacity;
    lp.fin.a.num_blocks = cache->num_blocks;
    lp.fin.a.max_blocks = cache->max_blocks;
    lp.fin.a.block_table = cache->block_table;
    lp.fin.a.seq_idx = seq_idx;
    lp.fin.a.pos = pos;
    lp.fin.a.n = n;
    lp.fin.a.rope = ctx->d_rope;
    lp.fin.a.max_pos = ctx->max_pos;
    lp.fin.a.status = ctx->d_status;
    lp.fin.y = y;
    lp.fin.kv_norm = static_cast<const uint16_t*>(kv_norm);
    lp.fin.eps = eps;
    lp.ws = y;
    lp.KB = d_model / 64;
    lp.S = S;
    lp.rows_box = rows_box;
    lp.sync = ctx->d_sync;
    MLA_CUDA(ctx, mla::launch_latent_proj(tw, tx, lp, static_cast<cudaStream_t>(stream)));
    return MLA_OK;
  }
  // more token blocks than fit on the GPU at once: split-K GEMM (the first
  // split stores, the others add in L2), then the per-token finish
  mla::OutProjParams gp{};
  gp.d_model = mla::ROW;
  gp.M = n;
  gp.KB = d_model / 64;
  gp.rows_box = rows_box;
  gp.y = y;
  gp.sync = ctx->d_op_sync;
  gp.status = ctx->d_status;
  mla::LatentFinishParams q{};
  q.a.cache = static_cast<uint16_t*>(cache->base);
  q.a.paged = cache->paged;
  q.a.num_seqs = cache->num_seqs;
  q.a.capacity = cache->capacity;
  q.a.num_blocks = cache->num_blocks;
  q.a.max_blocks = cache->max_blocks;
  q.a.block_table = cache->block_table;
  q.a.seq_idx = seq_idx;
  q.a.pos = pos;
  q.a.n = n;
  q.a.rope = ctx->d_rope;
  q.a.max_pos = ctx->max_pos;
  q.a.status = ctx->d_status;
  q.y = y;
  q.kv_norm = static_cast<const uint16_t*>(kv_norm);
  q.eps = eps;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, mla::launch_out_proj(tw, tx, gp, ctx->num_sms, s));
  MLA_CUDA(ctx, mla::launch_latent_finish(q, s));
  return MLA_OK;
}

// MHA-form prefill: workspace = the expanded keys and values of every
// sequence (max_len rounded up to 128 rows each), then the rotated queries.
static size_t prefill_mha_kv_bytes(int32_t H, int32_t B, int32_t max_len) {
  const size_t ml = ((size_t)max_len + 127) / 128 * 128;
  return ((size_t)B * ml * 2 * H * 128 * 2 + 255) / 256 * 256;
}

size_t mla_prefill_mha_workspace_size(int32_t H, int32_t B, int32_t T, int32_t max_len) {
  if (H <= 0 || B <= 0 || T <= 0 || max_len <= 0) return 0;
  return prefill_mha_kv_bytes(H, B, max_len) + ((size_t)B * T * H * mla::D_ROPE * 2 + 255) / 256 * 256;
}

mla_status_t mla_prefill_mha(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache, const void* w_uk, const void* w_uv,
                             const void* q_nope, const void* q_rope, const int32_t* q_pos, const int32_t* seq_lens,
                             int32_t B, int32_t T, int32_t max_len, float scale, void* workspace, size_t ws_bytes,
                             void* out, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return fail(ctx, MLA_ERR_UNSUPPORTED, "H=%d unsupported (16, 32, 64, 128)", H);
  if (mla_status_t s = check_cache(ctx, cache)) return s;
  if (B <= 0 || T <= 0) return fail(ctx, MLA_ERR_INVALID_ARG, "B and T must be positive");
  if (max_len < T) return fail(ctx, MLA_ERR_INVALID_ARG, "max_len (%d) must be at least T (%d)", max_len, T);
  if (B > cache->num_seqs) return fail(ctx, MLA_ERR_INVALID_ARG, "B=%d exceeds the cache's %d sequences", B,
                                       cache->num_seqs);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(ctx, MLA_ERR_INVALID_ARG, "scale must be positive");
  if (!w_uk || !w_uv || !q_nope || !q_rope || !q_pos || !seq_lens || !workspace || !out)
    return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(w_uk) || !aligned16(w_uv) || !aligned16(q_nope) || !aligned16(q_rope) || !aligned16(out) ||
      !aligned16(workspace))
    return fail(ctx, MLA_ERR_INVALID_ARG, "bf16 tensors and the workspace must be 16-byte aligned");
  const long long ml = ((long long)max_len + 127) / 128 * 128;
  if ((long long)B * ml >= (1ll << 31) || (long long)B * T * H >= (1ll << 31))
    return fail(ctx, MLA_ERR_UNSUPPORTED, "B*max_len or B*T*H too large");
  const size_t need = mla_prefill_mha_workspace_size(H, B, T, max_len);
  if (ws_bytes < need) return fail(ctx, MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  DeviceGuard g(ctx->device);
  uint16_t* kv = static_cast<uint16_t*>(workspace);
  uint16_t* q_rot = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + prefill_mha_kv_bytes(H, B, max_len));
  const uint64_t cache_rows = cache->paged ? (uint64_t)cache->num_blocks * mla::PAGE
                                           : (uint64_t)cache->num_seqs * cache->capacity;
  CUtensorMap tc, twk, twv, tqn, tqr, tkv;
  {
    const uint64_t dims[2] = {(uint64_t)mla::ROW, cache_rows};
    const uint64_t str[1] = {(uint64_t)mla::ROW * 2};
    const uint32_t box[2] = {64, 64};
    if (mla_status_t s = encode_map(ctx, &tc, cache->base, 2, dims, str, box, "cache")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)mla::D_C, (uint64_t)H * 128};
    const uint64_t str[1] = {(uint64_t)mla::D_C * 2};
    const uint32_t box[2] = {64, 256};
    if (mla_status_t s = encode_map(ctx, &twk, w_uk, 2, dims, str, box, "w_uk")) return s;
    if (mla_status_t s = encode_map(ctx, &twv, w_uv, 2, dims, str, box, "w_uv")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)H * mla::D_NOPE, (uint64_t)B * T};
    const uint64_t str[1] = {(uint64_t)H * mla::D_NOPE * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tqn, q_nope, 2, dims, str, box, "q_nope")) return s;
  }
  {
    const uint64_t dims[2] = {(uint64_t)H * mla::D_ROPE, (uint64_t)B * T};
    const uint64_t str[1] = {(uint64_t)H * mla::D_ROPE * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tqr, q_rot, 2, dims, str, box, "q_rot")) return s;
  }
  {
    // kv: the attention's loads and the expansion's stores, 64 x 128 boxes
    const uint64_t dims[2] = {(uint64_t)2 * H * 128, (uint64_t)B * ml};
    const uint64_t str[1] = {(uint64_t)2 * H * 128 * 2};
    const uint32_t box[2] = {64, 128};
    if (mla_status_t s = encode_map(ctx, &tkv, kv, 2, dims, str, box, "kv")) return s;
  }
  mla::PrefillMhaParams p{};
  p.B = B;
  p.H = H;
  p.T = T;
  p.max_len = max_len;
  p.ML = static_cast<int>(ml);
  p.paged = cache->paged;
  p.capacity = cache->capacity;
  p.num_seqs = cache->num_seqs;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = cache->max_blocks;
  p.block_table = cache->block_table;
  p.seq_lens = seq_lens;
  p.q_pos = q_pos;
  p.q_rope = static_cast<const uint16_t*>(q_rope);
  p.q_rot = q_rot;
  p.kv = kv;
  p.out = static_cast<uint16_t*>(out);
  p.rope = ctx->d_rope;
  p.max_pos = ctx->max_pos;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.num_ctas = ctx->num_sms;
  p.status = ctx->d_status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  MLA_CUDA(ctx, mla::launch_expand_kv(tc, twk, twv, tkv, p, s));
  MLA_CUDA(ctx, mla::launch_prefill_mha(tqn, tqr, tkv, tc, p, s));
  return MLA_OK;
}

// Step-time estimates of the two prefill forms (µs, the chunk's append
// included), fitted to steps measured on one GB300 (152 SMs, 2.07 GHz) over
// chunks of 16-1,024 tokens, H = 16 and 128, fresh prompts and 4,096-token
// prefixes. Absorbed form: the longer of two bounds, each with the
// per-query-row work of absorb_q, the fp32 o_lat round trip and expand_v: the
// attention's (query, key, head) triples at its measured rate, and its
// critical path, the key pages one split-KV unit walks (a sequence's Hq*H rows
// make C 64-row CTAs, floor(SMs / C) units share the batch's keys, and rows
// beyond one CTA per SM run in waves), which jumps where C passes 76 or 152.
// MHA form: a fixed part, the expansion's
// 128-token x 1-head tiles, the attention's critical path in key tiles per CTA
// (its items are (sequence, head, 128-query tile) and run persistently over the
// SMs) and its per-item cost; below ~30 µs its two launches and the append set
// the time.
namespace {
struct PrefillEstimate {
  double absorbed_us, mha_us;
};

PrefillEstimate estimate_prefill(int32_t H, int32_t B, int32_t T, const int32_t* seq_lens) {
  const double sms = 152.0;
  double triples = 0, pages = 0, exp_tiles = 0, key_tile_steps = 0, items = 0, longest = 0;
  for (int32_t b = 0; b < B; ++b) {
    const double L = seq_lens[b], prefix = L - T;
    triples += (double)H * ((double)T * (prefix + 1) + (double)T * (T - 1) / 2);
    pages += std::ceil(L / 64.0);
    exp_tiles += (double)H * std::ceil(L / 128.0);
    for (int32_t q0 = 0; q0 < T; q0 += 128) {
      const double last = prefix + std::min(T, q0 + 128) - 1;   // last key the query tile sees
      const double tiles = std::ceil((last + 1) / 128.0);
      key_tile_steps += (double)H * tiles;
      items += H;
      longest = std::max(longest, tiles);
    }
  }
  PrefillEstimate e;
  const double rows = (double)H * B * T;
  const double ctas = std::max(1.0, (double)T * H / 64.0);           // 64-row CTAs per sequence
  const double units = std::max(1.0, std::floor(sms / ctas));        // split-KV units
  const double crit = pages / units * std::max(1.0, ctas / sms);     // key pages per unit, in waves
  e.absorbed_us = std::max(22.5 + 3.18e-6 * triples + 2.24e-3 * rows, 25.5 + 1.796 * crit + 1.628e-3 * rows);
  e.mha_us = std::max(30.0, 20.7 + 32.7e-3 * exp_tiles + 0.956 * std::max(key_tile_steps / sms, longest) +
                                3.04 * items / sms);
  return e;
}
}  // namespace

mla_status_t mla_prefill_choose_form(int32_t H, int32_t B, int32_t T, const int32_t* seq_lens, int32_t fp8_cache,
                                     size_t ws_limit, int32_t* form, double* est_us) {
  if (!seq_lens || !form || B <= 0 || T <= 0) return MLA_ERR_INVALID_ARG;
  if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
  int32_t max_len = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (seq_lens[b] < T) return MLA_ERR_INVALID_ARG;
    max_len = std::max(max_len, seq_lens[b]);
  }
  // what each form accepts (the limits mla_decode_attn and mla_prefill_mha check)
  int N = 0, C = 0;
  const bool absorbed_ok = B <= mla::MAX_SEQS && (long long)T * H <= mla::MAX_ROWS_PER_SEQ &&
                           mla::attn_split(T * H, N, C) && (long long)B * T * H < (1ll << 31);
  const long long ml = ((long long)max_len + 127) / 128 * 128;
  bool mha_ok = !fp8_cache && (long long)B * ml < (1ll << 31) && (long long)B * T * H < (1ll << 31);
  if (mha_ok && ws_limit) mha_ok = mla_prefill_mha_workspace_size(H, B, T, max_len) <= ws_limit;
  if (!absorbed_ok && !mha_ok) return MLA_ERR_UNSUPPORTED;
  const PrefillEstimate e = estimate_prefill(H, B, T, seq_lens);
  if (est_us) {
    est_us[0] = e.absorbed_us;
    est_us[1] = e.mha_us;
  }
  *form = !absorbed_ok ? MLA_PREFILL_MHA : !mha_ok ? MLA_PREFILL_ABSORBED
                                         : (e.mha_us < e.absorbed_us ? MLA_PREFILL_MHA : MLA_PREFILL_ABSORBED);
  return MLA_OK;
}

mla_status_t mla_get_device_status(mla_ctx_t* ctx, void* stream, int32_t* status_out) {
  if (!ctx || !status_out) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  MLA_CUDA(ctx, cudaStreamSynchronize(s));
  MLA_CUDA(ctx, cudaMemcpy(&v, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost));
  MLA_CUDA(ctx, cudaMemset(ctx->d_status, 0, sizeof(int)));
  // a grid barrier or split-K wait that gave up leaves its words behind: start
  // them afresh (the stream is idle, so no wait is in flight on it)
  if (v & MLA_DEVICE_TIMEOUT) {
    MLA_CUDA(ctx, cudaMemset(ctx->d_sync, 0, mla::LP_SYNC_WORDS * sizeof(unsigned)));
    MLA_CUDA(ctx, cudaMemset(ctx->d_op_sync, 0, 3 * mla::OP_SYNC_TILES * sizeof(unsigned)));
  }
  *status_out = v;
  return MLA_OK;
}

mla_status_t mla_copy_async(mla_ctx_t* ctx, void* dst, const void* src, size_t bytes, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (bytes == 0) return MLA_OK;
  if (!dst || !src) return fail(ctx, MLA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(dst) || !aligned16(src) || bytes % 16)
    return fail(ctx, MLA_ERR_INVALID_ARG, "dst and src must be 16-byte aligned and bytes a multiple of 16");
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), sr = reinterpret_cast<uintptr_t>(src);
  if (d < sr + bytes && sr < d + bytes) return fail(ctx, MLA_ERR_INVALID_ARG, "dst and src overlap");
  DeviceGuard g(ctx->device);
  MLA_CUDA(ctx, mla::launch_copy(dst, src, bytes, ctx->num_sms, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

mla_status_t mla_debug_wait_timeout(mla_ctx_t* ctx, uint64_t limit_ns, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  if (limit_ns > 5000000000ull) return fail(ctx, MLA_ERR_INVALID_ARG, "limit_ns above 5 s");
  DeviceGuard g(ctx->device);
  MLA_CUDA(ctx, mla::launch_wait_probe(ctx->d_status, limit_ns, static_cast<cudaStream_t>(stream)));
  return MLA_OK;
}

}  // extern "C"


// ---------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory: the
// split-KV partials go to g_decode_scratch (its device address was looked up
// by mla_create) instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
extern "C" size_t mla_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" mla_status_t mla_decode_attn_static_scratch(mla_ctx_t* ctx, int32_t H, const mla_cache_t* cache,
                                                       const void* q_abs, const int32_t* seq_lens, int32_t B,
                                                       int32_t Hq, float scale, float* o_lat, float* lse,
                                                       void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  int N, C;
  // the same checks, status codes and messages as mla_decode_attn first
  if (mla_status_t s = check_decode_args(ctx, H, cache, q_abs, seq_lens, B, Hq, scale, o_lat, lse, N, C)) return s;
  const size_t need = mla_decode_workspace_size(ctx, H, B, Hq);
  if (need > kStaticScratchBytes)
    return fail(ctx, MLA_ERR_UNSUPPORTED,
                "H=%d B=%d Hq=%d needs %zu bytes of split-KV scratch but the static scratch holds %zu; "
                "use mla_decode_attn with a caller-provided workspace",
                H, B, Hq, need, kStaticScratchBytes);
  // Every partial the combine reads is written earlier in the same call, so
  // nothing in the scratch has to start at zero.
  return mla_decode_attn(ctx, H, cache, q_abs, seq_lens, B, Hq, scale, ctx->static_scratch, kStaticScratchBytes,
                         o_lat, lse, stream);
}
