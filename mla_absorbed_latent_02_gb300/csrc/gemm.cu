// Per-head projections of absorbed MLA on the 5th-generation tensor cores.
//
// absorb_q: key absorption, q_lat[r,h,:] = W_UK[h]^T q_nope[r,h,:] (512 <- 128),
//   because q^T (W_UK c) = (W_UK^T q)^T c ("DeepSeek MLA 吸收式缓存" §2.2;
//   "80 行 PyTorch 从零写 DeepSeek 的 MLA" §4, path B). The same kernel rotates
//   q_rope at the query position and writes the 576-wide absorbed query
//   q_abs = [q_lat | RoPE(q_rope)] (decoupled RoPE, "DeepSeek MLA 吸收式缓存" §2.4).
// expand_v: value absorption applied after aggregation, o[r,h,:] = W_UV[h] o_lat[r,h,:]
//   (128 <- 512) ("DeepSeek MLA 吸收式缓存" §2.3).
//
// Both are batched GEMMs with one weight matrix per head: M = B*Hq query rows,
// D in TMEM (fp32), operands staged in shared memory by TMA (128-byte swizzle).
#include "append_body.cuh"
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase trace (compile with -DMLA_TRACE=1): globaltimer stamps of the
// first CTAs of absorb_q (kernel 0) and expand_v (kernel 1), read back with
// mla_trace_read_gemm(). Off in normal builds.
#ifndef MLA_TRACE
#define MLA_TRACE 0
#endif
#if MLA_TRACE
__device__ unsigned long long g_mla_trace_gemm[2][64][8];
#define GTRACE(k, ev)                                                             \
  do {                                                                           \
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z); \
    if (cta < 64) g_mla_trace_gemm[(k)][cta][(ev)] = globaltimer();               \
  } while (0)
extern "C" int mla_trace_read_gemm(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace_gemm)) bytes = sizeof(g_mla_trace_gemm);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace_gemm, bytes);
}
#else
#define GTRACE(k, ev) \
  do {                \
  } while (0)
#endif

namespace mla {

namespace {

constexpr int ABS_NT = 128;            // output columns per CTA (absorb_q)
constexpr uint32_t KB_BYTES = 16384;   // 128 rows x 128 B

struct __align__(8) GemmBarriers {
  uint64_t full;
  uint64_t done;
  uint64_t stage_done[2];
  uint32_t tmem_base;
  int abort;
};

MLA_DEV uint8_t* align1k(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace

// One CTA of absorb_q: head h, output columns nb*ABS_NT .. +ABS_NT, query rows
// mb*128 .. +127; 160 threads: warps 0-3 own one query row each (RoPE,
// epilogue), warp 4 owns TMEM and one thread of it issues the TMA loads and the
// MMAs. A = q_nope rows of head h (K-major, 2 K-blocks of 64), B =
// W_UK[h][:, n0:n0+ABS_NT] (N-contiguous, MN-major, atoms of 64 columns x 128 K-rows).
MLA_DEV void absorb_q_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_w, const AbsorbParams& p, int h, int nb,
                          int mb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sa = smem;                       // 2 x 16 KB
  uint8_t* sb = smem + 2 * KB_BYTES;        // ABS_NT/64 x 16 KB
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(smem + (2 + ABS_NT / 64) * KB_BYTES);

  const int n0 = nb * ABS_NT;
  const int m0 = mb * 128;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) GTRACE(0, 0);

  const bool issuer = threadIdx.x == 128;
  if (issuer) {
    mbar_init(smem_u32(&bars->full), 1);
    mbar_init(smem_u32(&bars->done), 1);
    bars->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&bars->tmem_base), ABS_NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  pdl_trigger();
  // q_nope, W_UK, q_rope and q_pos are call inputs that no kernel of this library
  // writes: they are loaded (and the MMA runs) while the previous kernel of the
  // stream may still be running; only the writes of q_abs wait for it.
  if (threadIdx.x == 0) GTRACE(0, 1);

  if (issuer) {
    const uint32_t full = smem_u32(&bars->full);
    mbar_arrive_expect_tx(full, 2 * 128 * p.rows_box + (ABS_NT / 64) * KB_BYTES);
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(smem_u32(sa + kb * KB_BYTES), &tm_q, full, 64 * kb, h, m0);
    for (int a = 0; a < ABS_NT / 64; ++a) tma_load_3d(smem_u32(sb + a * KB_BYTES), &tm_w, full, n0 + 64 * a, 0, h);
    if (mbar_wait(full, 0, &bars->abort, p.status)) {
      GTRACE(0, 2);
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(128, ABS_NT, 0, 1);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t ad = smem_desc(smem_u32(sa + (k >> 2) * KB_BYTES) + (k & 3) * 32, 16, 1024, SMEM_SWIZZLE_128B);
        const uint64_t bd = smem_desc(smem_u32(sb) + k * 2048, KB_BYTES, 1024, SMEM_SWIZZLE_128B);
        mma_bf16_ss(tmem, ad, bd, idesc, k > 0);
      }
      mma_commit(smem_u32(&bars->done));
    }
  }

  // RoPE of the query's rope part (one thread per row): its loads (position,
  // then that position's cos/sin row) are issued before the epilogue waits for
  // the MMA, the rotation runs after the epilogue's stores.
  const int r = m0 + threadIdx.x;
  const bool rope_row = warp < 4 && nb == 0 && r < p.M;
  uint4 qr[8];
  float2 cs[32];
  bool rope_ok = false;
  if (rope_row) {
    const int pos = p.q_pos[r];
    const uint4* src = reinterpret_cast<const uint4*>(p.q_rope + ((long long)r * p.H + h) * D_ROPE);
#pragma unroll
    for (int c = 0; c < 8; ++c) qr[c] = src[c];
    rope_ok = pos >= 0 && pos < p.max_pos;
    if (!rope_ok) {
      atomicOr(p.status, MLA_DEVERR_BOUNDS);
    } else {
      const float4* tab = reinterpret_cast<const float4*>(p.rope + (long long)pos * (D_ROPE / 2));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 v = tab[i];
        cs[2 * i] = make_float2(v.x, v.y);
        cs[2 * i + 1] = make_float2(v.z, v.w);
      }
    }
  }

  if (threadIdx.x == 0) GTRACE(0, 3);
  __syncwarp();
  pdl_wait();
  const bool ok = warp < 4 && mbar_wait(smem_u32(&bars->done), 0, &bars->abort, p.status);
  if (threadIdx.x == 0) GTRACE(0, 4);
  tc_fence_after();
  if (ok) {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint16_t* dst = p.q_abs + ((long long)r * p.H + h) * ROW + n0;
#pragma unroll 1
    for (int c0 = 0; c0 < ABS_NT; c0 += 64) {
      uint32_t v[64];
#pragma unroll
      for (int c = 0; c < 64; c += 16) tmem_ld16(tmem + lane_base + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 64; c += 16) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + c));
      if (r < p.M) {
        uint4* d = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
        for (int c = 0; c < 64; c += 8)
          d[c / 8] = make_uint4(pack_bf16x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                pack_bf16x2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])),
                                pack_bf16x2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5])),
                                pack_bf16x2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7])));
      }
    }
  }
  if (rope_ok) {
    uint4* dst = reinterpret_cast<uint4*>(p.q_abs + ((long long)r * p.H + h) * ROW + D_C);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t in[4] = {qr[c].x, qr[c].y, qr[c].z, qr[c].w};
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = __uint_as_float(in[i] << 16);
        const float b = __uint_as_float(in[i] & 0xFFFF0000u);
        const float2 t = cs[4 * c + i];
        const float y0 = __fsub_rn(__fmul_rn(a, t.x), __fmul_rn(b, t.y));
        const float y1 = __fadd_rn(__fmul_rn(b, t.x), __fmul_rn(a, t.y));
        out[i] = pack_bf16x2(y0, y1);
      }
      dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) GTRACE(0, 5);
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, ABS_NT);
  }
}

// grid (H, 512/ABS_NT, ceil(M/128))
__global__ void __launch_bounds__(160) absorb_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                       const __grid_constant__ CUtensorMap tm_w,
                                                       AbsorbParams p) {
  absorb_q_cta(tm_q, tm_w, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// absorb_q and the cache append in one launch (they are independent: the query
// rows and the new cache rows): CTAs 0 .. n_abs-1 run absorb_q (CTA j = head
// j % H, column block (j / H) % 4, row block j / (4H)), the rest append 5 tokens
// each (one per warp) into the bf16 or FP8 cache.
template <bool FP8>
__global__ void __launch_bounds__(160) append_absorb_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                              const __grid_constant__ CUtensorMap tm_w,
                                                              AbsorbParams p, AppendParams a, int n_abs) {
  const int j = blockIdx.x;
  if (j < n_abs) {
    absorb_q_cta(tm_q, tm_w, p, j % p.H, (j / p.H) % (D_C / ABS_NT), j / (p.H * (D_C / ABS_NT)));
  } else {
    pdl_trigger();
    const int tok = (j - n_abs) * 5 + (threadIdx.x >> 5);
    if (FP8) append_token_fp8(a, tok, threadIdx.x & 31);
    else append_token(a, tok, threadIdx.x & 31);
  }
}

namespace {
constexpr size_t absorb_q_smem_bytes() { return (2 + ABS_NT / 64) * KB_BYTES + sizeof(GemmBarriers) + 1024; }
}  // namespace

cudaError_t launch_absorb_q(const CUtensorMap& tm_q, const CUtensorMap& tm_w, const AbsorbParams& p,
                            cudaStream_t s) {
  static DeviceFlags attr;
  const size_t smem = absorb_q_smem_bytes();
  cudaError_t e = once_per_device(attr, [&] {
    return cudaFuncSetAttribute(absorb_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  dim3 grid(p.H, D_C / ABS_NT, (p.M + 127) / 128);
  return launch_pdl(absorb_q_kernel, grid, dim3(160), smem, s, tm_q, tm_w, p);
}

cudaError_t launch_append_absorb_q(const CUtensorMap& tm_q, const CUtensorMap& tm_w, const AbsorbParams& p,
                                   const AppendParams& a, bool fp8, int num_sms, cudaStream_t s) {
  // One launch while absorb_q's CTAs fit on the GPU at once (measured: at
  // H = 128 its CTAs come in waves and the two launches are faster).
  const int n_abs = p.H * (D_C / ABS_NT) * ((p.M + 127) / 128);
  if (n_abs > num_sms) {
    if (a.n > 0) {
      const cudaError_t e = fp8 ? launch_append_fp8(a, s) : launch_append(a, s);
      if (e != cudaSuccess) return e;
    }
    return launch_absorb_q(tm_q, tm_w, p, s);
  }
  static DeviceFlags attr;
  const size_t smem = absorb_q_smem_bytes();
  const cudaError_t e = once_per_device(attr, [&] {
    const cudaError_t e0 =
        cudaFuncSetAttribute(append_absorb_q_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e0 != cudaSuccess) return e0;
    return cudaFuncSetAttribute(append_absorb_q_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  const dim3 grid(n_abs + (a.n + 4) / 5);
  return fp8 ? launch_pdl(append_absorb_q_kernel<true>, grid, dim3(160), smem, s, tm_q, tm_w, p, a, n_abs)
             : launch_pdl(append_absorb_q_kernel<false>, grid, dim3(160), smem, s, tm_q, tm_w, p, a, n_abs);
}

// grid (H, ceil(M/128)), 192 threads: one CTA per head and 128-row block, all
// 128 outputs (N = 128) and the whole 512-wide contraction, so every weight and
// o_lat byte is read once. Warp 0 streams K-blocks of 64 columns by TMA into a
// three-stage ring (W_UV[h] columns as the K-major B operand, the fp32 o_lat
// columns as two 32-column boxes); converter warps 2-5 (one row per thread)
// split each o_lat value into bf16 hi + lo (x = hi + lo + O(2^-17 |x|)) in the
// K-major swizzled A layout, two hi/lo stages; warp 1 issues
// D += A_hi B^T + A_lo B^T per K-block (8 MMAs, 64 in all).
namespace {
constexpr int EXP_NS = 3;                          // TMA stages (W + o_lat K-block)
constexpr int EXP_NH = 2;                          // hi/lo operand stages
constexpr uint32_t EXP_W = KB_BYTES;               // W_UV[h] rows 0..127 x 64 columns
constexpr uint32_t EXP_O = 2 * KB_BYTES;           // fp32 [128 rows x 64] as two 32-column boxes
constexpr uint32_t EXP_STAGE = EXP_W + EXP_O;
constexpr uint32_t EXP_HL = 2 * KB_BYTES;          // hi 16 KB | lo 16 KB
struct __align__(8) ExpandCtrl {
  uint64_t full[EXP_NS], empty[EXP_NS], hl_full[EXP_NH], hl_empty[EXP_NH], done;
  uint32_t tmem_base;
  int abort;
};
}  // namespace

__global__ void __launch_bounds__(192) expand_v_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                       const __grid_constant__ CUtensorMap tm_o,
                                                       ExpandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sring = smem;                         // EXP_NS x (W | o_lat)
  uint8_t* shl = sring + EXP_NS * EXP_STAGE;     // EXP_NH x (hi | lo)
  ExpandCtrl* ctl = reinterpret_cast<ExpandCtrl*>(shl + EXP_NH * EXP_HL);
  volatile int* abort = &ctl->abort;

  const int h = blockIdx.x;
  const int m0 = blockIdx.y * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) GTRACE(1, 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < EXP_NS; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1 + 4);   // the MMA commit (W) + the converter warps (o_lat)
    }
    for (int i = 0; i < EXP_NH; ++i) {
      mbar_init(smem_u32(&ctl->hl_full[i]), 4);
      mbar_init(smem_u32(&ctl->hl_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // the weight (a call input) of the first stages before the wait on the
      // previous kernel, o_lat (its output) after it
      for (int kb = 0; kb < EXP_NS; ++kb) {
        const uint32_t f = smem_u32(&ctl->full[kb]);
        mbar_arrive_expect_tx(f, EXP_W + 2 * 128 * p.rows_box);
        tma_load_3d(smem_u32(sring + kb * EXP_STAGE), &tm_w, f, 64 * kb, 0, h);
      }
      pdl_wait();
      for (int kb = 0; kb < 8; ++kb) {
        const int st = kb % EXP_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        uint8_t* stage = sring + st * EXP_STAGE;
        if (kb >= EXP_NS) {
          if (!mbar_wait(smem_u32(&ctl->empty[st]), ((kb / EXP_NS) & 1) ^ 1, abort, p.status)) break;
          mbar_arrive_expect_tx(f, EXP_W + 2 * 128 * p.rows_box);
          tma_load_3d(smem_u32(stage), &tm_w, f, 64 * kb, 0, h);
        }
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem_u32(stage + EXP_W + j * KB_BYTES), &tm_o, f, 64 * kb + 32 * j, h, m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
      bool ok = true;
      for (int kb = 0; kb < 8 && ok; ++kb) {
        const int st = kb % EXP_NS, hs = kb % EXP_NH;
        if (!(ok = mbar_wait(smem_u32(&ctl->hl_full[hs]), (kb / EXP_NH) & 1, abort, p.status))) break;
        if (kb == 0) GTRACE(1, 2);
        tc_fence_after();
        const uint32_t ahi = smem_u32(shl + hs * EXP_HL), alo = ahi + KB_BYTES;
        const uint32_t bw = smem_u32(sring + st * EXP_STAGE);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = smem_desc(bw + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
          mma_bf16_ss(tmem, smem_desc(ahi + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, (kb | k) != 0);
          mma_bf16_ss(tmem, smem_desc(alo + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, 1);
        }
        mma_commit(smem_u32(&ctl->hl_empty[hs]));
        mma_commit(smem_u32(&ctl->empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    // converters + epilogue: thread <-> row (TMEM lane 32*(warp%4) + lane)
    pdl_wait();
    if (threadIdx.x == 64) GTRACE(1, 1);
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = true;
    for (int kb = 0; kb < 8 && ok; ++kb) {
      const int st = kb % EXP_NS, hs = kb % EXP_NH;
      if (!(ok = mbar_wait(smem_u32(&ctl->full[st]), (kb / EXP_NS) & 1, abort, p.status))) break;
      if (!(ok = mbar_wait(smem_u32(&ctl->hl_empty[hs]), ((kb / EXP_NH) & 1) ^ 1, abort, p.status))) break;
      const uint8_t* src = sring + st * EXP_STAGE + EXP_W + row * 128;
      uint8_t* hi = shl + hs * EXP_HL + row * 128;
      uint8_t* lo = hi + KB_BYTES;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {           // 8 bf16 output chunks = 64 columns
        // fp32 columns 8*c8 .. 8*c8+7 live in box c8/4, chunks 2*(c8%4), 2*(c8%4)+1
        const uint8_t* box = src + (c8 >> 2) * KB_BYTES;
        const int c0 = 2 * (c8 & 3);
        const float4 x0 = *reinterpret_cast<const float4*>(box + ((c0 ^ (row & 7)) << 4));
        const float4 x1 = *reinterpret_cast<const float4*>(box + (((c0 + 1) ^ (row & 7)) << 4));
        const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hv[i] = pack_bf16x2(xs[2 * i], xs[2 * i + 1]);
          const float r0 = xs[2 * i] - __uint_as_float(hv[i] << 16);
          const float r1 = xs[2 * i + 1] - __uint_as_float(hv[i] & 0xFFFF0000u);
          lv[i] = pack_bf16x2(r0, r1);
        }
        const uint32_t off = (c8 ^ (row & 7)) << 4;
        *reinterpret_cast<uint4*>(hi + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(lo + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&ctl->empty[st]));
        mbar_arrive(smem_u32(&ctl->hl_full[hs]));
      }
    }
    if (ok) ok = mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
    if (threadIdx.x == 64) GTRACE(1, 4);
    tc_fence_after();
    const int r = m0 + row;
    if (ok) {
      // tcgen05.ld is warp-collective: every lane loads, rows past M store nothing
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((long long)r * p.H + h) * D_V);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        tmem_wait_ld();
        reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v));
        reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + 16));
        if (r < p.M) {
#pragma unroll
          for (int c = 0; c < 32; c += 8)
            dst[(c0 + c) / 8] = make_uint4(pack_bf16x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                           pack_bf16x2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])),
                                           pack_bf16x2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5])),
                                           pack_bf16x2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7])));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) GTRACE(1, 5);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Variant for few heads (one wave of clusters fills the GPU): grid (EXPAND_KS, H,
// ceil(M/128)) in clusters of EXPAND_KS CTAs along x, 192 threads. CTA j of a cluster contracts columns [128j, 128j+128) of the o_lat
// rows m0..m0+127 of head h with W_UV[h] (all 128 outputs): o_lat arrives by
// TMA as fp32 and converter warps 2-5 (one row per thread) split each value
// into bf16 hi + lo (x = hi + lo + O(2^-17 |x|)) in the K-major swizzled operand
// layout; one thread issues D = A_hi B^T + A_lo B^T (16 MMAs, N = 128). The
// fp32 partials of the cluster are summed through distributed shared memory:
// the valid rows of the block are dealt out in equal runs, one per CTA, and each
// CTA adds up the four partials of its run and writes them as bf16.
namespace {
struct __align__(8) ExpandClusterCtrl {
  uint64_t b_full, a_full, hl_full, done, recv_full;
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t EXC_B_BYTES = 2 * KB_BYTES;   // W_UV[h] rows 0..127, two 64-column K-blocks
constexpr uint32_t EXC_A_BYTES = 4 * KB_BYTES;   // fp32 [128 x 128] as four 32-column boxes
constexpr uint32_t EXC_HL_BYTES = 4 * KB_BYTES;  // per K-block: hi 16 KB | lo 16 KB
constexpr uint32_t EXC_RECV_BYTES = EXPAND_KS * 32 * 512;  // the cluster's partials of 32 output rows
// The valid rows of the row block at m0 are dealt out to the cluster's CTAs in
// equal runs: CTA k owns rows [k*R, k*R + n_k) of the block.
MLA_DEV int expand_run(int M, int m0) { return (min(128, M - m0) + EXPAND_KS - 1) / EXPAND_KS; }
MLA_DEV int expand_rows(int M, int m0, int k) {
  const int R = expand_run(M, m0);
  return max(0, min(min(128, M - m0), (k + 1) * R) - k * R);
}
}  // namespace

__global__ void __cluster_dims__(EXPAND_KS, 1, 1) __launch_bounds__(192)
    expand_v_cluster_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_o,
                    ExpandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sb = smem;                      // B operand
  uint8_t* sst = sb + EXC_B_BYTES;         // fp32 staging, then this CTA's partial sums
  uint8_t* shl = sst + EXC_A_BYTES;        // hi/lo A operand
  uint8_t* srecv = shl + EXC_HL_BYTES;     // partials of this CTA's output rows, slot k from CTA k
  ExpandClusterCtrl* ctl = reinterpret_cast<ExpandClusterCtrl*>(srecv + EXC_RECV_BYTES);
  volatile int* abort = &ctl->abort;

  const int j = blockIdx.x;                // rank in the cluster = K quarter
  const int h = blockIdx.y;
  const int m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) GTRACE(1, 0);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->b_full), 1);
    mbar_init(smem_u32(&ctl->a_full), 1);
    mbar_init(smem_u32(&ctl->hl_full), 4);
    mbar_init(smem_u32(&ctl->done), 1);
    mbar_init(smem_u32(&ctl->recv_full), 1);
    ctl->abort = 0;
    fence_mbar_init();
    // the cluster's partials of this CTA's valid output rows
    mbar_arrive_expect_tx(smem_u32(&ctl->recv_full), EXPAND_KS * expand_rows(p.M, m0, j) * 512);
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  // every CTA of the cluster has armed its recv_full before any copy targets it
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // the weight (a call input) before the wait on the previous kernel, o_lat after
      const uint32_t bf = smem_u32(&ctl->b_full), af = smem_u32(&ctl->a_full);
      mbar_arrive_expect_tx(bf, EXC_B_BYTES);
      for (int kb = 0; kb < 2; ++kb) tma_load_3d(smem_u32(sb + kb * KB_BYTES), &tm_w, bf, 128 * j + 64 * kb, 0, h);
      pdl_wait();
      mbar_arrive_expect_tx(af, 4 * 128 * p.rows_box);
      for (int q = 0; q < 4; ++q) tma_load_3d(smem_u32(sst + q * KB_BYTES), &tm_o, af, 128 * j + 32 * q, h, m0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
      bool ok = mbar_wait(smem_u32(&ctl->b_full), 0, abort, p.status);
      GTRACE(1, 2);
      if (ok) ok = mbar_wait(smem_u32(&ctl->hl_full), 0, abort, p.status);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint32_t ahi = smem_u32(shl + kb * 2 * KB_BYTES), alo = ahi + KB_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t bd = smem_desc(smem_u32(sb + kb * KB_BYTES) + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
            mma_bf16_ss(tmem, smem_desc(ahi + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, (kb | k) != 0);
            mma_bf16_ss(tmem, smem_desc(alo + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, 1);
          }
        }
        mma_commit(smem_u32(&ctl->done));
      }
    }
  } else {
    // converters, then the partial sums: thread <-> row (TMEM lane 32*(warp%4) + lane)
    pdl_wait();
    if (threadIdx.x == 64) GTRACE(1, 1);
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = mbar_wait(smem_u32(&ctl->a_full), 0, abort, p.status);
    if (ok) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        uint8_t* hi = shl + kb * 2 * KB_BYTES + row * 128;
        uint8_t* lo = hi + KB_BYTES;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {         // 8 bf16 output chunks = 64 columns
          // fp32 columns 64kb + 8c8 .. +7 live in box 2kb + c8/4, chunks 2(c8%4), 2(c8%4)+1
          const uint8_t* box = sst + (2 * kb + (c8 >> 2)) * KB_BYTES + row * 128;
          const int c0 = 2 * (c8 & 3);
          const float4 x0 = *reinterpret_cast<const float4*>(box + ((c0 ^ (row & 7)) << 4));
          const float4 x1 = *reinterpret_cast<const float4*>(box + (((c0 + 1) ^ (row & 7)) << 4));
          const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t hv[4], lv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hv[i] = pack_bf16x2(xs[2 * i], xs[2 * i + 1]);
            const float r0 = xs[2 * i] - __uint_as_float(hv[i] << 16);
            const float r1 = xs[2 * i + 1] - __uint_as_float(hv[i] & 0xFFFF0000u);
            lv[i] = pack_bf16x2(r0, r1);
          }
          const uint32_t off = (c8 ^ (row & 7)) << 4;
          *reinterpret_cast<uint4*>(hi + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          *reinterpret_cast<uint4*>(lo + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
        }
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctl->hl_full));
    if (ok) ok = mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
    if (threadIdx.x == 64) GTRACE(1, 4);
    tc_fence_after();
    if (ok) {
      // this CTA's fp32 partial of row `row` into the (consumed) staging
      // buffer, row-major (rows of CTA k's output at k * 16 KB), 16-byte chunk
      // c of a row at c ^ (row & 7)
      uint8_t* dst = sst + row * 512;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 64) {
        uint32_t v[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16)
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; c += 16) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + c));
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int ch = c0 / 4 + c;
          *reinterpret_cast<uint4*>(dst + ((ch ^ (row & 7)) << 4)) =
              make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
    }
  }
  // This CTA's partials of CTA k's valid rows travel by bulk copy into slot j
  // of CTA k's receive buffer, counted on CTA k's recv_full.
  if (warp >= 2) {
    if (threadIdx.x == 64) GTRACE(1, 6);
    named_bar_sync(1, 128);
    if (threadIdx.x == 64) {
      GTRACE(1, 7);
#pragma unroll
      for (int k = 0; k < EXPAND_KS; ++k) {
        const int rows = expand_rows(p.M, m0, k);
        if (rows > 0)
          bulk_copy_to_cluster(mapa_shared(smem_u32(srecv) + j * 16384, k),
                               smem_u32(sst) + k * expand_run(p.M, m0) * 512, rows * 512,
                               mapa_shared(smem_u32(&ctl->recv_full), k));
      }
      bulk_commit();
    }
  }
  if (warp >= 2) {
    // this CTA's rows of the output: the sum of the four partials, 4 threads
    // per row (32 columns each)
    const int t = threadIdx.x - 64;
    const int rr = t >> 2, cg = t & 3;
    const int nrows = expand_rows(p.M, m0, j);
    const int row = j * expand_run(p.M, m0) + rr;   // row in the block (its swizzle)
    const bool got = nrows > 0 && mbar_wait(smem_u32(&ctl->recv_full), 0, abort, p.status);
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
#pragma unroll
    for (int src = 0; src < EXPAND_KS; ++src) {
      const uint8_t* base = srecv + src * 16384 + rr * 512;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ch = 8 * cg + i;
        const float4 x = *reinterpret_cast<const float4*>(base + ((ch ^ (row & 7)) << 4));
        acc[4 * i] += x.x;
        acc[4 * i + 1] += x.y;
        acc[4 * i + 2] += x.z;
        acc[4 * i + 3] += x.w;
      }
    }
    const int r = m0 + row;
    if (got && rr < nrows && *abort == 0) {
      uint4* out = reinterpret_cast<uint4*>(p.out + ((long long)r * p.H + h) * D_V + 32 * cg);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        out[i] = make_uint4(pack_bf16x2(acc[8 * i], acc[8 * i + 1]), pack_bf16x2(acc[8 * i + 2], acc[8 * i + 3]),
                            pack_bf16x2(acc[8 * i + 4], acc[8 * i + 5]), pack_bf16x2(acc[8 * i + 6], acc[8 * i + 7]));
    }
  }
  // the outgoing copies have read this CTA's partials before it exits
  if (threadIdx.x == 64) bulk_wait_read();
  if (threadIdx.x == 64) GTRACE(1, 3);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) GTRACE(1, 5);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

size_t expand_v_smem_bytes() { return EXP_NS * EXP_STAGE + EXP_NH * EXP_HL + sizeof(ExpandCtrl) + 1024; }
size_t expand_v_cluster_smem_bytes() {
  return EXC_B_BYTES + EXC_A_BYTES + EXC_HL_BYTES + EXC_RECV_BYTES + sizeof(ExpandClusterCtrl) + 1024;
}

// One CTA per (head, 128-row block) when that already fills the GPU; with few
// heads the cluster variant splits each contraction over EXPAND_KS SMs.
cudaError_t launch_expand_v(const CUtensorMap& tm_w, const CUtensorMap& tm_o, const ExpandParams& p, int num_sms,
                            cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    const cudaError_t e0 = cudaFuncSetAttribute(expand_v_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)expand_v_smem_bytes());
    if (e0 != cudaSuccess) return e0;
    return cudaFuncSetAttribute(expand_v_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)expand_v_cluster_smem_bytes());
  });
  if (e != cudaSuccess) return e;
  const int mblocks = (p.M + 127) / 128;
  if (p.H * mblocks * EXPAND_KS <= num_sms)
    return launch_pdl(expand_v_cluster_kernel, dim3(EXPAND_KS, p.H, mblocks), dim3(192),
                      expand_v_cluster_smem_bytes(), s, tm_w, tm_o, p);
  return launch_pdl(expand_v_kernel, dim3(p.H, mblocks), dim3(192), expand_v_smem_bytes(), s, tm_w, tm_o, p);
}

}  // namespace mla
