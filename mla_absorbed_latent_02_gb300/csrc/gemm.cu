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
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

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

// grid (H, 512/ABS_NT, ceil(M/128)), 128 threads.
// A = q_nope rows of head h (K-major, 2 K-blocks of 64), B = W_UK[h][:, n0:n0+256]
// (N-contiguous, MN-major, 4 atoms of 64 columns x 128 K-rows).
__global__ void __launch_bounds__(128) absorb_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                       const __grid_constant__ CUtensorMap tm_w,
                                                       AbsorbParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sa = smem;                       // 2 x 16 KB
  uint8_t* sb = smem + 2 * KB_BYTES;        // ABS_NT/64 x 16 KB
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(smem + (2 + ABS_NT / 64) * KB_BYTES);

  const int h = blockIdx.x;
  const int n0 = blockIdx.y * ABS_NT;
  const int m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->full), 1);
    mbar_init(smem_u32(&bars->done), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), ABS_NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  pdl_trigger();
  pdl_wait();

  if (threadIdx.x == 0) {
    const uint32_t full = smem_u32(&bars->full);
    mbar_arrive_expect_tx(full, (2 + ABS_NT / 64) * KB_BYTES);
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(smem_u32(sa + kb * KB_BYTES), &tm_q, full, 64 * kb, h, m0);
    for (int a = 0; a < ABS_NT / 64; ++a) tma_load_3d(smem_u32(sb + a * KB_BYTES), &tm_w, full, n0 + 64 * a, 0, h);
    if (mbar_wait(full, 0, &bars->abort, p.status)) {
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

  // RoPE of the query's rope part (one thread per row), while the MMA runs.
  const int r = m0 + threadIdx.x;
  if (blockIdx.y == 0 && r < p.M) {
    const int pos = p.q_pos[r];
    uint4* dst = reinterpret_cast<uint4*>(p.q_abs + ((long long)r * p.H + h) * ROW + D_C);
    const uint4* src = reinterpret_cast<const uint4*>(p.q_rope + ((long long)r * p.H + h) * D_ROPE);
    if (pos < 0 || pos >= p.max_pos) {
      atomicOr(p.status, MLA_DEVERR_BOUNDS);
    } else {
      const float2* tab = p.rope + (long long)pos * (D_ROPE / 2);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = src[c];
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = __uint_as_float(in[i] << 16);
          const float b = __uint_as_float(in[i] & 0xFFFF0000u);
          const float2 cs = tab[4 * c + i];
          const float y0 = __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y));
          const float y1 = __fadd_rn(__fmul_rn(b, cs.x), __fmul_rn(a, cs.y));
          out[i] = pack_bf16x2(y0, y1);
        }
        dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }

  __syncwarp();
  const bool ok = mbar_wait(smem_u32(&bars->done), 0, &bars->abort, p.status);
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
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ABS_NT);
}

cudaError_t launch_absorb_q(const CUtensorMap& tm_q, const CUtensorMap& tm_w, const AbsorbParams& p,
                            cudaStream_t s) {
  static bool attr = false;
  const size_t smem = (2 + ABS_NT / 64) * KB_BYTES + sizeof(GemmBarriers) + 1024;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.H, D_C / ABS_NT, (p.M + 127) / 128);
  return launch_pdl(absorb_q_kernel, grid, dim3(128), smem, s, tm_q, tm_w, p);
}

// grid (H, 128/EXPAND_NT, ceil(M/128)), 192 threads.
// A = o_lat rows of head h (fp32), streamed by TMA in 64-column K-blocks into a
// two-stage fp32 staging ring; converter warps 2-5 (one row per thread) split
// each value into bf16 hi + lo (x = hi + lo + O(2^-17 |x|)) in the K-major
// swizzled operand layout; B = W_UV[h] rows n0..n0+EXPAND_NT-1 (K-major, all 8
// K-blocks by TMA). One thread issues D += A_hi B^T + A_lo B^T per K-block.
namespace {
struct __align__(8) ExpandCtrl {
  uint64_t b_full, a_full[2], a_empty[2], hl_full[2], hl_empty[2], done;
  uint32_t tmem_base;
  int abort;
};
}  // namespace

__global__ void __launch_bounds__(192) expand_v_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                       const __grid_constant__ CUtensorMap tm_o,
                                                       ExpandParams p) {
  constexpr uint32_t B_KB = EXPAND_NT * 128;     // bytes per B K-block
  constexpr uint32_t STAGE = 2 * KB_BYTES;       // fp32 [128 rows x 64] as two 32-column boxes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  uint8_t* sb = smem;                            // 8 x B_KB
  uint8_t* sst = sb + 8 * B_KB;                  // 2 staging stages
  uint8_t* shl = sst + 2 * STAGE;                // 2 x (hi 16 KB | lo 16 KB)
  ExpandCtrl* ctl = reinterpret_cast<ExpandCtrl*>(shl + 2 * STAGE);
  volatile int* abort = &ctl->abort;

  const int h = blockIdx.x;
  const int n0 = blockIdx.y * EXPAND_NT;
  const int m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->b_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->a_full[i]), 1);
      mbar_init(smem_u32(&ctl->a_empty[i]), 4);
      mbar_init(smem_u32(&ctl->hl_full[i]), 4);
      mbar_init(smem_u32(&ctl->hl_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), EXPAND_NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bf = smem_u32(&ctl->b_full);
      mbar_arrive_expect_tx(bf, 8 * B_KB);
      for (int kb = 0; kb < 8; ++kb) tma_load_3d(smem_u32(sb + kb * B_KB), &tm_w, bf, 64 * kb, n0, h);
      for (int kb = 0; kb < 8; ++kb) {
        const int st = kb & 1;
        if (!mbar_wait(smem_u32(&ctl->a_empty[st]), ((kb >> 1) & 1) ^ 1, abort, p.status)) break;
        const uint32_t af = smem_u32(&ctl->a_full[st]);
        mbar_arrive_expect_tx(af, STAGE);
        for (int j = 0; j < 2; ++j)
          tma_load_3d(smem_u32(sst + st * STAGE + j * KB_BYTES), &tm_o, af, 64 * kb + 32 * j, h, m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, EXPAND_NT, 0, 0);
      bool ok = mbar_wait(smem_u32(&ctl->b_full), 0, abort, p.status);
      for (int kb = 0; kb < 8 && ok; ++kb) {
        const int st = kb & 1;
        if (!(ok = mbar_wait(smem_u32(&ctl->hl_full[st]), (kb >> 1) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t ahi = smem_u32(shl + st * STAGE), alo = ahi + KB_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = smem_desc(smem_u32(sb + kb * B_KB) + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
          mma_bf16_ss(tmem, smem_desc(ahi + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, (kb | k) != 0);
          mma_bf16_ss(tmem, smem_desc(alo + k * 32, 16, 1024, SMEM_SWIZZLE_128B), bd, idesc, 1);
        }
        mma_commit(smem_u32(&ctl->hl_empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    // converters + epilogue: thread <-> row (TMEM lane 32*(warp%4) + lane)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool ok = true;
    for (int kb = 0; kb < 8 && ok; ++kb) {
      const int st = kb & 1;
      if (!(ok = mbar_wait(smem_u32(&ctl->a_full[st]), (kb >> 1) & 1, abort, p.status))) break;
      if (!(ok = mbar_wait(smem_u32(&ctl->hl_empty[st]), ((kb >> 1) & 1) ^ 1, abort, p.status))) break;
      const uint8_t* src = sst + st * STAGE + row * 128;
      uint8_t* hi = shl + st * STAGE + row * 128;
      uint8_t* lo = hi + KB_BYTES;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {           // 8 bf16 output chunks = 64 columns
        // fp32 columns 8*c8 .. 8*c8+7 live in box j = c8/4, chunks 2*(c8%4), 2*(c8%4)+1
        const uint8_t* box = src + (c8 >> 2) * KB_BYTES;
        const int c0 = 2 * (c8 & 3);
        const float4 x0 = *reinterpret_cast<const float4*>(box + (((c0) ^ (row & 7)) << 4));
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
        const uint32_t off = ((c8 ^ (row & 7)) << 4);
        *reinterpret_cast<uint4*>(hi + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4*>(lo + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&ctl->a_empty[st]));
        mbar_arrive(smem_u32(&ctl->hl_full[st]));
      }
    }
    if (ok) ok = mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
    tc_fence_after();
    if (ok) {
      const int r = m0 + row;
      uint32_t v[EXPAND_NT];
#pragma unroll
      for (int c = 0; c < EXPAND_NT; c += 16)
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < EXPAND_NT; c += 16) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + c));
      if (r < p.M) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + ((long long)r * p.H + h) * D_V + n0);
#pragma unroll
        for (int c = 0; c < EXPAND_NT; c += 8)
          dst[c / 8] = make_uint4(pack_bf16x2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                  pack_bf16x2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])),
                                  pack_bf16x2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5])),
                                  pack_bf16x2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, EXPAND_NT);
  }
}

size_t expand_v_smem_bytes() { return 8 * EXPAND_NT * 128 + 4 * 2 * KB_BYTES + sizeof(ExpandCtrl) + 1024; }

cudaError_t launch_expand_v(const CUtensorMap& tm_w, const CUtensorMap& tm_o, const ExpandParams& p,
                            cudaStream_t s) {
  static bool attr = false;
  const size_t smem = expand_v_smem_bytes();
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expand_v_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.H, D_V / EXPAND_NT, (p.M + 127) / 128);
  return launch_pdl(expand_v_kernel, grid, dim3(192), smem, s, tm_w, tm_o, p);
}

}  // namespace mla
