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

constexpr int ABS_NT = 256;            // output columns per CTA (absorb_q)
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
  uint8_t* sb = smem + 2 * KB_BYTES;        // 4 x 16 KB
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(smem + 6 * KB_BYTES);

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

  if (threadIdx.x == 0) {
    const uint32_t full = smem_u32(&bars->full);
    mbar_arrive_expect_tx(full, 6 * KB_BYTES);
    for (int kb = 0; kb < 2; ++kb) tma_load_3d(smem_u32(sa + kb * KB_BYTES), &tm_q, full, 64 * kb, h, m0);
    for (int a = 0; a < 4; ++a) tma_load_3d(smem_u32(sb + a * KB_BYTES), &tm_w, full, n0 + 64 * a, 0, h);
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
    for (int c = 0; c < ABS_NT; c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + lane_base + c, v);
      tmem_wait_ld();
      reg_fence16(v);
      if (r < p.M) {
        uint4 o0, o1;
        o0.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
        o0.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
        o0.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
        o0.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
        o1.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
        o1.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
        o1.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
        o1.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
        reinterpret_cast<uint4*>(dst + c)[0] = o0;
        reinterpret_cast<uint4*>(dst + c)[1] = o1;
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
  const size_t smem = 6 * KB_BYTES + sizeof(GemmBarriers) + 1024;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.H, D_C / ABS_NT, (p.M + 127) / 128);
  absorb_q_kernel<<<grid, 128, smem, s>>>(tm_q, tm_w, p);
  return cudaGetLastError();
}

// grid (H, 128/EXPAND_NT, ceil(M/128)), 128 threads.
// A = o_lat rows of head h, fp32 split into bf16 hi + lo parts written by the
// threads (K-major, two stages of one 64-wide K-block), B = W_UV[h] rows
// n0..n0+63 (K-major, 8 K-blocks by TMA). D += A_hi B^T + A_lo B^T.
__global__ void __launch_bounds__(128) expand_v_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                       ExpandParams p) {
  int* status = p.status;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  constexpr uint32_t B_KB = EXPAND_NT * 128;   // bytes per B K-block
  uint8_t* sb = smem;                          // 8 x B_KB
  uint8_t* sa = smem + 8 * B_KB;               // 2 stages x (hi 16 KB, lo 16 KB)
  GemmBarriers* bars = reinterpret_cast<GemmBarriers*>(sa + 4 * KB_BYTES);

  const int h = blockIdx.x;
  const int n0 = blockIdx.y * EXPAND_NT;
  const int m0 = blockIdx.z * 128;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->full), 1);
    mbar_init(smem_u32(&bars->stage_done[0]), 1);
    mbar_init(smem_u32(&bars->stage_done[1]), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), EXPAND_NT);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (threadIdx.x == 0) {
    const uint32_t full = smem_u32(&bars->full);
    mbar_arrive_expect_tx(full, 8 * B_KB);
    for (int kb = 0; kb < 8; ++kb) tma_load_3d(smem_u32(sb + kb * B_KB), &tm_w, full, 64 * kb, n0, h);
  }

  bool ok = true;
  uint32_t stage_phase[2] = {0, 0};
  const int sub_row = threadIdx.x >> 4;   // 0..7
  const int col4 = threadIdx.x & 15;      // float4 index within the 64-wide block
#pragma unroll 1
  for (int kb = 0; kb < 8 && ok; ++kb) {
    const int st = kb & 1;
    if (kb >= 2) {
      ok = mbar_wait(smem_u32(&bars->stage_done[st]), stage_phase[st], &bars->abort, status);
      stage_phase[st] ^= 1;
      if (!ok) break;
    }
    uint8_t* ahi = sa + st * 2 * KB_BYTES;
    uint8_t* alo = ahi + KB_BYTES;
#pragma unroll 4
    for (int pass = 0; pass < 16; ++pass) {
      const int row = pass * 8 + sub_row;
      const int r = m0 + row;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < p.M)
        x = reinterpret_cast<const float4*>(p.o_lat + ((long long)r * p.H + h) * D_C + kb * 64)[col4];
      const uint32_t h01 = pack_bf16x2(x.x, x.y), h23 = pack_bf16x2(x.z, x.w);
      const float rx = x.x - __uint_as_float(h01 << 16), ry = x.y - __uint_as_float(h01 & 0xFFFF0000u);
      const float rz = x.z - __uint_as_float(h23 << 16), rw = x.w - __uint_as_float(h23 & 0xFFFF0000u);
      const uint32_t l01 = pack_bf16x2(rx, ry), l23 = pack_bf16x2(rz, rw);
      const uint32_t off = row * 128 + ((((col4 >> 1) ^ (row & 7)) << 4) | ((col4 & 1) << 3));
      *reinterpret_cast<uint2*>(ahi + off) = make_uint2(h01, h23);
      *reinterpret_cast<uint2*>(alo + off) = make_uint2(l01, l23);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
      if (kb == 0) ok = mbar_wait(smem_u32(&bars->full), 0, &bars->abort, status);
      if (ok) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, EXPAND_NT, 0, 0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = smem_desc(smem_u32(sb + kb * B_KB) + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
          const uint64_t ah = smem_desc(smem_u32(ahi) + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
          const uint64_t al = smem_desc(smem_u32(alo) + k * 32, 16, 1024, SMEM_SWIZZLE_128B);
          mma_bf16_ss(tmem, ah, bd, idesc, (kb | k) != 0);
          mma_bf16_ss(tmem, al, bd, idesc, 1);
        }
        mma_commit(smem_u32(&bars->stage_done[st]));
      }
    }
    __syncthreads();
    ok = ok && !bars->abort;
  }
  // stage 1 was committed last (kb = 7) and covers every earlier MMA.
  if (ok) ok = mbar_wait(smem_u32(&bars->stage_done[1]), stage_phase[1], &bars->abort, status);
  tc_fence_after();
  if (ok) {
    const int r = m0 + threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint16_t* dst = p.out + ((long long)r * p.H + h) * D_V + n0;
#pragma unroll 1
    for (int c = 0; c < EXPAND_NT; c += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + lane_base + c, v);
      tmem_wait_ld();
      reg_fence16(v);
      if (r < p.M) {
        uint4 o0, o1;
        o0.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
        o0.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
        o0.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
        o0.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
        o1.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
        o1.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
        o1.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
        o1.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
        reinterpret_cast<uint4*>(dst + c)[0] = o0;
        reinterpret_cast<uint4*>(dst + c)[1] = o1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, EXPAND_NT);
}

cudaError_t launch_expand_v(const CUtensorMap& tm_w, const ExpandParams& p, cudaStream_t s) {
  static bool attr = false;
  const size_t smem = 8 * EXPAND_NT * 128 + 4 * KB_BYTES + sizeof(GemmBarriers) + 1024;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(expand_v_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(p.H, D_V / EXPAND_NT, (p.M + 127) / 128);
  expand_v_kernel<<<grid, 128, smem, s>>>(tm_w, p);
  return cudaGetLastError();
}

}  // namespace mla
