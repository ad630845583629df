// Output projection of the attention block: y = W_O concat_h(o_h).
//
// o [M, H, 128] bf16 is the per-head output of expand_v (head-major, so each
// row is the concatenation the module's view(B, L, n_h * d_h) produces), W_O
// [d_model, H*128] bf16 the nn.Linear(n_h * d_h -> d_model) weight ("80 行
// PyTorch 从零写 DeepSeek 的 MLA" §2, the forward's last line; "DeepSeek-V2-Lite
// 真实权重执行审计" §3.3, o_proj / wo), y [M, d_model] fp32.
//
// Decode rows are few (M = B*Hq) and the contraction is long (K = H*128), so the
// weight is spread over many SMs by splitting K: grid (d_model/128, KS,
// ceil(M/NB)); CTA (f, ks, mb) contracts K-blocks [ks*KB/KS, (ks+1)*KB/KS) of 64
// columns for output features 128f .. 128f+127 (the last tile may be partial:
// the weight's missing rows read as zeros) and rows of its row block, with
// tokens on the MMA's N axis ("swap AB": D^T[feature x row] = W_O tile . x^T, both
// operands K-major, 128-byte swizzle, four-stage TMA ring). After a transpose
// through shared memory the partials are added into y with 16-byte reductions
// in L2 (4 consecutive features of a row each). y needs no zero-fill before the
// call: the first split of a tile to start (a ticket in global memory) zeroes
// the tile while its products run and then raises the tile's flag; every split
// checks the flag before adding (by then it is almost always up). A split only
// ever waits for one that is already running and waits for nothing itself, so
// no co-residency is needed. The last split of a tile clears its words for the
// next call. With one split the partial is stored.
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {

namespace {

constexpr int OP_NS = 4;                    // TMA stages
constexpr uint32_t OP_A_BYTES = 16384;      // W_O tile: 128 features x 64 columns

struct __align__(8) OutProjCtrl {
  uint64_t full[OP_NS], empty[OP_NS], done;
  uint32_t tmem_base;
  int abort;
  unsigned ticket;         // this split's arrival order at its tile
};

MLA_DEV unsigned ld_acquire_gpu_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
MLA_DEV void st_release_gpu_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

MLA_DEV uint8_t* op_align1k(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// N of the MMA: the row block's height rounded up to 16 (the tcgen05 step for M = 128).
template <int NB>
__global__ void __launch_bounds__(192) out_proj_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                       const __grid_constant__ CUtensorMap tm_x,
                                                       OutProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = op_align1k(smem_raw);
  constexpr uint32_t B_BYTES = 128u * NB;  // NB rows x 64 columns x 2 bytes
  constexpr uint32_t STAGE = OP_A_BYTES + B_BYTES;
  OutProjCtrl* ctl = reinterpret_cast<OutProjCtrl*>(smem + OP_NS * STAGE);
  volatile int* abort = &ctl->abort;

  const int f0 = blockIdx.x * 128;
  const int ks = blockIdx.y;
  const int m0 = blockIdx.z * NB;
  const int kb0 = static_cast<int>((long long)ks * p.KB / gridDim.y);
  const int kb1 = static_cast<int>((long long)(ks + 1) * p.KB / gridDim.y);
  const int nkb = kb1 - kb0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t TMEM_COLS = NB <= 32 ? 32u : (NB <= 64 ? 64u : (NB <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int i = 0; i < OP_NS; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // weight tiles (a call input) of the first stages before the wait on the
      // previous kernel, the activations after it
      for (int i = 0; i < nkb && i < OP_NS; ++i) {
        const uint32_t f = smem_u32(&ctl->full[i]);
        mbar_arrive_expect_tx(f, OP_A_BYTES + 128u * p.rows_box);
        tma_load_2d(smem_u32(smem + i * STAGE), &tm_w, f, 64 * (kb0 + i), f0);
      }
      pdl_wait();
      for (int i = 0; i < nkb; ++i) {
        const int st = i % OP_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        uint8_t* stage = smem + st * STAGE;
        if (i >= OP_NS) {
          if (!mbar_wait(smem_u32(&ctl->empty[st]), ((i / OP_NS) & 1) ^ 1, abort, p.status)) break;
          mbar_arrive_expect_tx(f, OP_A_BYTES + 128u * p.rows_box);
          tma_load_2d(smem_u32(stage), &tm_w, f, 64 * (kb0 + i), f0);
        }
        tma_load_2d(smem_u32(stage + OP_A_BYTES), &tm_x, f, 64 * (kb0 + i), m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NB, 0, 0);
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        const int st = i % OP_NS;
        if (!(ok = mbar_wait(smem_u32(&ctl->full[st]), (i / OP_NS) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + st * STAGE), b = a + OP_A_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, smem_desc(a + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                      smem_desc(b + 32 * k, 16, 1024, SMEM_SWIZZLE_128B), idesc, (i | k) != 0);
        mma_commit(smem_u32(&ctl->empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    // The partial D^T[feature x row] goes through shared memory (the ring is free
    // once the MMAs are done) into row-major order, so that each reduction adds 4
    // consecutive features of a row (red.global.add.v4.f32): thread <-> feature
    // 32*(warp%4) + lane (its TMEM lane) for the copy; every lane loads
    // (tcgen05.ld is warp-collective).
    pdl_wait();
    const int q = warp & 3;
    const int fl = q * 32 + lane;                 // feature within the tile
    const int t = threadIdx.x - 64;               // 0..127
    const int rows = min(NB, p.M - m0);
    const int KS = gridDim.y;
    unsigned* words = p.sync + 3 * (blockIdx.z * gridDim.x + blockIdx.x);   // ticket, zeroed, done
    if (KS > 1) {
      if (t == 0) ctl->ticket = atomicAdd(words, 1u);
      named_bar_sync(1, 128);
      if (ctl->ticket == 0u) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int i = t; i < rows * 32; i += 128) {
          const int r = i >> 5, f4 = (i & 31) * 4;
          if (f0 + f4 < p.d_model) *reinterpret_cast<float4*>(p.y + (long long)(m0 + r) * p.d_model + f0 + f4) = z;
        }
        named_bar_sync(1, 128);
        if (t == 0) {
          __threadfence();
          st_release_gpu_u32(words + 1, 1u);
        }
      }
    }
    const bool ok = nkb > 0 && mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
    tc_fence_after();
    float* stage_t = reinterpret_cast<float*>(smem);   // [NB rows][132] (4 floats of padding)
    if (ok) {
#pragma unroll 1
      for (int c0 = 0; c0 < NB; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
        tmem_wait_ld();
        reg_fence16(v);
#pragma unroll
        for (int c = 0; c < 16; ++c) stage_t[(c0 + c) * 132 + fl] = __uint_as_float(v[c]);
      }
    }
    if (KS > 1 && t == 0 && ctl->ticket != 0u) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_gpu_u32(words + 1) == 0u) {
        if (globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
          atomicOr(p.status, MLA_DEVERR_TIMEOUT);
          *abort = 1;
          break;
        }
        __nanosleep(32);
      }
    }
    named_bar_sync(1, 128);
    if (ok && *abort == 0) {
#pragma unroll 1
      for (int i = t; i < rows * 32; i += 128) {
        const int r = i >> 5, f4 = (i & 31) * 4;
        if (f0 + f4 < p.d_model) {
          const float4 v = *reinterpret_cast<const float4*>(stage_t + r * 132 + f4);
          float* dst = p.y + (long long)(m0 + r) * p.d_model + f0 + f4;
          if (KS == 1) {
            *reinterpret_cast<float4*>(dst) = v;
          } else {
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v.x), "f"(v.y), "f"(v.z),
                         "f"(v.w)
                         : "memory");
          }
        }
      }
    }
    // every split of the tile has taken its ticket and is past its wait once
    // the done count is full: clear the words for the next call
    if (KS > 1 && t == 0 && atomicAdd(words + 2, 1u) == static_cast<unsigned>(KS - 1)) {
      words[0] = 0u;
      words[1] = 0u;
      words[2] = 0u;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NB>
size_t out_proj_smem() {
  return OP_NS * (OP_A_BYTES + 128u * NB) + sizeof(OutProjCtrl) + 1024;
}

template <int NB>
cudaError_t launch_nb(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p, dim3 grid,
                      cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(out_proj_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)out_proj_smem<NB>());
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(out_proj_kernel<NB>, grid, dim3(192), out_proj_smem<NB>(), s, tm_w, tm_x, p);
}

// ---------------------------------------------------------------------------
// The value up-projection folded into the output projection:
//   W_OV[f, h*512 + c] = sum_v W_O[f, h*128 + v] W_UV[h][v, c]
// so that y = W_OV concat_h(o_lat[., h, :]) replaces expand_v followed by the
// output projection (the value absorption of "DeepSeek MLA 吸收式缓存" §2.3
// carried into the module's last line, "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2).
// A one-time weight transform: CUDA-core tiles of 64 features x 64 latent
// columns of one head, K = 128, fp32 accumulation, bf16 (nearest even) out.
__global__ void __launch_bounds__(256) absorb_w_o_kernel(const uint16_t* __restrict__ w_o,
                                                         const uint16_t* __restrict__ w_uv, uint16_t* w_ov,
                                                         int H, int d_model) {
  __shared__ uint16_t so[64][130];   // W_O rows f0.., columns v of head h (bf16 bits)
  __shared__ uint16_t su[128][66];   // W_UV[h] rows v, latent columns c0..
  const int c0 = blockIdx.x * 64, f0 = blockIdx.y * 64, h = blockIdx.z;
  const int tid = threadIdx.x;
  for (int i = tid; i < 64 * 128; i += 256) {
    const int f = i >> 7, v = i & 127;
    so[f][v] = w_o[(long long)(f0 + f) * H * D_V + h * D_V + v];
  }
  for (int i = tid; i < 128 * 64; i += 256) {
    const int v = i >> 6, c = i & 63;
    su[v][c] = w_uv[((long long)h * D_V + v) * D_C + c0 + c];
  }
  __syncthreads();
  const int tf = tid >> 4, tc = tid & 15;   // 4 x 4 outputs: features tf + 16i, columns tc + 16j
  float acc[4][4] = {};
#pragma unroll 4
  for (int v = 0; v < 128; ++v) {
    float a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = __uint_as_float(static_cast<uint32_t>(so[tf + 16 * i][v]) << 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = __uint_as_float(static_cast<uint32_t>(su[v][tc + 16 * j]) << 16);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t r = pack_bf16x2(acc[i][j], 0.f);
      w_ov[(long long)(f0 + tf + 16 * i) * H * D_C + h * D_C + c0 + tc + 16 * j] = static_cast<uint16_t>(r & 0xFFFFu);
    }
}

// y = W_OV x for x = o_lat [M, H*512] fp32 (the attention's output, heads
// concatenated head-major): the output projection's split-K GEMM with the
// activations loaded in fp32 (TMA, 32-column boxes, 128-byte swizzle) and
// rounded to bf16 (nearest even) into the MMA's K-major operand by the four
// epilogue warps, which are idle until the products are done. Each CTA covers
// FT feature tiles of 128 (FT accumulators of NB columns), so one converted
// activation tile serves FT weight tiles.
template <int NB>
struct OpLatCfg {
  static constexpr int FT = NB <= 128 ? 4 : 1;                        // feature tiles per CTA
  static constexpr uint32_t A_BYTES = FT * OP_A_BYTES;                // FT weight tiles
  static constexpr uint32_t XF_BYTES = 256u * NB;                     // fp32 x: NB rows x 64 columns
  static constexpr uint32_t XB_BYTES = 128u * NB;                     // bf16 x
  static constexpr uint32_t STAGE = A_BYTES + XF_BYTES + XB_BYTES;
  static constexpr int NS = (3 * STAGE <= 200u * 1024u) ? 3 : 2;      // stages
  static constexpr uint32_t TMEM_NEED = FT * NB;
  static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 32 ? 32u : (TMEM_NEED <= 64 ? 64u :
                                        (TMEM_NEED <= 128 ? 128u : (TMEM_NEED <= 256 ? 256u : 512u)));
};

struct __align__(8) OpLatCtrl {
  uint64_t full[4], conv[4], empty[4], done;
  uint32_t tmem_base;
  int abort;
};

template <int NB>
__global__ void __launch_bounds__(192) out_proj_latent_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                              const __grid_constant__ CUtensorMap tm_x,
                                                              OutProjParams p) {
  using K = OpLatCfg<NB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = op_align1k(smem_raw);
  OpLatCtrl* ctl = reinterpret_cast<OpLatCtrl*>(smem + K::NS * K::STAGE);
  volatile int* abort = &ctl->abort;

  const int f0 = blockIdx.x * 128 * K::FT;
  const int ks = blockIdx.y;
  const int m0 = blockIdx.z * NB;
  const int kb0 = static_cast<int>((long long)ks * p.KB / gridDim.y);
  const int kb1 = static_cast<int>((long long)(ks + 1) * p.KB / gridDim.y);
  const int nkb = kb1 - kb0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < K::NS; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->conv[i]), 4);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), K::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  const uint32_t xf_tx = 2u * 128u * p.rows_box;   // two 32-column fp32 boxes of rows_box rows

  if (warp == 0) {
    if (lane == 0) {
      auto load_w = [&](int i, int st, uint32_t f) {
        for (int ft = 0; ft < K::FT; ++ft)
          tma_load_2d(smem_u32(smem + st * K::STAGE + ft * OP_A_BYTES), &tm_w, f, 64 * (kb0 + i), f0 + 128 * ft);
      };
      for (int i = 0; i < nkb && i < K::NS; ++i) {
        const uint32_t f = smem_u32(&ctl->full[i]);
        mbar_arrive_expect_tx(f, K::A_BYTES + xf_tx);
        load_w(i, i, f);
      }
      pdl_wait();
      for (int i = 0; i < nkb; ++i) {
        const int st = i % K::NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        uint8_t* stage = smem + st * K::STAGE;
        if (i >= K::NS) {
          if (!mbar_wait(smem_u32(&ctl->empty[st]), ((i / K::NS) & 1) ^ 1, abort, p.status)) break;
          mbar_arrive_expect_tx(f, K::A_BYTES + xf_tx);
          load_w(i, st, f);
        }
        for (int bx = 0; bx < 2; ++bx)
          tma_load_2d(smem_u32(stage + K::A_BYTES + bx * 128u * NB), &tm_x, f, 64 * (kb0 + i) + 32 * bx, m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NB, 0, 0);
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        const int st = i % K::NS;
        if (!(ok = mbar_wait(smem_u32(&ctl->conv[st]), (i / K::NS) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + st * K::STAGE), b = a + K::A_BYTES + K::XF_BYTES;
#pragma unroll
        for (int ft = 0; ft < K::FT; ++ft)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(tmem + ft * NB, smem_desc(a + ft * OP_A_BYTES + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                        smem_desc(b + 32 * k, 16, 1024, SMEM_SWIZZLE_128B), idesc, (i | k) != 0);
        mma_commit(smem_u32(&ctl->empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    pdl_wait();
    const int t = threadIdx.x - 64;               // 0..127
    bool ok = true;
    // convert: 16-byte bf16 chunk c8 (columns 8*c8 .. 8*c8+7) of row r comes
    // from fp32 chunks 2*(c8 & 3), 2*(c8 & 3) + 1 of box c8 >> 2 (both swizzled
    // by row, chunk j of row r at j ^ (r % 8))
#pragma unroll 1
    for (int i = 0; i < nkb && ok; ++i) {
      const int st = i % K::NS;
      if (!(ok = mbar_wait(smem_u32(&ctl->full[st]), (i / K::NS) & 1, abort, p.status))) break;
      const uint32_t xf = smem_u32(smem + st * K::STAGE + K::A_BYTES);
      const uint32_t xb = xf + K::XF_BYTES;
#pragma unroll 1
      for (int task = t; task < NB * 8; task += 128) {
        const int r = task >> 3, c8 = task & 7;
        const uint32_t box = xf + (c8 >> 2) * 128u * NB + r * 128;
        const int j0 = 2 * (c8 & 3);
        float4 v0, v1;
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v0.x), "=f"(v0.y), "=f"(v0.z), "=f"(v0.w)
                     : "r"(box + (((j0) ^ (r & 7)) << 4)));
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v1.x), "=f"(v1.y), "=f"(v1.z), "=f"(v1.w)
                     : "r"(box + (((j0 + 1) ^ (r & 7)) << 4)));
        const uint32_t dst = xb + r * 128 + ((c8 ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pack_bf16x2(v0.x, v0.y)),
                     "r"(pack_bf16x2(v0.z, v0.w)), "r"(pack_bf16x2(v1.x, v1.y)), "r"(pack_bf16x2(v1.z, v1.w))
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->conv[st]));
    }
    // epilogue per feature tile: as the output projection (transpose through
    // shared memory into row-major order, 16-byte L2 reductions of 4
    // consecutive features)
    const int q = warp & 3;
    const int fl = q * 32 + lane;
    ok = ok && nkb > 0 && mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
    tc_fence_after();
    float* stage_t = reinterpret_cast<float*>(smem);   // [NB rows][132]
    const int rows = min(NB, p.M - m0);
#pragma unroll 1
    for (int ft = 0; ft < K::FT && ok; ++ft) {
      const int fb = f0 + 128 * ft;
#pragma unroll 1
      for (int c0 = 0; c0 < NB; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + ft * NB + c0, v);
        tmem_wait_ld();
        reg_fence16(v);
#pragma unroll
        for (int c = 0; c < 16; ++c) stage_t[(c0 + c) * 132 + fl] = __uint_as_float(v[c]);
      }
      named_bar_sync(1, 128);
#pragma unroll 1
      for (int i = t; i < rows * 32; i += 128) {
        const int r = i >> 5, f4 = (i & 31) * 4;
        if (fb + f4 < p.d_model) {
          const float4 v = *reinterpret_cast<const float4*>(stage_t + r * 132 + f4);
          float* dst = p.y + (long long)(m0 + r) * p.d_model + fb + f4;
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v.x), "f"(v.y), "f"(v.z),
                       "f"(v.w)
                       : "memory");
        }
      }
      named_bar_sync(1, 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, K::TMEM_COLS);
  }
}

template <int NB>
size_t out_proj_latent_smem() {
  return OpLatCfg<NB>::NS * OpLatCfg<NB>::STAGE + sizeof(OpLatCtrl) + 1024;
}

template <int NB>
cudaError_t launch_lat_nb(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p, dim3 grid,
                          cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(out_proj_latent_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)out_proj_latent_smem<NB>());
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(out_proj_latent_kernel<NB>, grid, dim3(192), out_proj_latent_smem<NB>(), s, tm_w, tm_x, p);
}

}  // namespace

int out_proj_nb(int M) {
  const int r = M >= 256 ? 256 : ((M + 15) / 16) * 16;
  return r <= 32 ? 32 : (r <= 64 ? 64 : (r <= 128 ? 128 : 256));
}

cudaError_t launch_out_proj(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p, int num_sms,
                            cudaStream_t s) {
  const int NB = out_proj_nb(p.M);
  const int tiles = (p.d_model + 127) / 128, mblocks = (p.M + NB - 1) / NB;
  // about two CTAs per SM, each with at least four 64-column blocks (fewer
  // partials to add when the contraction is short)
  int KS = (2 * num_sms) / (tiles * mblocks);
  const int ks_max = p.KB / 4 > 1 ? p.KB / 4 : 1;
  KS = KS < 1 ? 1 : (KS > ks_max ? ks_max : KS);
  if (tiles * mblocks > OP_SYNC_TILES) KS = 1;   // a split tile needs its words
  const dim3 grid(tiles, KS, mblocks);
  switch (NB) {
    case 32: return launch_nb<32>(tm_w, tm_x, p, grid, s);
    case 64: return launch_nb<64>(tm_w, tm_x, p, grid, s);
    case 128: return launch_nb<128>(tm_w, tm_x, p, grid, s);
    default: return launch_nb<256>(tm_w, tm_x, p, grid, s);
  }
}

}  // namespace mla

namespace mla {

cudaError_t launch_absorb_w_o(const uint16_t* w_o, const uint16_t* w_uv, uint16_t* w_ov, int H, int d_model,
                              cudaStream_t s) {
  absorb_w_o_kernel<<<dim3(D_C / 64, d_model / 64, H), 256, 0, s>>>(w_o, w_uv, w_ov, H, d_model);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_latent(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const OutProjParams& p,
                                   int num_sms, cudaStream_t s) {
  const int NB = out_proj_nb(p.M);
  const int ft = NB <= 128 ? 4 : 1;   // OpLatCfg<NB>::FT
  const int cols = ((p.d_model + 127) / 128 + ft - 1) / ft, mblocks = (p.M + NB - 1) / NB;
  int KS = (2 * num_sms) / (cols * mblocks);
  const int ks_max = p.KB / 4 > 1 ? p.KB / 4 : 1;
  KS = KS < 1 ? 1 : (KS > ks_max ? ks_max : KS);
  const dim3 grid(cols, KS, mblocks);
  switch (NB) {
    case 32: return launch_lat_nb<32>(tm_w, tm_x, p, grid, s);
    case 64: return launch_lat_nb<64>(tm_w, tm_x, p, grid, s);
    case 128: return launch_lat_nb<128>(tm_w, tm_x, p, grid, s);
    default: return launch_lat_nb<256>(tm_w, tm_x, p, grid, s);
  }
}

}  // namespace mla
