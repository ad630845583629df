// Latent producer in one launch: the new tokens' cache rows from their hidden
// states ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §2, Wdkv / Wkr; "DeepSeek-V2-Lite
// 真实权重执行审计" §3.3, kv_a_proj_with_mqa and kv_a_layernorm; "DeepSeek MLA
// 吸收式缓存" §2.4, the 576-element cached row):
//   y = W_KV_A h                          (576 <- d_model, fp32 accumulation)
//   row = [ bf16(RMSNorm(y[0:512])) | RoPE_pos(bf16(y[512:576])) ]
//
// A decode step projects few tokens (n = B) through a long contraction
// (d_model = 2048 or 7168), so the weight (2.4 or 8.3 MB) is spread over the
// whole GPU by splitting K, as in the output projection. One cooperative launch,
// two phases separated by a grid-wide barrier:
//  1. CTA (f, s, mb): output features 128f .. 128f+127 (five tiles cover the
//     576; the last reads zeros past row 575), K-blocks s*KB/S .. (s+1)*KB/S of
//     64 columns, token rows of block mb. tcgen05 MMA with tokens on N ("swap
//     AB": D^T[feature x token] = W tile . h^T), four-stage TMA ring. The fp32
//     partial goes to its own slot ws[s][token][feature] of the workspace: no
//     zero-fill and no atomics, and the sum in phase 2 has a fixed order.
//  2. after the barrier, one CTA per token adds the S partials of each feature
//     in order (eight splits' loads in flight at a time) and one warp finishes the row
//     (RMSNorm, bf16, RoPE contract, cache write).
// The barrier counts arrivals on one word of the context (its top bit flips
// once every CTA has arrived); every wait is bounded (MLA_DEVERR_TIMEOUT,
// phase 2 skipped). Cooperative launch keeps every CTA resident, so the barrier
// cannot wait for a CTA that never runs. The launch also allows programmatic
// dependent launch: weight tiles load before the wait on the previous kernel,
// the hidden states and every workspace write after it.
#include "append_body.cuh"
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase stamps (compile with -DMLA_TRACE=1): globaltimer at the
// start, before the barrier, after it and at the end of each CTA.
#if MLA_TRACE
__device__ unsigned long long g_lp_trace[256][4];
#define LP_STAMP(ev)                                                                                        \
  do {                                                                                                      \
    const unsigned c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);                     \
    if (threadIdx.x == 0 && c_ < 256) g_lp_trace[c_][(ev)] = mla::globaltimer();                            \
  } while (0)
extern "C" int mla_trace_read_lp(void* host, size_t bytes) {
  if (bytes > sizeof(g_lp_trace)) bytes = sizeof(g_lp_trace);
  return (int)cudaMemcpyFromSymbol(host, g_lp_trace, bytes);
}
#else
#define LP_STAMP(ev) \
  do {               \
  } while (0)
#endif

namespace mla {

namespace {

constexpr int LP_NS = 4;                    // TMA stages
constexpr uint32_t LP_A_BYTES = 16384;      // W_KV_A tile: 128 features x 64 columns

struct __align__(8) LpCtrl {
  uint64_t full[LP_NS], empty[LP_NS], done;
  uint32_t tmem_base;
  int abort;
};

MLA_DEV uint8_t* lp_align1k(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

MLA_DEV unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

MLA_DEV unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of all CTAs (called by every thread). One word counts the
// arrivals: CTA 0 adds 2^31 - (CTAs - 1) and every other CTA adds 1, so each
// round adds exactly 2^31 and flips the top bit, which is what the CTAs wait
// for; the low bits come back to where they were, so the word needs no reset.
// Thread 0 of each CTA fences (the CTA's writes, ordered before it by the CTA
// barrier) before its arrival and after it sees the flip. Returns false when it
// gave up waiting (status set).
MLA_DEV bool grid_barrier(unsigned* word, int* status) {
  __syncthreads();
  __shared__ int ok_s;
  if (threadIdx.x == 0) {
    const unsigned nctas = gridDim.x * gridDim.y * gridDim.z;
    const bool first = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
    __threadfence();
    const unsigned old = atomicAdd(word, first ? 0x80000000u - (nctas - 1) : 1u);
    int ok = 1;
    const uint64_t t0 = globaltimer();
    while (((old ^ ld_relaxed_gpu(word)) & 0x80000000u) == 0) {
      if (globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
        atomicOr(status, MLA_DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

template <int NB>
__global__ void __launch_bounds__(192, 1) latent_proj_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                             const __grid_constant__ CUtensorMap tm_x,
                                                             LatentProjParams q) {
  LP_STAMP(0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = lp_align1k(smem_raw);
  constexpr uint32_t B_BYTES = 128u * NB;  // NB token rows x 64 columns x 2 bytes
  constexpr uint32_t STAGE = LP_A_BYTES + B_BYTES;
  LpCtrl* ctl = reinterpret_cast<LpCtrl*>(smem + LP_NS * STAGE);
  volatile int* abort = &ctl->abort;
  const AppendParams& a = q.fin.a;

  const int f0 = blockIdx.x * 128;
  const int s = blockIdx.y;
  const int m0 = blockIdx.z * NB;
  const int kb0 = static_cast<int>((long long)s * q.KB / gridDim.y);
  const int kb1 = static_cast<int>((long long)(s + 1) * q.KB / gridDim.y);
  const int nkb = kb1 - kb0;               // >= 1: the launcher keeps S <= KB
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t TMEM_COLS = NB <= 32 ? 32u : (NB <= 64 ? 64u : (NB <= 128 ? 128u : 256u));

  if (threadIdx.x == 0) {
    for (int i = 0; i < LP_NS; ++i) {
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

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      // weight tiles (a call input) of the first stages before the wait on the
      // previous kernel of the stream, the hidden states after it
      for (int i = 0; i < nkb && i < LP_NS; ++i) {
        const uint32_t f = smem_u32(&ctl->full[i]);
        mbar_arrive_expect_tx(f, LP_A_BYTES + 128u * q.rows_box);
        tma_load_2d(smem_u32(smem + i * STAGE), &tm_w, f, 64 * (kb0 + i), f0);
      }
      pdl_wait();
      for (int i = 0; i < nkb; ++i) {
        const int st = i % LP_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        uint8_t* stage = smem + st * STAGE;
        if (i >= LP_NS) {
          if (!mbar_wait(smem_u32(&ctl->empty[st]), ((i / LP_NS) & 1) ^ 1, abort, a.status)) break;
          mbar_arrive_expect_tx(f, LP_A_BYTES + 128u * q.rows_box);
          tma_load_2d(smem_u32(stage), &tm_w, f, 64 * (kb0 + i), f0);
        }
        tma_load_2d(smem_u32(stage + LP_A_BYTES), &tm_x, f, 64 * (kb0 + i), m0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NB, 0, 0);
      bool good = true;
      for (int i = 0; i < nkb && good; ++i) {
        const int st = i % LP_NS;
        if (!(good = mbar_wait(smem_u32(&ctl->full[st]), (i / LP_NS) & 1, abort, a.status))) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + st * STAGE), sb = sa + LP_A_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, smem_desc(sa + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                      smem_desc(sb + 32 * k, 16, 1024, SMEM_SWIZZLE_128B), idesc, (i | k) != 0);
        mma_commit(smem_u32(&ctl->empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    // partial D^T[feature x token] -> ws[s][token][feature]: thread <-> feature
    // 32*(warp%4) + lane (its TMEM lane), 16 tokens per TMEM load; for each token
    // a warp stores 32 consecutive floats
    const int fq = warp & 3;
    const int fl = fq * 32 + lane;
    pdl_wait();   // the previous call may still read the workspace
    ok = mbar_wait(smem_u32(&ctl->done), 0, abort, a.status);
    tc_fence_after();
    if (ok) {
      const int rows = min(NB, a.n - m0);
      float* base = q.ws + ((long long)s * a.n + m0) * ROW + f0 + fl;
      const bool feat = f0 + fl < ROW;
#pragma unroll 1
      for (int c0 = 0; c0 < NB && c0 < rows; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(fq * 32) << 16) + c0, v);
        tmem_wait_ld();
        reg_fence16(v);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (feat && c0 + c < rows) __stcg(base + (long long)(c0 + c) * ROW, __uint_as_float(v[c]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (*abort) ok = false;
  const unsigned nctas = gridDim.x * gridDim.y * gridDim.z;
  LP_STAMP(1);
  if (!grid_barrier(q.sync, a.status) || !ok) return;
  LP_STAMP(2);

  // phase 2: one CTA per token; thread t adds the S partials of features
  // 4t .. 4t+3 in order (float4 loads, eight splits in flight at a time), then
  // warp 0 finishes the row from shared memory
  const int S = gridDim.y;
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  float* yrow = reinterpret_cast<float*>(smem);   // the TMA ring is free now
  for (int tok = cta; tok < a.n; tok += nctas) {
    if (threadIdx.x < ROW / 4) {
      const float4* src = reinterpret_cast<const float4*>(q.ws + (long long)tok * ROW) + threadIdx.x;
      const long long step = (long long)a.n * ROW / 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int k0 = 0; k0 < S; k0 += 8) {
        float4 part[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          part[k] = k0 + k < S ? __ldcg(src + (k0 + k) * step) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc.x += part[k].x;
          acc.y += part[k].y;
          acc.z += part[k].z;
          acc.w += part[k].w;
        }
      }
      reinterpret_cast<float4*>(yrow)[threadIdx.x] = acc;
    }
    __syncthreads();
    if (warp == 0) {
      float c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = yrow[16 * lane + i];
      finish_latent_row(a, tok, lane, c, make_float2(yrow[D_C + 2 * lane], yrow[D_C + 2 * lane + 1]), q.fin.kv_norm,
                        q.fin.eps);
    }
    __syncthreads();
  }
  LP_STAMP(3);
}

template <int NB>
size_t lp_smem() {
  return LP_NS * (LP_A_BYTES + 128u * NB) + sizeof(LpCtrl) + 1024;
}

template <int NB>
cudaError_t lp_launch_nb(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const LatentProjParams& q, dim3 grid,
                         cudaStream_t st) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(latent_proj_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)lp_smem<NB>());
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = lp_smem<NB>();
  cfg.stream = st;
  cudaLaunchAttribute attr1[2];
  attr1[0].id = cudaLaunchAttributeCooperative;
  attr1[0].val.cooperative = 1;
  attr1[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr1[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, latent_proj_kernel<NB>, tm_w, tm_x, q);
}

}  // namespace

int latent_proj_splits(int n, int KB, int num_sms) {
  const int NB = out_proj_nb(n);
  const int mblocks = (n + NB - 1) / NB;
  if (LP_FEATURE_TILES * mblocks > num_sms) return 0;   // too many token blocks to keep resident
  int S = num_sms / (LP_FEATURE_TILES * mblocks);
  const int cap = LP_MAX_SPLITS / mblocks;
  if (S > cap) S = cap;
  if (S > KB) S = KB;
  return S < 1 ? 1 : S;
}

cudaError_t launch_latent_proj(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const LatentProjParams& q,
                               cudaStream_t st) {
  const int NB = out_proj_nb(q.fin.a.n);
  const dim3 grid(LP_FEATURE_TILES, q.S, (q.fin.a.n + NB - 1) / NB);
  switch (NB) {
    case 32: return lp_launch_nb<32>(tm_w, tm_x, q, grid, st);
    case 64: return lp_launch_nb<64>(tm_w, tm_x, q, grid, st);
    case 128: return lp_launch_nb<128>(tm_w, tm_x, q, grid, st);
    default: return lp_launch_nb<256>(tm_w, tm_x, q, grid, st);
  }
}

}  // namespace mla
