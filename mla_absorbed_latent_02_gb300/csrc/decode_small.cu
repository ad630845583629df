// The whole absorbed decode step for short sequences in one launch: append the
// new token, absorb the query, attend over the latent cache and expand the
// result ("DeepSeek MLA 吸收式缓存" §2.2-§2.4; "80 行 PyTorch 从零写 DeepSeek 的 MLA"
// §4-§5), for the latency-bound case (a handful of sequences of at most a few
// thousand tokens, e.g. the V2-Lite single step of 26 tokens), where the four
// calls of the general path cost four dependent kernel launches.
//
// A cluster of four CTAs serves one (sequence b, head h); CTA j owns latent
// columns 128j .. 128j+127. Everything is a matrix-vector product at this size,
// so it runs on CUDA cores in fp32:
//   q_lat[c]  = sum_d W_UK[h][d][c] q_nope[d]                 (own columns)
//   s_t       = q_lat . c_t + RoPE(q_rope) . k_rope_t         (partial per CTA,
//               the RoPE part in CTA 0; the four partials added through
//               distributed shared memory in a fixed order)
//   p         = softmax(scale s),  o_lat[c] = sum_t p_t c_t[c]  (own columns)
//   o[v]      = sum_c W_UV[h][v][c] o_lat[c]                  (partial per CTA,
//               added through distributed shared memory)
// The new token (position L_b - 1) is taken from the call's inputs, rotated by
// the cache writer's contract, and written to the cache by the cluster of head
// 0; no CTA reads it back from the cache in this launch.
#include "append_body.cuh"
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase stamps (compile with -DMLA_TRACE=1): globaltimer at eight
// points of each CTA, read back with mla_trace_read_small().
#if MLA_TRACE
__device__ unsigned long long g_small_trace[512][8];
#define SM_STAMP(ev)                                                                           \
  do {                                                                                         \
    const unsigned c_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);        \
    if (threadIdx.x == 0 && c_ < 512) g_small_trace[c_][(ev)] = mla::globaltimer();            \
  } while (0)
extern "C" int mla_trace_read_small(void* host, size_t bytes) {
  if (bytes > sizeof(g_small_trace)) bytes = sizeof(g_small_trace);
  return (int)cudaMemcpyFromSymbol(host, g_small_trace, bytes);
}
#else
#define SM_STAMP(ev) \
  do {               \
  } while (0)
#endif

namespace mla {

namespace {

constexpr int SM_COLS = D_C / 4;   // latent columns per CTA
constexpr int SM_PAD = 8;          // bf16 of padding per weight row in shared memory
constexpr int RC_TOK = 128;        // tokens whose rows are staged in shared memory at a time

struct __align__(16) SmallSmem {
  alignas(16) uint16_t wuk[D_NOPE][SM_COLS + SM_PAD];   // W_UK[h][d][own columns]
  alignas(16) uint16_t wuv[D_V][SM_COLS + SM_PAD];      // W_UV[h][v][own columns]
  alignas(16) float q[D_NOPE];                          // q_nope
  alignas(16) float qr[D_ROPE];                         // RoPE'd q_rope (bf16 values)
  alignas(16) float ql[SM_COLS];                        // q_lat, own columns
  alignas(16) float ol[SM_COLS];                        // o_lat, own columns
  alignas(16) float cn[SM_COLS];                        // the new token's latent, own columns
  alignas(16) float kn[D_ROPE];                         // the new token's RoPE'd key (bf16 values)
  alignas(16) float op[D_V];                            // partial o
  alignas(16) float red[2][4];
  alignas(16) uint16_t rc[RC_TOK][SM_COLS + 4];         // staged rows, own columns (bf16; 8-byte rows)
  alignas(16) uint16_t rk[RC_TOK][D_ROPE + 2];          // staged RoPE keys (CTA 0)
  alignas(16) float s[SMALL_MAX_LEN];                   // partial scores (read by the cluster)
  alignas(16) float pr[SMALL_MAX_LEN];                  // scores, then weights
};

MLA_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

MLA_DEV float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

MLA_DEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
MLA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MLA_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

MLA_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
MLA_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Reductions over the CTA's 128 threads.
MLA_DEV float block_max(float v, SmallSmem& sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sm.red[0][threadIdx.x >> 5] = v;
  __syncthreads();
  const float r = fmaxf(fmaxf(sm.red[0][0], sm.red[0][1]), fmaxf(sm.red[0][2], sm.red[0][3]));
  __syncthreads();
  return r;
}
MLA_DEV float block_sum(float v, SmallSmem& sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sm.red[1][threadIdx.x >> 5] = v;
  __syncthreads();
  const float r = (sm.red[1][0] + sm.red[1][1]) + (sm.red[1][2] + sm.red[1][3]);
  __syncthreads();
  return r;
}

__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(128) decode_small_kernel(SmallStepParams p) {
  extern __shared__ uint8_t smem_raw[];
  SmallSmem& sm = *reinterpret_cast<SmallSmem*>(smem_raw);
  const int j = static_cast<int>(cluster_rank());
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const AppendParams& a = p.a;
  const int c0 = j * SM_COLS;
  SM_STAMP(0);
  pdl_trigger();

  // call inputs (weights, queries, the new token, lengths): before the wait.
  // The weight slices go straight to shared memory (cp.async, 16 bytes each,
  // every copy in flight at once): W_UK in one group, W_UV in a second one that
  // is only waited for before the last product.
  {
    const uint4* wk = reinterpret_cast<const uint4*>(p.w_uk + (long long)h * D_NOPE * D_C + c0);
    const uint4* wv = reinterpret_cast<const uint4*>(p.w_uv + (long long)h * D_V * D_C + c0);
#pragma unroll
    for (int i = tid; i < D_NOPE * SM_COLS / 8; i += 128) {
      const int r = i >> 4, ch = i & 15;
      cp_async16(smem_u32(&sm.wuk[r][8 * ch]), wk + (long long)r * (D_C / 8) + ch);
    }
    cp_async_commit();
#pragma unroll
    for (int i = tid; i < D_V * SM_COLS / 8; i += 128) {
      const int r = i >> 4, ch = i & 15;
      cp_async16(smem_u32(&sm.wuv[r][8 * ch]), wv + (long long)r * (D_C / 8) + ch);
    }
    cp_async_commit();
  }
  const int L = p.seq_lens[b];
  const bool len_ok = L >= 1 && L <= SMALL_MAX_LEN && L - 1 < a.max_pos;
  {
    const uint16_t* qn = p.q_nope + ((long long)b * p.H + h) * D_NOPE;
    sm.q[tid] = __uint_as_float(static_cast<uint32_t>(qn[tid]) << 16);
    sm.cn[tid] = __uint_as_float(static_cast<uint32_t>(a.c_kv[(long long)b * D_C + c0 + tid]) << 16);
    if (tid < D_ROPE / 2 && len_ok) {
      // RoPE of the query and of the new key at position L - 1 (the cache
      // writer's float32 contract, rounded to bf16)
      const uint32_t qw = reinterpret_cast<const uint32_t*>(p.q_rope + ((long long)b * p.H + h) * D_ROPE)[tid];
      const uint32_t kw = reinterpret_cast<const uint32_t*>(a.k_rope + (long long)b * D_ROPE)[tid];
      const uint32_t qrot = rope_pair(a, L - 1, tid, bf16_lo(qw), bf16_hi(qw));
      const uint32_t krot = rope_pair(a, L - 1, tid, bf16_lo(kw), bf16_hi(kw));
      sm.qr[2 * tid] = bf16_lo(qrot);
      sm.qr[2 * tid + 1] = bf16_hi(qrot);
      sm.kn[2 * tid] = bf16_lo(krot);
      sm.kn[2 * tid + 1] = bf16_hi(krot);
    }
  }
  cp_async_wait<1>();   // this thread's W_UK copies
  __syncthreads();
  // q_lat, own columns (thread = column), fixed order over d
  {
    float acc = 0.f;
#pragma unroll 8
    for (int d = 0; d < D_NOPE; ++d) acc = fmaf(bf16_lo(sm.wuk[d][tid]), sm.q[d], acc);
    sm.ql[tid] = acc;
  }
  SM_STAMP(1);
  pdl_wait();   // the cache rows of earlier steps may come from the previous kernel
  __syncthreads();
  SM_STAMP(2);

  if (!len_ok) {
    cp_async_wait<0>();
    // length out of range for this path: no attention is defined here
    for (int c = tid; c < SM_COLS; c += 128) p.o_lat[((long long)b * p.H + h) * D_C + c0 + c] = 0.f;
    if (j == 0 && tid < D_V) p.out[((long long)b * p.H + h) * D_V + tid] = 0;
    if (j == 0 && tid == 0) {
      p.lse[(long long)b * p.H + h] = -INFINITY;
      atomicOr(a.status, L < 1 || L > SMALL_MAX_LEN ? MLA_DEVERR_LENGTH : MLA_DEVERR_BOUNDS);
    }
    return;   // the whole cluster (one sequence) takes this path; no shared memory is read remotely
  }

  // Tokens are taken in chunks of RC_TOK: each chunk's own-column slice of
  // the cached rows (and, in CTA 0, its RoPE keys) is staged in shared memory
  // by coalesced warp loads (a token row per warp, sixteen in flight), then
  // used by thread-per-token dot products (scores) and, after the softmax,
  // thread-per-column sums (o_lat). Sequences of at most RC_TOK tokens stage
  // their rows once; longer ones stage each chunk again for o_lat.
  const int nold = L - 1;   // cached tokens; the new one (position L - 1) comes from cn / kn
  auto stage = [&](int base) {
    const int n = min(RC_TOK, nold - base);
#pragma unroll 1
    for (int t0 = warp; t0 < n; t0 += 4 * 16) {
      uint2 cw[16];
      uint32_t kw[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = t0 + 4 * u;
        cw[u] = make_uint2(0, 0);
        kw[u] = 0;
        if (t < n) {
          const long long row = cache_row(a, b, base + t);
          if (row >= 0) {
            const uint16_t* r = a.cache + row * ROW;
            cw[u] = *reinterpret_cast<const uint2*>(r + c0 + 4 * lane);
            if (j == 0) kw[u] = reinterpret_cast<const uint32_t*>(r + D_C)[lane];
          } else if (lane == 0) {
            atomicOr(a.status, MLA_DEVERR_BOUNDS);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int t = t0 + 4 * u;
        if (t < n) {
          *reinterpret_cast<uint2*>(&sm.rc[t][4 * lane]) = cw[u];
          if (j == 0) *reinterpret_cast<uint32_t*>(&sm.rk[t][2 * lane]) = kw[u];
        }
      }
    }
  };
  // partial scores, thread = token
#pragma unroll 1
  for (int base = 0; base < nold; base += RC_TOK) {
    stage(base);
    __syncthreads();
    const int t = base + tid;
    if (tid < RC_TOK && t < nold) {
      float v = 0.f;
#pragma unroll 8
      for (int c = 0; c < SM_COLS; c += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(&sm.rc[tid][c]);
        v = fmaf(sm.ql[c], bf16_lo(w), v);
        v = fmaf(sm.ql[c + 1], bf16_hi(w), v);
      }
      if (j == 0) {
#pragma unroll 8
        for (int i = 0; i < D_ROPE; i += 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(&sm.rk[tid][i]);
          v = fmaf(sm.qr[i], bf16_lo(w), v);
          v = fmaf(sm.qr[i + 1], bf16_hi(w), v);
        }
      }
      sm.s[t] = v;
    }
    __syncthreads();
  }
  if (warp == 0) {
    // the new token, from the call's inputs (lane: 4 own columns, one RoPE pair)
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) v = fmaf(sm.ql[4 * lane + i], sm.cn[4 * lane + i], v);
    if (j == 0) v = fmaf(sm.qr[2 * lane], sm.kn[2 * lane], fmaf(sm.qr[2 * lane + 1], sm.kn[2 * lane + 1], v));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sm.s[L - 1] = v;
  }
  SM_STAMP(3);
  cluster_sync();
  SM_STAMP(4);
  // full scores: the four partials in cluster rank order (identical in every CTA)
  {
    const uint32_t s_addr = smem_u32(sm.s);
    float mx = -INFINITY;
    for (int t = tid; t < L; t += 128) {
      float v = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) v += ld_cluster_f32(mapa_shared(s_addr + 4u * t, r));
      v *= p.scale;
      sm.pr[t] = v;
      mx = fmaxf(mx, v);
    }
    mx = block_max(mx, sm);
    float sum = 0.f;
    for (int t = tid; t < L; t += 128) {
      const float e = __expf(sm.pr[t] - mx);
      sm.pr[t] = e;
      sum += e;
    }
    sum = block_sum(sum, sm);
    if (j == 0 && tid == 0) p.lse[(long long)b * p.H + h] = mx + __logf(sum);
    // o_lat, own columns (thread = column), tokens in order
    float acc = 0.f;
#pragma unroll 1
    for (int base = 0; base < nold; base += RC_TOK) {
      if (nold > RC_TOK) {   // the chunk's rows are no longer staged
        __syncthreads();
        stage(base);
        __syncthreads();
      }
      const int n = min(RC_TOK, nold - base);
#pragma unroll 4
      for (int t = 0; t < n; ++t) acc = fmaf(sm.pr[base + t], bf16_lo(sm.rc[t][tid]), acc);
    }
    acc = fmaf(sm.pr[L - 1], sm.cn[tid], acc);
    const float ol = acc * (1.f / sum);
    sm.ol[tid] = ol;
    p.o_lat[((long long)b * p.H + h) * D_C + c0 + tid] = ol;
  }
  SM_STAMP(5);
  cp_async_wait<0>();   // this thread's W_UV copies
  __syncthreads();
  // partial o = W_UV[h][:, own columns] o_lat[own columns], thread = output v
  {
    float x = 0.f;
#pragma unroll 4
    for (int c = 0; c < SM_COLS; c += 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(&sm.wuv[tid][c]);
      x = fmaf(sm.ol[c], bf16_lo(w.x), x);
      x = fmaf(sm.ol[c + 1], bf16_hi(w.x), x);
      x = fmaf(sm.ol[c + 2], bf16_lo(w.y), x);
      x = fmaf(sm.ol[c + 3], bf16_hi(w.y), x);
      x = fmaf(sm.ol[c + 4], bf16_lo(w.z), x);
      x = fmaf(sm.ol[c + 5], bf16_hi(w.z), x);
      x = fmaf(sm.ol[c + 6], bf16_lo(w.w), x);
      x = fmaf(sm.ol[c + 7], bf16_hi(w.w), x);
    }
    sm.op[tid] = x;
  }
  SM_STAMP(6);
  cluster_sync();
  if (tid < 32) {
    // o[v], v = 32j + tid: the four partials in cluster rank order, bf16 out
    const int v = 32 * j + tid;
    const uint32_t op_addr = smem_u32(sm.op) + 4u * v;
    float x = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) x += ld_cluster_f32(mapa_shared(op_addr, r));
    p.out[((long long)b * p.H + h) * D_V + v] = static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
  }
  if (h == 0 && warp == 1) {
    // the new token's cache row, own columns; CTA 0 also writes the RoPE key
    const long long row = cache_row(a, b, L - 1);
    if (row < 0) {
      if (lane == 0) atomicOr(a.status, MLA_DEVERR_BOUNDS);
    } else {
      uint16_t* dst = a.cache + row * ROW;
      reinterpret_cast<uint2*>(dst + c0)[lane] =
          reinterpret_cast<const uint2*>(a.c_kv + (long long)b * D_C + c0)[lane];
      if (j == 0)
        reinterpret_cast<uint32_t*>(dst + D_C)[lane] = pack_bf16x2(sm.kn[2 * lane], sm.kn[2 * lane + 1]);
    }
  }
  cluster_sync();   // no CTA leaves while the cluster still reads its shared memory
  SM_STAMP(7);
}

}  // namespace

size_t small_step_smem_bytes() { return sizeof(SmallSmem); }

cudaError_t launch_small_step(const SmallStepParams& p, int B, cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(decode_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(SmallSmem));
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_small_kernel, dim3(4, p.H, B), dim3(128), sizeof(SmallSmem), s, p);
}

}  // namespace mla
