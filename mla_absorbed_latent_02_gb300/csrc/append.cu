// Cache append: one 576-element bf16 row per token,
//   row = [ c_kv (512, copied verbatim) | RoPE_pos(k_rope) (64) ].
// The shared latent plus the decoupled 64-dim RoPE key is the whole per-token
// state of absorbed MLA ("DeepSeek MLA 吸收式缓存" §2.4 and §4.1; the
// cache-concat step of "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2).
//
// RoPE pairs are interleaved (x[2i], x[2i+1]) with inverse frequency
// 1/base^(2i/64) ("80 行 PyTorch 从零写 DeepSeek 的 MLA", Appendix A). The
// rotation is done in float32 with separately rounded multiplies and adds
// (no FMA) against a host-built float32 cos/sin table, then rounded to bf16
// (nearest even), so the stored bytes are reproducible.
#include "append_body.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {

// One warp per token (the bodies: append_body.cuh).
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  pdl_trigger();
  append_token(p, (blockIdx.x * blockDim.x + threadIdx.x) >> 5, threadIdx.x & 31);
}

__global__ void __launch_bounds__(256) append_fp8_kernel(AppendParams p) {
  pdl_trigger();
  append_token_fp8(p, (blockIdx.x * blockDim.x + threadIdx.x) >> 5, threadIdx.x & 31);
}

// Latent producer, second half: y [n, 576] fp32 holds W_KV_A h of each new token
// (latent | RoPE key). One warp per token: optional RMSNorm of the 512 latent
// values (lane j owns columns 16j .. 16j+15), rounding to bf16, then the RoPE key
// rounded to bf16 and rotated by the cache writer's contract (lane i owns pair i).
__global__ void __launch_bounds__(256) latent_finish_kernel(LatentFinishParams q) {
  const AppendParams& p = q.a;
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (tok >= p.n) return;
  const float* y = q.y + (long long)tok * ROW;
  float c[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = reinterpret_cast<const float4*>(y + 16 * lane)[i];
    c[4 * i] = v.x;
    c[4 * i + 1] = v.y;
    c[4 * i + 2] = v.z;
    c[4 * i + 3] = v.w;
  }
  finish_latent_row(p, tok, lane, c, reinterpret_cast<const float2*>(y + D_C)[lane], q.kv_norm, q.eps);
}

cudaError_t launch_latent_finish(const LatentFinishParams& q, cudaStream_t s) {
  if (q.a.n <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (q.a.n + warps_per_block - 1) / warps_per_block;
  return launch_pdl(latent_finish_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, s, q);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (p.n + warps_per_block - 1) / warps_per_block;
  return launch_pdl(append_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, s, p);
}

cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (p.n + warps_per_block - 1) / warps_per_block;
  return launch_pdl(append_fp8_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, s, p);
}

// Bounded-wait probe: waits on an mbarrier that nothing completes. Used by the
// tests to check that a wait that runs out reports MLA_DEVERR_TIMEOUT and the
// context stays usable.
__global__ void wait_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    if (!mbar_wait_ns(smem_u32(&bar), 0, limit_ns)) atomicOr(status, MLA_DEVERR_TIMEOUT);
    mbar_arrive(smem_u32(&bar));  // leave the barrier in a completed phase
  }
}

cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

// n16 16-byte words from src to dst; either side may be pinned host memory that
// the device addresses directly. Launched as a plain kernel (no programmatic
// dependent launch on either side): it starts after the previous kernel in the
// stream has completed, and the next kernel starts only after every word has
// landed, so a kernel that reads the copied data early (before its own
// dependency wait) still sees it.
__global__ void __launch_bounds__(256) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                   size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // four loads in flight per thread: the host link's latency is paid once
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, int num_sms, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  size_t blocks = (n16 + 255) / 256;
  const size_t cap = static_cast<size_t>(num_sms) * 4;
  if (blocks > cap) blocks = cap;
  copy_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<uint4*>(dst),
                                                            static_cast<const uint4*>(src), n16);
  return cudaGetLastError();
}

}  // namespace mla
