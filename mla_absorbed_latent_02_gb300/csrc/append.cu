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
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {

// One warp per token: 64 x 16 B of latent, then 8 lanes rotate 4 pairs each.
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  const int tok = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (tok >= p.n) return;
  const int s = p.seq_idx[tok];
  const int t = p.pos[tok];
  long long row = -1;
  if (s >= 0 && s < p.num_seqs && t >= 0 && t < p.max_pos) {
    if (p.paged) {
      const int blk = t / PAGE;
      if (blk < p.max_blocks) {
        const int id = p.block_table[(long long)s * p.max_blocks + blk];
        if (id >= 0 && id < p.num_blocks) row = (long long)id * PAGE + (t % PAGE);
      }
    } else if (t < p.capacity) {
      row = (long long)s * p.capacity + t;
    }
  }
  if (row < 0) {
    if (lane == 0) atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(p.cache + row * ROW);
  const uint4* src = reinterpret_cast<const uint4*>(p.c_kv + (long long)tok * D_C);
  dst[lane] = src[lane];
  dst[lane + 32] = src[lane + 32];
  if (lane < 8) {
    const uint4 kr = reinterpret_cast<const uint4*>(p.k_rope + (long long)tok * D_ROPE)[lane];
    const float2* tab = p.rope + (long long)t * (D_ROPE / 2) + 4 * lane;
    const uint32_t in[4] = {kr.x, kr.y, kr.z, kr.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(in[i] << 16);
      const float b = __uint_as_float(in[i] & 0xFFFF0000u);
      const float2 cs = tab[i];
      const float y0 = __fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y));
      const float y1 = __fadd_rn(__fmul_rn(b, cs.x), __fmul_rn(a, cs.y));
      out[i] = pack_bf16x2(y0, y1);
    }
    dst[64 + lane] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (p.n + warps_per_block - 1) / warps_per_block;
  return launch_pdl(append_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, s, p);
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

}  // namespace mla
