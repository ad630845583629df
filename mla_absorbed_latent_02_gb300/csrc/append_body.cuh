// Per-token bodies of the cache append (bf16 and FP8 rows), shared by the append
// kernels and the fused append + absorb_q launch. Each runs on one warp: it
// reads the token's inputs (call inputs no kernel of this library writes)
// before the wait on the previous kernel of the stream and writes the cache row
// (which an attention call before it may still be reading) after it. The
// caller triggers its dependents.
#pragma once

#include <cuda_fp8.h>

#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {
// Cache row of token position t of sequence s, or -1 when it has none.
MLA_DEV long long cache_row(const AppendParams& p, int s, int t) {
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
  return row;
}

// The cache writer's RoPE contract for one interleaved pair (x0, x1) (bf16
// values) at angle index i of position t: float32 rotation with separately
// rounded products and sums against the float32 table, rounded to bf16.
MLA_DEV uint32_t rope_pair(const AppendParams& p, int t, int i, float x0, float x1) {
  const float2 cs = p.rope[(long long)t * (D_ROPE / 2) + i];
  const float y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
  const float y1 = __fadd_rn(__fmul_rn(x1, cs.x), __fmul_rn(x0, cs.y));
  return pack_bf16x2(y0, y1);
}

// bf16 row: 64 x 16 B of latent, then 8 lanes rotate 4 pairs each.
MLA_DEV void append_token(const AppendParams& p, int tok, int lane) {
  if (tok >= p.n) {
    pdl_wait();
    return;
  }
  const int s = p.seq_idx[tok];
  const int t = p.pos[tok];
  const long long row = cache_row(p, s, t);
  const uint4* src = reinterpret_cast<const uint4*>(p.c_kv + (long long)tok * D_C);
  const uint4 c0 = src[lane], c1 = src[lane + 32];
  uint4 kr = make_uint4(0, 0, 0, 0);
  if (lane < 8) kr = reinterpret_cast<const uint4*>(p.k_rope + (long long)tok * D_ROPE)[lane];
  pdl_wait();
  if (row < 0) {
    if (lane == 0) atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(p.cache + row * ROW);
  dst[lane] = c0;
  dst[lane + 32] = c1;
  if (lane < 8) {
    const uint32_t in[4] = {kr.x, kr.y, kr.z, kr.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      out[i] = rope_pair(p, t, 4 * lane + i, __uint_as_float(in[i] << 16), __uint_as_float(in[i] & 0xFFFF0000u));
    dst[64 + lane] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}


// FP8 row: lane j owns latent columns 16j ..
// 16j+15. The row's largest magnitude (a warp max) fixes the token's scale
// sigma = 2^e, the smallest power of two with amax / sigma <= 448 = 1.75 * 2^8
// (at least 2^-64); each c / sigma (an exact scaling) is rounded to the nearest
// e4m3 code (ties to even). The RoPE key is rotated and rounded exactly as the
// bf16 cache stores it, then sigma and 12 zero bytes end the row.
MLA_DEV void append_token_fp8(const AppendParams& p, int tok, int lane) {
  if (tok >= p.n) {
    pdl_wait();
    return;
  }
  const int s = p.seq_idx[tok];
  const int t = p.pos[tok];
  const long long row = cache_row(p, s, t);
  const uint4* src = reinterpret_cast<const uint4*>(p.c_kv + (long long)tok * D_C + 16 * lane);
  const uint4 c0 = src[0], c1 = src[1];
  uint4 kr = make_uint4(0, 0, 0, 0);
  if (lane < 8) kr = reinterpret_cast<const uint4*>(p.k_rope + (long long)tok * D_ROPE)[lane];
  pdl_wait();
  if (row < 0) {
    if (lane == 0) atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return;
  }
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // amax = m * 2^k (1 <= m < 2): e = k - 8, or k - 7 when m > 1.75
  const uint32_t ab = __float_as_uint(amax);
  const int ef = static_cast<int>(ab >> 23);
  int e = ef == 0 ? FP8_SCALE_EXP_MIN : ef - 127 - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = max(e, FP8_SCALE_EXP_MIN);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * inv, v[4 * i + 1] * inv), __NV_SATFINITE,
                                                 __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv),
                                                 __NV_SATFINITE, __NV_E4M3);
    q[i] = lo | (hi << 16);
  }
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.cache) + row * ROW8;
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
  if (lane < 8) {
    const uint32_t in[4] = {kr.x, kr.y, kr.z, kr.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      out[i] = rope_pair(p, t, 4 * lane + i, __uint_as_float(in[i] << 16), __uint_as_float(in[i] & 0xFFFF0000u));
    reinterpret_cast<uint4*>(dst + ROW8_ROPE)[lane] = make_uint4(out[0], out[1], out[2], out[3]);
  } else if (lane == 8) {
    reinterpret_cast<uint4*>(dst + ROW8_SCALE)[0] = make_uint4(static_cast<uint32_t>(127 + e) << 23, 0, 0, 0);
  }
}

// Latent producer, last step for one token (one warp): c holds the token's 16
// projected latent values 16*lane .. 16*lane+15 and kr its raw RoPE-key pair
// `lane` (float32). Optional RMSNorm of the 512 latent values
// (c / sqrt(mean(c^2) + eps) * kv_norm, float32), rounding to bf16, and the RoPE
// key rounded to bf16 then rotated by the cache writer's contract; the row goes
// to (seq_idx[tok], pos[tok]) with the append addressing (out-of-cache rows set
// MLA_DEVERR_BOUNDS and are skipped).
MLA_DEV void finish_latent_row(const AppendParams& p, int tok, int lane, float (&c)[16], float2 kr,
                               const uint16_t* kv_norm, float eps) {
  const int s = p.seq_idx[tok];
  const int t = p.pos[tok];
  const long long row = cache_row(p, s, t);
  if (row < 0) {
    if (lane == 0) atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return;
  }
  if (kv_norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = __fmaf_rn(c[i], c[i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rms = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, 512.f), eps));
    const uint4* gw = reinterpret_cast<const uint4*>(kv_norm + 16 * lane);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 g = gw[i];
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        c[8 * i + 2 * j] = __fdiv_rn(c[8 * i + 2 * j], rms) * __uint_as_float(gv[j] << 16);
        c[8 * i + 2 * j + 1] = __fdiv_rn(c[8 * i + 2 * j + 1], rms) * __uint_as_float(gv[j] & 0xFFFF0000u);
      }
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(p.cache + row * ROW);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    dst[2 * lane + i] = make_uint4(pack_bf16x2(c[8 * i], c[8 * i + 1]), pack_bf16x2(c[8 * i + 2], c[8 * i + 3]),
                                   pack_bf16x2(c[8 * i + 4], c[8 * i + 5]), pack_bf16x2(c[8 * i + 6], c[8 * i + 7]));
  // RoPE key: pair `lane`, its raw values rounded to bf16 first (the contract's input)
  const uint32_t raw = pack_bf16x2(kr.x, kr.y);
  reinterpret_cast<uint32_t*>(p.cache + row * ROW + D_C)[lane] =
      rope_pair(p, t, lane, __uint_as_float(raw << 16), __uint_as_float(raw & 0xFFFF0000u));
}

}  // namespace mla
