// Prefill of long prompt chunks in the expanded (MHA) form.
//
// The absorbed form ("DeepSeek MLA 吸收式缓存" §2.2-2.3) attends in the 576-wide
// latent space: 2*H*(576+512) flops per (query, key) pair. For a chunk of T new
// tokens the naive form ("80 行 PyTorch 从零写 DeepSeek 的 MLA" §2, §3: keys and
// values expanded per head, k = [W_UK c ; RoPE(k_rope)], v = W_UV c) costs
// 2*H*(192+128) flops per pair after expanding each cached token once
// (2*H*256*512 flops per key), so it wins once a key is seen by a few hundred
// queries: FlashMLA ships its dense prefill in this MHA mode ("DeepSeek MLA
// 吸收式缓存" §6.1). Two launches:
//
//  expand_kv_kernel   kv[b, t, :] = [W_UK c_t | W_UV c_t] for every cached token
//                     (all heads; bf16 out, fp32 accumulation): a tcgen05 GEMM
//                     with tokens on M (128-token tiles read from the latent
//                     cache, contiguous or paged) and 256 weight rows on N. Rows
//                     from the sequence end to the end of its last 128-token tile
//                     are written as zeros, so that masked keys carry no garbage
//                     into P.V. The epilogue warps, idle during the products,
//                     first rotate the queries' RoPE part (the float32 contract
//                     of the cache writer and absorb_q) into q_rot.
//  mha_prefill_kernel causal softmax attention of one 128-query tile of one head
//                     per CTA: S = Q K^T over K = 192 (Q = [q_nope | q_rot],
//                     K = [K_nope | the cached RoPE key]) into tensor memory
//                     (two buffers), fp32 online softmax with a lazy rescale of
//                     O, P in bf16, O += P V (V MN-major) in tensor memory, then
//                     O / l rounded to bf16. Query j of a sequence sits at
//                     position L - T + j and sees keys 0 .. L - T + j (bottom-right
//                     causal, as the absorbed path).
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {

namespace {

constexpr uint32_t BOX16K = 16384;   // 128 rows x 64 bf16 columns, 128-byte swizzle
constexpr uint32_t BOX8K = 8192;     // 64 rows x 64 columns

// Cache row of token t of sequence b, or -1 (sets MLA_DEVERR_BOUNDS) when the
// block table or the capacity does not hold it.
MLA_DEV long long mha_cache_row(const PrefillMhaParams& p, int b, int t) {
  if (p.paged) {
    const int page = t / PAGE;
    const int id = page < p.max_blocks ? p.block_table[(long long)b * p.max_blocks + page] : -1;
    if (id < 0 || id >= p.num_blocks) {
      atomicOr(p.status, MLA_DEVERR_BOUNDS);
      return -1;
    }
    return (long long)id * PAGE + t % PAGE;
  }
  if (b >= p.num_seqs || t >= p.capacity) {
    atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return -1;
  }
  return (long long)b * p.capacity + t;
}

// ---------------------------------------------------------------------------
// K/V expansion. Grid (H column tiles of 256 over the 2*H*128 outputs, ML/128
// token tiles, B); 192 threads: warp 0 the TMA producer, warp 1 the MMA issuer,
// warps 2-5 RoPE of the queries, then the epilogue.
// ---------------------------------------------------------------------------
constexpr int EX_NS = 4;                       // stages
constexpr uint32_t EX_A = BOX16K;              // 128 tokens x 64 latent columns
constexpr uint32_t EX_B = 2 * BOX16K;          // 256 weight rows x 64 columns
constexpr uint32_t EX_STAGE = EX_A + EX_B;
constexpr uint32_t EX_PITCH = 528;             // staging row: 256 bf16 + 16 bytes of padding

struct __align__(8) ExCtrl {
  uint64_t full[EX_NS], empty[EX_NS], done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t ex_smem() { return EX_NS * EX_STAGE + sizeof(ExCtrl) + 1024; }

MLA_DEV uint8_t* align1k(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// RoPE of one (query token, head) row of 64 values: pairs (x0, x1) rotated by
// the position's float32 cos/sin with separately rounded products and sums,
// then rounded to bf16 (the cache writer's contract).
MLA_DEV void rope_q_row(const PrefillMhaParams& p, long long item) {
  const long long tok = item / p.H;
  const int pos = p.q_pos[tok];
  const uint4* src = reinterpret_cast<const uint4*>(p.q_rope + item * D_ROPE);
  uint4* dst = reinterpret_cast<uint4*>(p.q_rot + item * D_ROPE);
  if (pos < 0 || pos >= p.max_pos) {
    atomicOr(p.status, MLA_DEVERR_BOUNDS);
    return;
  }
  const float4* tab = reinterpret_cast<const float4*>(p.rope + (long long)pos * (D_ROPE / 2));
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 q = src[c];
    const float4 t0 = tab[2 * c], t1 = tab[2 * c + 1];
    const uint32_t in[4] = {q.x, q.y, q.z, q.w};
    const float2 cs[4] = {make_float2(t0.x, t0.y), make_float2(t0.z, t0.w), make_float2(t1.x, t1.y),
                          make_float2(t1.z, t1.w)};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(in[i] << 16);
      const float b = __uint_as_float(in[i] & 0xFFFF0000u);
      const float y0 = __fsub_rn(__fmul_rn(a, cs[i].x), __fmul_rn(b, cs[i].y));
      const float y1 = __fadd_rn(__fmul_rn(b, cs[i].x), __fmul_rn(a, cs[i].y));
      out[i] = pack_bf16x2(y0, y1);
    }
    dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__global__ void __launch_bounds__(192, 1) expand_kv_kernel(const __grid_constant__ CUtensorMap tm_cache,
                                                           const __grid_constant__ CUtensorMap tm_wuk,
                                                           const __grid_constant__ CUtensorMap tm_wuv,
                                                           PrefillMhaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  ExCtrl* ctl = reinterpret_cast<ExCtrl*>(smem + EX_NS * EX_STAGE);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x;                 // 256-column tile: K_nope heads 2nt, 2nt+1, or V heads
  const int t0 = blockIdx.y * 128;
  const int b = blockIdx.z;
  // the sequence length is a call input that no kernel of this library writes
  const int L = p.seq_lens[b];
  const bool len_ok = L >= 0 && L <= p.max_len;
  const bool active = len_ok && t0 < L;

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && !len_ok) atomicOr(p.status, MLA_DEVERR_LENGTH);
    for (int i = 0; i < EX_NS; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_cache);
    tma_prefetch_desc(&tm_wuk);
    tma_prefetch_desc(&tm_wuv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  const uint32_t s0 = smem_u32(smem);
  const int hh = p.H / 2;                    // column tiles per weight
  const CUtensorMap* tw = nt < hh ? &tm_wuk : &tm_wuv;
  const int wrow = (nt < hh ? nt : nt - hh) * 256;

  if (warp == 0) {
    if (lane == 0 && active) {
      // the two 64-token pages of the tile (the block table is a call input)
      long long rows[2];
      uint32_t a_bytes = 0;
      for (int pg = 0; pg < 2; ++pg) {
        const int t = t0 + 64 * pg;
        rows[pg] = t < L ? mha_cache_row(p, b, t) : -1;
        if (rows[pg] >= 0) a_bytes += BOX8K;
      }
      // weight tiles (a call input) of the first stages before the wait on the
      // previous kernel, the cache rows (which it may write) after it; one
      // arrival per stage expects both
      for (int i = 0; i < EX_NS; ++i) {
        const uint32_t f = smem_u32(&ctl->full[i]);
        mbar_arrive_expect_tx(f, EX_B + a_bytes);
        tma_load_2d(s0 + i * EX_STAGE + EX_A, tw, f, 64 * i, wrow);
      }
      pdl_wait();
      int i = 0;
      for (; i < 8; ++i) {
        const int st = i % EX_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        const uint32_t stage = s0 + st * EX_STAGE;
        if (i >= EX_NS) {
          if (!mbar_wait(smem_u32(&ctl->empty[st]), ((i / EX_NS) & 1) ^ 1, abort, p.status)) break;
          mbar_arrive_expect_tx(f, EX_B + a_bytes);
          tma_load_2d(stage + EX_A, tw, f, 64 * i, wrow);
        }
        for (int pg = 0; pg < 2; ++pg)
          if (rows[pg] >= 0) tma_load_2d(stage + pg * BOX8K, &tm_cache, f, 64 * i, static_cast<int>(rows[pg]));
      }
      if (i < 8) {
        // gave up: let the copies already issued (up to EX_NS stages) land before the CTA exits
        const int last = i < EX_NS ? EX_NS : i;
        for (int k = last - 1; k >= 0 && k >= last - EX_NS; --k)
          mbar_wait_ns(smem_u32(&ctl->full[k % EX_NS]), (k / EX_NS) & 1, 20000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && active) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 0);
      bool ok = true;
      for (int i = 0; i < 8 && ok; ++i) {
        const int st = i % EX_NS;
        if (!(ok = mbar_wait(smem_u32(&ctl->full[st]), (i / EX_NS) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t a = s0 + st * EX_STAGE, bw = a + EX_A;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, smem_desc(a + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                      smem_desc(bw + 32 * k, 16, 1024, SMEM_SWIZZLE_128B), idesc, (i | k) != 0);
        mma_commit(smem_u32(&ctl->empty[st]));
      }
      mma_commit(smem_u32(&ctl->done));
    }
  } else {
    // RoPE of the queries, spread over every CTA of the grid (q_rot is written
    // only after the wait: the previous call may still read it)
    pdl_wait();
    const int t = threadIdx.x - 64;          // 0..127
    {
      const long long ncta = (long long)gridDim.x * gridDim.y * gridDim.z;
      const long long cta = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
      const long long items = (long long)p.B * p.T * p.H;
      for (long long it = cta * 128 + t; it < items; it += ncta * 128) rope_q_row(p, it);
    }
    if (active) {
      const bool ok = mbar_wait(smem_u32(&ctl->done), 0, abort, p.status);
      tc_fence_after();
      const int q = warp & 3;                // TMEM lane quarter
      const int r = q * 32 + lane;           // token row of the tile
      uint8_t* stage = smem;                 // [128][EX_PITCH] bf16 rows (the ring is free)
      if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
          tmem_wait_ld();
          reg_fence16(v);
          const bool live = t0 + r < L;      // rows past the sequence end are zeros
          uint4 w0, w1;
          w0.x = live ? pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])) : 0u;
          w0.y = live ? pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])) : 0u;
          w0.z = live ? pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])) : 0u;
          w0.w = live ? pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])) : 0u;
          w1.x = live ? pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9])) : 0u;
          w1.y = live ? pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11])) : 0u;
          w1.z = live ? pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13])) : 0u;
          w1.w = live ? pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15])) : 0u;
          *reinterpret_cast<uint4*>(stage + r * EX_PITCH + c0 * 2) = w0;
          *reinterpret_cast<uint4*>(stage + r * EX_PITCH + c0 * 2 + 16) = w1;
        }
      }
      named_bar_sync(1, 128);
      if (ok) {
        // one 512-byte row per warp instruction (32 lanes x 16 bytes)
        const long long rs = 2ll * p.H * 128;   // kv row stride (elements)
        uint16_t* dst0 = p.kv + ((long long)b * p.ML + t0) * rs + (long long)nt * 256;
#pragma unroll 1
        for (int rr = q; rr < 128; rr += 4)
          *reinterpret_cast<uint4*>(dst0 + rr * rs + lane * 8) =
              *reinterpret_cast<const uint4*>(stage + rr * EX_PITCH + lane * 16);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// Causal attention in the expanded form. Grid (H, ceil(T/128), B), 256
// threads: warp 0 loads Q and the K tiles (TMA), warp 3 the V tiles, warp 1
// issues S = Q K^T, warp 2 issues O += P V, warps 4-7 run the softmax (thread
// = query row = TMEM lane). Shared memory: Q 48 KB | K 2 x 48 KB | V 32 KB |
// P 32 KB; tensor memory: S in two 128-column buffers, O in 128 columns.
// ---------------------------------------------------------------------------
constexpr uint32_t AT_Q = 3 * BOX16K;          // [nope 0:64 | nope 64:128 | rope] x 128 rows, K-major
constexpr uint32_t AT_K = 3 * BOX16K;          // the same for 128 keys
constexpr uint32_t AT_V = 2 * BOX16K;          // [dims 0:64 | dims 64:128] x 128 keys (MN-major B)
constexpr uint32_t AT_P = 2 * BOX16K;          // [keys 0:64 | keys 64:128] x 128 queries, K-major
constexpr uint32_t OFF_K = AT_Q;
constexpr uint32_t OFF_V = OFF_K + 2 * AT_K;
constexpr uint32_t OFF_P = OFF_V + AT_V;
constexpr uint32_t OFF_CTL = OFF_P + AT_P;
constexpr uint32_t COL_O = 256;                // S buffers at columns 0 and 128
constexpr float MHA_RESCALE_LOG2 = 8.0f;       // lazy rescale of O: running max may lag by 2^8

struct __align__(8) AtCtrl {
  uint64_t q_full, k_full[2], k_empty[2], v_full, v_empty;
  uint64_t s_full[2], s_free[2], p_full, pv_done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t at_smem() { return OFF_CTL + sizeof(AtCtrl) + 1024; }

__global__ void __launch_bounds__(256, 1) mha_prefill_kernel(const __grid_constant__ CUtensorMap tm_qn,
                                                             const __grid_constant__ CUtensorMap tm_qr,
                                                             const __grid_constant__ CUtensorMap tm_kv,
                                                             const __grid_constant__ CUtensorMap tm_cache,
                                                             PrefillMhaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  AtCtrl* ctl = reinterpret_cast<AtCtrl*>(smem + OFF_CTL);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int qt = gridDim.y - 1 - blockIdx.y;     // the query tiles that see the most keys start first
  const int b = blockIdx.z;
  const int L = p.seq_lens[b];                   // a call input: read before the wait
  const bool len_ok = L >= p.T && L <= p.max_len;
  const int q0 = qt * 128;
  const int qlast = min(q0 + 127, p.T - 1);
  const int nkt = len_ok ? (L - p.T + qlast + 1 + 127) / 128 : 0;   // key tiles up to the last query's limit

  if (threadIdx.x == 0) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && !len_ok) atomicOr(p.status, MLA_DEVERR_LENGTH);
    mbar_init(smem_u32(&ctl->q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->k_full[i]), 1);
      mbar_init(smem_u32(&ctl->k_empty[i]), 1);
      mbar_init(smem_u32(&ctl->s_full[i]), 1);
      mbar_init(smem_u32(&ctl->s_free[i]), 4);
    }
    mbar_init(smem_u32(&ctl->v_full), 1);
    mbar_init(smem_u32(&ctl->v_empty), 1);
    mbar_init(smem_u32(&ctl->p_full), 4);
    mbar_init(smem_u32(&ctl->pv_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_qn);
    tma_prefetch_desc(&tm_qr);
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_cache);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  const uint32_t sQ = smem_u32(smem), sK = sQ + OFF_K, sV = sQ + OFF_V, sP = sQ + OFF_P;
  const int kvrow0 = b * p.ML;                   // the sequence's first row in kv

  if (warp == 0) {
    if (lane == 0 && nkt > 0) {
      // q_rot and kv are written by the previous kernel, the cache rows by the
      // append before it
      pdl_wait();
      const uint32_t qf = smem_u32(&ctl->q_full);
      mbar_arrive_expect_tx(qf, AT_Q);
      for (int hf = 0; hf < 2; ++hf) tma_load_2d(sQ + hf * BOX16K, &tm_qn, qf, h * D_NOPE + 64 * hf, b * p.T + q0);
      tma_load_2d(sQ + 2 * BOX16K, &tm_qr, qf, h * D_ROPE, b * p.T + q0);
      int j = 0;
      for (; j < nkt; ++j) {
        const int st = j & 1;
        if (!mbar_wait(smem_u32(&ctl->k_empty[st]), ((j >> 1) & 1) ^ 1, abort, p.status)) break;
        const uint32_t kf = smem_u32(&ctl->k_full[st]);
        long long rows[2];
        uint32_t bytes = 2 * BOX16K;
        for (int pg = 0; pg < 2; ++pg) {
          const int t = 128 * j + 64 * pg;
          rows[pg] = t < L ? mha_cache_row(p, b, t) : -1;
          if (rows[pg] >= 0) bytes += BOX8K;
        }
        mbar_arrive_expect_tx(kf, bytes);
        const uint32_t dst = sK + st * AT_K;
        for (int hf = 0; hf < 2; ++hf) tma_load_2d(dst + hf * BOX16K, &tm_kv, kf, h * D_NOPE + 64 * hf, kvrow0 + 128 * j);
        for (int pg = 0; pg < 2; ++pg)
          if (rows[pg] >= 0) tma_load_2d(dst + 2 * BOX16K + pg * BOX8K, &tm_cache, kf, D_C, static_cast<int>(rows[pg]));
      }
      if (j < nkt) {
        // gave up: let the copies already issued land before the CTA exits
        mbar_wait_ns(qf, 0, 20000000ull);
        for (int k = j - 1; k >= 0 && k >= j - 2; --k)
          mbar_wait_ns(smem_u32(&ctl->k_full[k & 1]), (k >> 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 3) {
    if (lane == 0 && nkt > 0) {
      pdl_wait();
      const uint32_t vf = smem_u32(&ctl->v_full);
      int j = 0;
      for (; j < nkt; ++j) {
        if (!mbar_wait(smem_u32(&ctl->v_empty), (j & 1) ^ 1, abort, p.status)) break;
        mbar_arrive_expect_tx(vf, AT_V);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(sV + hf * BOX16K, &tm_kv, vf, (p.H + h) * D_V + 64 * hf, kvrow0 + 128 * j);
      }
      if (j < nkt && j > 0) mbar_wait_ns(vf, (j - 1) & 1, 20000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0 && nkt > 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);
      bool ok = mbar_wait(smem_u32(&ctl->q_full), 0, abort, p.status);
      for (int j = 0; j < nkt && ok; ++j) {
        const int st = j & 1;
        // the softmax has read the scores of tile j - 2 from this buffer
        if (j >= 2 && !(ok = mbar_wait(smem_u32(&ctl->s_free[st]), ((j - 2) >> 1) & 1, abort, p.status))) break;
        if (!(ok = mbar_wait(smem_u32(&ctl->k_full[st]), (j >> 1) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t d = tmem + 128 * st;
        const uint32_t kt = sK + st * AT_K;
#pragma unroll
        for (int kb = 0; kb < 3; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(d, smem_desc(sQ + kb * BOX16K + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                        smem_desc(kt + kb * BOX16K + 32 * k, 16, 1024, SMEM_SWIZZLE_128B), ID_S, (kb | k) != 0);
        mma_commit(smem_u32(&ctl->s_full[st]));
        mma_commit(smem_u32(&ctl->k_empty[st]));
      }
    }
  } else if (warp == 2) {
    if (lane == 0 && nkt > 0) {
      constexpr uint32_t ID_PV = idesc_bf16_f32(128, 128, 0, 1);
      bool ok = true;
      for (int j = 0; j < nkt && ok; ++j) {
        if (!(ok = mbar_wait(smem_u32(&ctl->p_full), j & 1, abort, p.status))) break;
        if (!(ok = mbar_wait(smem_u32(&ctl->v_full), j & 1, abort, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(tmem + COL_O, smem_desc(sP + kb * BOX16K + 32 * k, 16, 1024, SMEM_SWIZZLE_128B),
                        smem_desc(sV + (kb * 64 + 16 * k) * 128, BOX16K, 1024, SMEM_SWIZZLE_128B), ID_PV,
                        (j | kb | k) != 0);
        mma_commit(smem_u32(&ctl->v_empty));
        mma_commit(smem_u32(&ctl->pv_done));
      }
    }
  } else if (nkt > 0) {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                      // TMEM lane quarter
    const int r = q * 32 + lane;                 // query row of the tile
    const int qi = q0 + r;
    const bool rowv = qi < p.T;
    const int lim = L - p.T + qi;                // last key this query sees
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int st = j & 1;
      if (!(ok = mbar_wait(smem_u32(&ctl->s_full[st]), (j >> 1) & 1, abort, p.status))) break;
      tc_fence_after();
      float x[128];
      {
        uint32_t v[128];
#pragma unroll
        for (int k = 0; k < 8; ++k) tmem_ld16(tmem + lane_addr + 128 * st + 16 * k, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * k));
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + 16 * k));
#pragma unroll
        for (int i = 0; i < 128; ++i) x[i] = __uint_as_float(v[i]);
      }
      // this S buffer may take the scores of tile j + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[st]));
      // causal mask (select, not add: masked keys may be garbage) and scale
      const int kb0 = 128 * j;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        x[i] = (rowv && kb0 + i <= lim) ? x[i] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
      const bool need = mt > m_run + MHA_RESCALE_LOG2;
      const float mn = need ? mt : m_run;
      const float alpha = need ? (m_run == -INFINITY ? 0.f : fast_exp2(m_run - mn)) : 1.f;
      // P and O are free once the previous tile's P.V is done
      if (j > 0) {
        if (!(ok = mbar_wait(smem_u32(&ctl->pv_done), (j - 1) & 1, abort, p.status))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 16) {
            uint32_t v[16];
            const uint32_t ta = tmem + lane_addr + COL_O + c0;
            tmem_ld16(ta, v);
            tmem_wait_ld();
            reg_fence16(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st16(ta, v);
          }
          tmem_wait_st();
        }
      }
      l *= alpha;
      m_run = mn;
      const float moff = m_run == -INFINITY ? 0.f : m_run;
      // P = exp2(x - m) in bf16 (l sums the rounded values), row r of the
      // K-major 128-byte-swizzled A operand: keys 64kb.. in box kb, 16-byte
      // chunk c of row r at c ^ (r % 8)
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n0 = 8 * c8 + 2 * i;
          w[i] = pack_bf16x2(fast_exp2(x[n0] - moff), fast_exp2(x[n0 + 1] - moff));
          l += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xFFFF0000u);
        }
        const uint32_t addr = sP + (c8 >> 3) * BOX16K + r * 128 + ((((c8 & 7) ^ (r & 7))) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
    }
    // epilogue: O / l in bf16
    if (ok && mbar_wait(smem_u32(&ctl->pv_done), (nkt - 1) & 1, abort, p.status)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (((long long)b * p.T + qi) * p.H + h) * D_V);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + COL_O + c0, v);
        tmem_wait_ld();
        reg_fence16(v);
        if (rowv) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
          dst[c0 / 8] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[c0 / 8 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_expand_kv(const CUtensorMap& tm_cache, const CUtensorMap& tm_wuk, const CUtensorMap& tm_wuv,
                             const PrefillMhaParams& p, cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(expand_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ex_smem());
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(expand_kv_kernel, dim3(p.H, p.ML / 128, p.B), dim3(192), ex_smem(), s, tm_cache, tm_wuk, tm_wuv,
                    p);
}

cudaError_t launch_prefill_mha(const CUtensorMap& tm_qn, const CUtensorMap& tm_qr, const CUtensorMap& tm_kv,
                               const CUtensorMap& tm_cache, const PrefillMhaParams& p, cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(mha_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)at_smem());
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(mha_prefill_kernel, dim3(p.H, (p.T + 127) / 128, p.B), dim3(256), at_smem(), s, tm_qn, tm_qr,
                    tm_kv, tm_cache, p);
}

}  // namespace mla
