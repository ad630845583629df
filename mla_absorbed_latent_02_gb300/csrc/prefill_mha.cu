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
//  mha_prefill_kernel causal softmax attention, persistent (one CTA per SM
//                     walking 128-query tiles of one head, longest first):
//                     S = Q K^T over K = 192 (Q = [q_nope | q_rot], K = [K_nope
//                     | the cached RoPE key]) into tensor memory (three S/P
//                     buffers), fp32 online softmax with a lazy rescale of O, P
//                     in bf16 written over its S buffer and read from there by
//                     O += P V (V MN-major), then O / l rounded to bf16. Query
//                     j of a sequence sits at position L - T + j and sees keys
//                     0 .. L - T + j (bottom-right causal, as the absorbed path).
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"
#include "prefill_mha.cuh"

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
// token tiles, B); 224 threads: warp 0 loads the weight tiles and warp 6 the
// latent rows (TMA; one thread keeps only a few copies moving, so each operand
// has its own), warp 1 issues the MMAs, warps 2-5 rotate the queries, then run
// the epilogue. Two stages, so that two CTAs fit on an SM and one's epilogue
// overlaps the other's products.
// ---------------------------------------------------------------------------
constexpr int EX_NS = 2;                       // stages
constexpr uint32_t EX_A = BOX16K;              // 128 tokens x 64 latent columns
constexpr uint32_t EX_B = 2 * BOX16K;          // 256 weight rows x 64 columns
constexpr uint32_t EX_STAGE = EX_A + EX_B;

struct __align__(8) ExCtrl {
  uint64_t full[EX_NS], empty[EX_NS], done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t ex_smem() { return EX_NS * EX_STAGE + sizeof(ExCtrl) + 1024; }

// Named barrier that also ANDs a predicate over its threads: every thread
// leaves with the same verdict, so that a bounded wait that gave up in one
// thread stops the whole group at the same point (no later barrier or
// warp-collective tensor-memory access is left with missing threads).
MLA_DEV bool bar_red_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x 16, bf16) read from tensor memory,
// row i in lane i, two consecutive K elements per 32-bit column.
MLA_DEV void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Hint a TMA box into L2 (no shared memory, no completion).
MLA_DEV void tma_prefetch_2d(const void* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y) : "memory");
}

// TMA store of one box from this CTA's shared memory (bulk group).
MLA_DEV void tma_store_2d(const void* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}

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

__global__ void __launch_bounds__(224, 2) expand_kv_kernel(const __grid_constant__ CUtensorMap tm_cache,
                                                           const __grid_constant__ CUtensorMap tm_wuk,
                                                           const __grid_constant__ CUtensorMap tm_wuv,
                                                           const __grid_constant__ CUtensorMap tm_kvst,
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
      mbar_init(smem_u32(&ctl->full[i]), 2);   // the weight and the latent producer
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_cache);
    tma_prefetch_desc(&tm_wuk);
    tma_prefetch_desc(&tm_wuv);
    tma_prefetch_desc(&tm_kvst);
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
      // weight tiles: a call input, so the first stages go before the wait on
      // the previous kernel
      int i = 0;
      for (; i < 8; ++i) {
        const int st = i % EX_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        if (i >= EX_NS && !mbar_wait(smem_u32(&ctl->empty[st]), ((i / EX_NS) & 1) ^ 1, abort, p.status)) break;
        mbar_arrive_expect_tx(f, EX_B);
        tma_load_2d(s0 + st * EX_STAGE + EX_A, tw, f, 64 * i, wrow);
      }
      if (i < 8)   // gave up: let the copies already issued land before the CTA exits
        for (int k = i - 1; k >= 0 && k >= i - EX_NS; --k)
          mbar_wait_ns(smem_u32(&ctl->full[k % EX_NS]), (k / EX_NS) & 1, 20000000ull);
    }
  } else if (warp == 6) {
    if (lane == 0 && active) {
      // the two 64-token pages of the tile (the block table is a call input);
      // the cache rows themselves may come from the previous kernel
      long long rows[2];
      uint32_t a_bytes = 0;
      for (int pg = 0; pg < 2; ++pg) {
        const int t = t0 + 64 * pg;
        rows[pg] = t < L ? mha_cache_row(p, b, t) : -1;
        if (rows[pg] >= 0) a_bytes += BOX8K;
      }
      pdl_wait();
      int i = 0;
      for (; i < 8; ++i) {
        const int st = i % EX_NS;
        const uint32_t f = smem_u32(&ctl->full[st]);
        if (i >= EX_NS && !mbar_wait(smem_u32(&ctl->empty[st]), ((i / EX_NS) & 1) ^ 1, abort, p.status)) break;
        mbar_arrive_expect_tx(f, a_bytes);
        for (int pg = 0; pg < 2; ++pg)
          if (rows[pg] >= 0)
            tma_load_2d(s0 + st * EX_STAGE + pg * BOX8K, &tm_cache, f, 64 * i, static_cast<int>(rows[pg]));
      }
      if (i < 8)
        for (int k = i - 1; k >= 0 && k >= i - EX_NS; --k)
          mbar_wait_ns(smem_u32(&ctl->full[k % EX_NS]), (k / EX_NS) & 1, 20000000ull);
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
      mbar_wait_ns(smem_u32(&ctl->done), 0, 100000000ull);   // before the CTA frees tensor memory
    }
  } else if (warp < 6) {
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
      const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->done), 0, abort, p.status));
      tc_fence_after();
      const int q = warp & 3;                // TMEM lane quarter
      const int r = q * 32 + lane;           // token row of the tile
      // the tile in bf16 through shared memory (the ring is free): four boxes
      // of 64 columns x 128 rows, 128-byte swizzled (16-byte chunk c of row r
      // at c ^ (r % 8)), written out by four TMA stores
      const uint32_t stage = s0;
      if (ok) {
        const bool live = t0 + r < L;        // rows past the sequence end are zeros
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
          tmem_wait_ld();
          reg_fence16(v);
          uint32_t u[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            u[c] = live ? pack_bf16x2(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])) : 0u;
          const uint32_t box = stage + (c0 >> 6) * BOX16K + r * 128;
          const int ch = (c0 & 63) >> 3;       // 16-byte chunk of the row within its box
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(box + (((ch) ^ (r & 7)) << 4)), "r"(u[0]),
                       "r"(u[1]), "r"(u[2]), "r"(u[3])
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(box + (((ch + 1) ^ (r & 7)) << 4)), "r"(u[4]),
                       "r"(u[5]), "r"(u[6]), "r"(u[7])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (ok && t == 0) {
        const int y = b * p.ML + t0;
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) tma_store_2d(&tm_kvst, stage + bx * BOX16K, nt * 256 + 64 * bx, y);
        bulk_commit();
        // the stores complete (not only their reads of shared memory) before the
        // CTA leaves, so that the attention's wait on this kernel covers them
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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
// Causal attention in the expanded form: a persistent kernel, one CTA per SM,
// walking work items (one 128-query tile of one head of one sequence) dealt
// out longest first in snake order (mha_item_index). 384 threads:
// warp 0 loads Q and the K tiles (K_nope from kv, the RoPE keys from the
// cache rows) and warp 3 the V tiles (TMA), so that no K load waits behind a
// V stage; warp 1 issues S = Q K^T, warp 2 issues O += P V,
// warps 4-11 run the softmax in two groups of four warps (thread = query row
// = TMEM lane; group g owns the score columns, P keys and O columns 64g ..
// 64g+63 of its rows, and the two exchange the row maxima through shared
// memory). P (bf16) is written over the first 64 columns of its own S buffer
// in tensor memory and is the A operand of P.V from there; three S/P buffers,
// so the scores run up to two tiles ahead of the P.V that frees a buffer and
// the softmax of tile n+1 never waits for the P.V of tile n (only a rescale
// of O does). Barrier phases run on across items, so the next item's queries
// and keys load while the current one ends; its queries are hinted into L2
// once the current item's keys are issued. The epilogue writes O through small
// per-warp shared-memory stripes, one 128-byte row segment per 8 lanes.
// Shared memory: Q 48 KB | K 2 x 48 KB | V 2 x 32 KB | 8 KB of stripes;
// tensor memory: S/P in three 128-column buffers, O in 128 columns.
// ---------------------------------------------------------------------------
constexpr uint32_t AT_Q = 3 * BOX16K;          // [nope 0:64 | nope 64:128 | rope] x 128 rows, K-major
constexpr uint32_t AT_K = 3 * BOX16K;          // the same for 128 keys
constexpr uint32_t AT_V = 2 * BOX16K;          // [dims 0:64 | dims 64:128] x 128 keys (MN-major B)
constexpr uint32_t OFF_K = AT_Q;
constexpr uint32_t OFF_V = OFF_K + 2 * AT_K;
constexpr uint32_t OFF_CTL = OFF_V + 2 * AT_V;
constexpr int AT_NS = 3;                       // S/P buffers in tensor memory
constexpr uint32_t COL_O = 128 * AT_NS;        // S/P buffers at columns 0, 128, 256; O after them
constexpr float MHA_RESCALE_LOG2 = 8.0f;       // lazy rescale of O: running max may lag by 2^8

struct __align__(16) AtCtrl {
  uint64_t q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2];
  // pv_done by S/P buffer: up to AT_NS P.V can be outstanding, so one barrier
  // waited by parity could alias a phase two tiles back
  uint64_t s_full[AT_NS], s_free[AT_NS], p_full[AT_NS], pv_done[AT_NS], o_empty, mma_final;
  uint32_t tmem_base;
  int abort;
  float red[2][2][128];   // by tile parity and group: each row's partial score maximum
  float lsum[2][128];     // by group: each row's partial normaliser
  uint4 ostage[8][64];    // per softmax warp: 8 rows x 128 bytes of O on their way out
};

constexpr size_t at_smem() { return OFF_CTL + sizeof(AtCtrl) + 1024; }

// Work item i: query tile qt (the tiles with the most keys first), sequence b,
// head h, and its key-tile count (0 for a sequence whose length is out of range).
struct MhaItem {
  int b, h, q0, L, nkt;
};
MLA_DEV MhaItem mha_item(const PrefillMhaParams& p, int i) {
  const int nqt = (p.T + 127) / 128;
  const int per = p.H * p.B;
  MhaItem it;
  const int qt = nqt - 1 - i / per;
  const int rest = i % per;
  it.b = rest / p.H;
  it.h = rest % p.H;
  it.q0 = qt * 128;
  it.L = p.seq_lens[it.b];   // a call input: read before the wait
  const int qlast = min(it.q0 + 127, p.T - 1);
  it.nkt = (it.L >= p.T && it.L <= p.max_len) ? (it.L - p.T + qlast + 1 + 127) / 128 : 0;
  return it;
}

// The k-th item of this CTA: the items (longest first) are dealt out in
// rounds of gridDim.x, alternately in CTA order and in reverse (snake order),
// which evens out the key tiles per CTA far better than plain rounds (the
// busiest CTA of a 1,024-token prompt at H=128: 3 % above the mean instead of
// 10 %, counting each item's start as 1.5 tiles).
MLA_DEV int mha_item_index(int k) {
  const int g = gridDim.x;
  return k * g + ((k & 1) ? g - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
}

__global__ void __launch_bounds__(384, 1) mha_prefill_kernel(const __grid_constant__ CUtensorMap tm_qn,
                                                             const __grid_constant__ CUtensorMap tm_qr,
                                                             const __grid_constant__ CUtensorMap tm_kv,
                                                             const __grid_constant__ CUtensorMap tm_cache,
                                                             PrefillMhaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  AtCtrl* ctl = reinterpret_cast<AtCtrl*>(smem + OFF_CTL);
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = ((p.T + 127) / 128) * p.H * p.B;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    mbar_init(smem_u32(&ctl->q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->k_full[i]), 1);
      mbar_init(smem_u32(&ctl->k_empty[i]), 1);
      mbar_init(smem_u32(&ctl->v_full[i]), 1);
      mbar_init(smem_u32(&ctl->v_empty[i]), 1);
    }
    for (int i = 0; i < AT_NS; ++i) {
      mbar_init(smem_u32(&ctl->s_full[i]), 1);
      mbar_init(smem_u32(&ctl->s_free[i]), 1);    // the P.V that read this buffer's P
      mbar_init(smem_u32(&ctl->p_full[i]), 8);    // every softmax warp
    }
    for (int i = 0; i < AT_NS; ++i) mbar_init(smem_u32(&ctl->pv_done[i]), 1);
    mbar_init(smem_u32(&ctl->o_empty), 8);
    mbar_init(smem_u32(&ctl->mma_final), 2);    // both MMA issuers
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
  const uint32_t sQ = smem_u32(smem), sK = sQ + OFF_K, sV = sQ + OFF_V;

  if (warp == 0) {
    if (lane == 0) {
      // q_rot and kv are written by the previous kernel, the cache rows by the
      // append before it
      pdl_wait();
      const uint32_t qf = smem_u32(&ctl->q_full);
      uint32_t n = 0, k = 0;   // key tiles and items issued
      bool ok = true;
      for (int ik = 0, i = mha_item_index(0); i < n_items && ok; i = mha_item_index(++ik)) {
        const MhaItem it = mha_item(p, i);
        if (it.nkt == 0) {
          if (it.h == 0 && it.q0 == 0) atomicOr(p.status, MLA_DEVERR_LENGTH);
          continue;
        }
        if (!(ok = mbar_wait(smem_u32(&ctl->q_empty), (k & 1) ^ 1, abort, p.status))) break;
        mbar_arrive_expect_tx(qf, AT_Q);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_2d(sQ + hf * BOX16K, &tm_qn, qf, it.h * D_NOPE + 64 * hf, it.b * p.T + it.q0);
        tma_load_2d(sQ + 2 * BOX16K, &tm_qr, qf, it.h * D_ROPE, it.b * p.T + it.q0);
        ++k;
        const int kvrow0 = it.b * p.ML;   // the sequence's first row in kv
        auto page_row = [&](int t) -> long long { return t < it.L ? mha_cache_row(p, it.b, t) : -1; };
        for (int j = 0; j < it.nkt; ++j) {
          const int st = n & 1;
          if (!(ok = mbar_wait(smem_u32(&ctl->k_empty[st]), ((n >> 1) & 1) ^ 1, abort, p.status))) break;
          const uint32_t kf = smem_u32(&ctl->k_full[st]);
          long long rows[2];
          uint32_t bytes = 2 * BOX16K;
          for (int pg = 0; pg < 2; ++pg) {
            rows[pg] = page_row(128 * j + 64 * pg);
            if (rows[pg] >= 0) bytes += BOX8K;
          }
          mbar_arrive_expect_tx(kf, bytes);
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sK + st * AT_K + hf * BOX16K, &tm_kv, kf, it.h * D_NOPE + 64 * hf, kvrow0 + 128 * j);
          for (int pg = 0; pg < 2; ++pg)
            if (rows[pg] >= 0)
              tma_load_2d(sK + st * AT_K + 2 * BOX16K + pg * BOX8K, &tm_cache, kf, D_C, static_cast<int>(rows[pg]));
          ++n;
        }
        // the next item's queries into L2: this thread only waits for the
        // query buffer next (one TMA op costs its issuing thread ~0.2-0.3 us,
        // so hints are kept to the idle point of the loop)
        if (ok && mha_item_index(ik + 1) < n_items) {
          const MhaItem nx = mha_item(p, mha_item_index(ik + 1));
          if (nx.nkt > 0) {
            for (int hf = 0; hf < 2; ++hf) tma_prefetch_2d(&tm_qn, nx.h * D_NOPE + 64 * hf, nx.b * p.T + nx.q0);
            tma_prefetch_2d(&tm_qr, nx.h * D_ROPE, nx.b * p.T + nx.q0);
          }
        }
      }
      if (!ok) {
        // gave up: let the copies already issued land before the CTA exits
        if (k > 0) mbar_wait_ns(qf, (k - 1) & 1, 20000000ull);
        for (uint32_t m = n; m > 0 && m + 2 > n; --m)
          mbar_wait_ns(smem_u32(&ctl->k_full[(m - 1) & 1]), ((m - 1) >> 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 3) {
    if (lane == 0) {
      pdl_wait();
      uint32_t n = 0;   // tiles whose V is issued
      bool ok = true;
      for (int ik = 0, i = mha_item_index(0); i < n_items && ok; i = mha_item_index(++ik)) {
        const MhaItem it = mha_item(p, i);
        const int kvrow0 = it.b * p.ML;
        for (int j = 0; j < it.nkt; ++j) {
          const int vs = n & 1;
          if (!(ok = mbar_wait(smem_u32(&ctl->v_empty[vs]), ((n >> 1) & 1) ^ 1, abort, p.status))) break;
          const uint32_t vf = smem_u32(&ctl->v_full[vs]);
          mbar_arrive_expect_tx(vf, AT_V);
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sV + vs * AT_V + hf * BOX16K, &tm_kv, vf, (p.H + it.h) * D_V + 64 * hf, kvrow0 + 128 * j);
          ++n;
        }
      }
      if (!ok)
        for (uint32_t m = n; m > 0 && m + 2 > n; --m)
          mbar_wait_ns(smem_u32(&ctl->v_full[(m - 1) & 1]), ((m - 1) >> 1) & 1, 20000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);
      uint32_t n = 0, k = 0;
      bool ok = true;
      for (int ik = 0, i = mha_item_index(0); i < n_items && ok; i = mha_item_index(++ik)) {
        const MhaItem it = mha_item(p, i);
        if (it.nkt == 0) continue;
        if (!(ok = mbar_wait(smem_u32(&ctl->q_full), k & 1, abort, p.status))) break;
        for (int j = 0; j < it.nkt; ++j) {
          const int sb = n % AT_NS, ks = n & 1;
          // the P.V of tile n - 3 has read its P from this buffer
          if (n >= AT_NS &&
              !(ok = mbar_wait(smem_u32(&ctl->s_free[sb]), ((n - AT_NS) / AT_NS) & 1, abort, p.status)))
            break;
          if (!(ok = mbar_wait(smem_u32(&ctl->k_full[ks]), (n >> 1) & 1, abort, p.status))) break;
          tc_fence_after();
          const uint32_t kt = sK + ks * AT_K;
#pragma unroll
          for (int kb = 0; kb < 3; ++kb)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16_ss(tmem + 128 * sb, smem_desc(sQ + kb * BOX16K + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B),
                          smem_desc(kt + kb * BOX16K + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B), ID_S, (kb | kk) != 0);
          mma_commit(smem_u32(&ctl->s_full[sb]));
          mma_commit(smem_u32(&ctl->k_empty[ks]));
          ++n;
        }
        if (!ok) break;
        mma_commit(smem_u32(&ctl->q_empty));   // the next item's queries may load
        ++k;
      }
      // every MMA of both issuers has completed once mma_final flips (before
      // the CTA frees tensor memory)
      mma_commit(smem_u32(&ctl->mma_final));
      mbar_wait_ns(smem_u32(&ctl->mma_final), 0, 100000000ull);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      constexpr uint32_t ID_PV = idesc_bf16_f32(128, 128, 0, 1);
      uint32_t n = 0, k = 0;
      bool ok = true;
      for (int ik = 0, i = mha_item_index(0); i < n_items && ok; i = mha_item_index(++ik)) {
        const MhaItem it = mha_item(p, i);
        if (it.nkt == 0) continue;
        // O of the previous item has been read by the epilogue
        if (k > 0 && !(ok = mbar_wait(smem_u32(&ctl->o_empty), (k - 1) & 1, abort, p.status))) break;
        for (int j = 0; j < it.nkt; ++j) {
          const int sb = n % AT_NS, vs = n & 1;
          if (!(ok = mbar_wait(smem_u32(&ctl->p_full[sb]), (n / AT_NS) & 1, abort, p.status))) break;
          if (!(ok = mbar_wait(smem_u32(&ctl->v_full[vs]), (n >> 1) & 1, abort, p.status))) break;
          tc_fence_after();
          // A = P from tensor memory (row = lane, two bf16 keys per column:
          // keys 16kk .. 16kk+15 in columns 8kk .. 8kk+7 of the buffer)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + COL_O, tmem + 128 * sb + 8 * kk,
                        smem_desc(sV + vs * AT_V + 16 * kk * 128, BOX16K, 1024, SMEM_SWIZZLE_128B), ID_PV,
                        (j | kk) != 0);
          mma_commit(smem_u32(&ctl->v_empty[vs]));
          mma_commit(smem_u32(&ctl->s_free[sb]));
          mma_commit(smem_u32(&ctl->pv_done[sb]));
          ++n;
        }
        ++k;
      }
      mma_commit(smem_u32(&ctl->mma_final));
      mbar_wait_ns(smem_u32(&ctl->mma_final), 0, 100000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                      // TMEM lane quarter
    const int grp = (warp - 4) >> 2;             // columns 64grp .. 64grp+63
    const int cb = 64 * grp;
    const int r = q * 32 + lane;                 // query row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const float sl2 = p.scale_log2;
    // Every softmax thread runs every iteration and every barrier; a wait
    // that gave up clears `ok` for the whole group at the next barrier, and
    // the rest then does nothing.
    bool ok = true;
    uint32_t n = 0;
    for (int ik = 0, i = mha_item_index(0); i < n_items; i = mha_item_index(++ik)) {
      const MhaItem it = mha_item(p, i);
      if (it.nkt == 0) continue;
      const int qi = it.q0 + r;
      const bool rowv = qi < p.T;
      const int lim = rowv ? it.L - p.T + qi : -1;   // last key this query sees
      float m_run = -INFINITY, l = 0.f;   // running maximum (scaled, log2 units), this group's sum
      for (int j = 0; j < it.nkt; ++j, ++n) {
        const int st = n & 1, sb = n % AT_NS;   // maxima exchange by parity, S/P buffer
        if (ok) ok = mbar_wait(smem_u32(&ctl->s_full[sb]), (n / AT_NS) & 1, abort, p.status);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        float x[64];
        if (ok) {
          uint32_t v[64];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld16(tmem + lane_addr + 128 * sb + cb + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(v + 16 * c));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + 16 * c));
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(v[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = -INFINITY;
        }
        // causal mask on the tiles that reach past a row's limit (select, not
        // add: masked keys may be garbage); the scale is applied with the max
        const int kb0 = 128 * j + cb;
        float mt = -INFINITY;
        if (kb0 + 63 <= lim) {
#pragma unroll
          for (int c = 0; c < 64; ++c) mt = fmaxf(mt, x[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            x[c] = kb0 + c <= lim ? x[c] : -INFINITY;
            mt = fmaxf(mt, x[c]);
          }
        }
        // the barrier also orders both groups' reads of this S buffer before
        // either group writes its P over it
        ctl->red[st][grp][r] = mt * sl2;
        tc_fence_before();
        ok = bar_red_and(1, 256, ok);
        tc_fence_after();
        mt = fmaxf(ctl->red[st][0][r], ctl->red[st][1][r]);
        const bool need = mt > m_run + MHA_RESCALE_LOG2;
        const float mn = need ? mt : m_run;
        const float alpha = need ? (m_run == -INFINITY ? 0.f : fast_exp2(m_run - mn)) : 1.f;
        const float moff = mn == -INFINITY ? 0.f : mn;
        // P = exp2(x * scale_log2 - m) in bf16 (l sums the unrounded values)
        uint32_t w[32];
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = fast_exp2(fmaf(x[2 * c], sl2, -moff));
          const float p1 = fast_exp2(fmaf(x[2 * c + 1], sl2, -moff));
          w[c] = pack_bf16x2(p0, p1);
          ls += p0 + p1;
        }
        // O holds the previous tile's products once its P.V is done: rescale
        // it only when the running maximum moved (rare)
        if (j > 0 && ok && __any_sync(0xffffffffu, need)) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ctl->pv_done[(n - 1) % AT_NS]), ((n - 1) / AT_NS) & 1,
                                                 abort, p.status));
          tc_fence_after();
          if (ok) {
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 16) {
              uint32_t v[16];
              const uint32_t ta = tmem + lane_addr + COL_O + cb + c0;
              tmem_ld16(ta, v);
              tmem_wait_ld();
              reg_fence16(v);
#pragma unroll
              for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
              tmem_st16(ta, v);
            }
          }
        }
        l = l * alpha + ls;
        m_run = mn;
        // P of this group's 64 keys over columns 32grp .. 32grp+31 of the S
        // buffer (its scores are in registers already)
        if (ok) {
          tmem_st16(tmem + lane_addr + 128 * sb + 32 * grp, *reinterpret_cast<const uint32_t(*)[16]>(w));
          tmem_st16(tmem + lane_addr + 128 * sb + 32 * grp + 16, *reinterpret_cast<const uint32_t(*)[16]>(w + 16));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(smem_u32(&ctl->p_full[sb]));
      }
      // epilogue: O / l in bf16, each group its 64 columns of the row; then O
      // may take the next item's products
      ctl->lsum[grp][r] = l;
      ok = bar_red_and(1, 256, ok);
      // the item's last P.V (the P.V complete in issue order)
      if (ok) ok = mbar_wait(smem_u32(&ctl->pv_done[(n - 1) % AT_NS]), ((n - 1) / AT_NS) & 1, abort, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float lt = ctl->lsum[0][r] + ctl->lsum[1][r];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        // this row's 64 columns in bf16: eight 16-byte chunks
        uint4 o[8];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_addr + COL_O + cb + c0, v);
          tmem_wait_ld();
          reg_fence16(v);
          uint32_t u[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            u[c] = pack_bf16x2(__uint_as_float(v[2 * c]) * inv, __uint_as_float(v[2 * c + 1]) * inv);
          o[c0 / 8] = make_uint4(u[0], u[1], u[2], u[3]);
          o[c0 / 8 + 1] = make_uint4(u[4], u[5], u[6], u[7]);
        }
        // out through this warp's stripe, 8 rows at a time: the 8 lanes of a
        // round put their rows in (chunk c of row m at c ^ m), then every lane
        // writes one 16-byte chunk, 8 lanes per 128-byte row segment
        uint4* stripe = ctl->ostage[warp - 4];
        const int wrow0 = it.q0 + q * 32;            // the warp's first query row
#pragma unroll 1
        for (int k8 = 0; k8 < 4; ++k8) {
          if ((lane >> 3) == k8) {
            const int m = lane & 7;
#pragma unroll
            for (int c = 0; c < 8; ++c) stripe[m * 8 + (c ^ m)] = o[c];
          }
          __syncwarp();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int m = (lane >> 3) + 4 * hh, c = lane & 7;
            const int qrow = wrow0 + 8 * k8 + m;
            if (qrow < p.T) {
              uint4* dst = reinterpret_cast<uint4*>(p.out + (((long long)it.b * p.T + qrow) * p.H + it.h) * D_V + cb);
              dst[c] = stripe[m * 8 + (c ^ m)];
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(smem_u32(&ctl->o_empty));
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
                             const CUtensorMap& tm_kvst, const PrefillMhaParams& p, cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(expand_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ex_smem());
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(expand_kv_kernel, dim3(p.H, p.ML / 128, p.B), dim3(224), ex_smem(), s, tm_cache, tm_wuk, tm_wuv,
                    tm_kvst, p);
}

cudaError_t launch_prefill_mha(const CUtensorMap& tm_qn, const CUtensorMap& tm_qr, const CUtensorMap& tm_kv,
                               const CUtensorMap& tm_cache, const PrefillMhaParams& p, cudaStream_t s) {
  static DeviceFlags attr;
  const cudaError_t e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(mha_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)at_smem());
  });
  if (e != cudaSuccess) return e;
  const int items = (p.T + 127) / 128 * p.H * p.B;
  return launch_pdl(mha_prefill_kernel, dim3(items < p.num_ctas ? items : p.num_ctas), dim3(384), at_smem(), s, tm_qn,
                    tm_qr, tm_kv, tm_cache, p);
}

}  // namespace mla
