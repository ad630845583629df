// Absorbed-MLA decode attention over the 576-wide latent cache.
//
// For each sequence b and query row g = (j, h):
//   s_t   = scale * (q_abs[g] . row_t),  row_t = [c_kv_t | RoPE(k_rope_t)]
//   p     = softmax over t < L_b - (Hq - 1 - j)   (bottom-right causal)
//   o_lat = sum_t p_t c_kv_t,  lse = log sum_t exp(s_t)
// This is the absorbed form of MLA ("DeepSeek MLA 吸收式缓存" §2.2-§2.3;
// "80 行 PyTorch 从零写 DeepSeek 的 MLA" §5): every head reads the same cached
// row, a multi-query attention with a 576-wide key and a 512-wide value
// ("DeepSeek MLA 吸收式缓存" §6.1, MQA mode).
//
// GB300 design (one CTA per SM, persistent):
//  * Tokens are the MMA's M axis ("swap AB"): a 128-token tile of the cache is
//    the A operand of both contractions and is read from HBM once for all the
//    heads of the CTA.
//      S^T[128 tok x N] = C[128 x 576] . Q[N x 576]^T      (tcgen05, K-major A/B)
//      O^T[512 x N]    += C[:, :512]^T . P^T[128 x N]       (tcgen05, MN-major A)
//    N = query rows per CTA (16, 32 or 64); G > 64 rows are spread over C CTAs
//    that walk the same tokens (the second read of a tile comes from L2).
//  * Cache tiles arrive by TMA in 64x64 boxes (one paged block of 64 tokens,
//    64 columns) with the 128-byte swizzle. Latent columns are staged in
//    32 KB "pair" slots (128 tokens x 128 columns), the RoPE columns in 16 KB
//    slots that hold P after the score MMA has read them.
//  * Warp roles: warps 0 and 3 issue TMA (one page of each tile each), warp 1
//    issues the score MMAs, warp 2 owns TMEM and issues the P.C MMAs,
//    warps 4-11 (two groups of four, each owning half of the query rows) run
//    the fp32 online softmax (one token row per thread) and the epilogue.
//    Rescaling of O is lazy: only when a running max grows by more than 2^8.
//  * Split-KV: the flattened list of (sequence, tile) is cut into U equal
//    ranges, one per unit; a sequence cut across units writes normalised
//    partials + lse that the combine kernel merges by log-sum-exp.
#include "attn_sched.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase trace (compile with -DMLA_TRACE=1): SM clock stamps of the
// pipeline events of the first tiles of the first CTAs, read back with
// mla_trace_read(). Off in normal builds.
#ifndef MLA_TRACE
#define MLA_TRACE 0
#endif
#if MLA_TRACE
#define MLA_TRACE_CTAS 8
#define MLA_TRACE_TILES 32
#define MLA_TRACE_EVENTS 12
__device__ long long g_mla_trace[MLA_TRACE_CTAS][MLA_TRACE_TILES][MLA_TRACE_EVENTS];
#define TRACE_EV(ev, tile)                                                          \
  do {                                                                              \
    if (blockIdx.x < MLA_TRACE_CTAS && (tile) < MLA_TRACE_TILES)                    \
      g_mla_trace[blockIdx.x][(tile)][(ev)] = clock64();                            \
  } while (0)
__device__ unsigned long long g_mla_trace_cta[1024][4];
#define TRACE_CTA(ev)                                                     \
  do {                                                                    \
    if (blockIdx.x < 1024) g_mla_trace_cta[blockIdx.x][(ev)] = globaltimer(); \
  } while (0)
extern "C" int mla_trace_read(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace)) bytes = sizeof(g_mla_trace);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace, bytes);
}
__device__ unsigned long long g_mla_trace_comb[1024][3];
#define TRACE_COMB(ev)                                                                         \
  do {                                                                                         \
    const unsigned cta = blockIdx.x + gridDim.x * blockIdx.y;                                  \
    if (cta < 1024 && threadIdx.x == 0) g_mla_trace_comb[cta][(ev)] = globaltimer();           \
  } while (0)
extern "C" int mla_trace_read_comb(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace_comb)) bytes = sizeof(g_mla_trace_comb);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace_comb, bytes);
}
extern "C" int mla_trace_read_cta(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace_cta)) bytes = sizeof(g_mla_trace_cta);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace_cta, bytes);
}
#else
#define TRACE_EV(ev, tile) \
  do {                     \
  } while (0)
#define TRACE_CTA(ev) \
  do {                \
  } while (0)
#define TRACE_COMB(ev) \
  do {                 \
  } while (0)
#endif

namespace mla {

namespace {

constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;   // lazy-rescale threshold (log2 units)
constexpr uint32_t PAIR_BYTES = 32768; // 128 tokens x 128 latent columns
constexpr uint32_t HALF_BYTES = 16384; // 128 tokens x 64 columns
constexpr uint32_t BOX_BYTES = 8192;   // 64 tokens x 64 columns (one TMA box)
constexpr int NP_MAX = 5, NR_MAX = 2;

template <int N>
struct Cfg {
  static constexpr int NP = (N == 64) ? 4 : 5;  // latent pair slots
  static constexpr int NR = (N == 16) ? 2 : 1;  // rope / P slots
  static constexpr uint32_t Q_BYTES = 9u * N * 128u;
  static constexpr uint32_t OFF_PAIR = Q_BYTES;
  static constexpr uint32_t OFF_ROPE = OFF_PAIR + NP * PAIR_BYTES;
  static constexpr uint32_t OFF_CTRL = OFF_ROPE + NR * HALF_BYTES;
  static constexpr uint32_t TMEM_COLS = (6 * N <= 128) ? 128u : (6 * N <= 256 ? 256u : 512u);
  static constexpr uint32_t COL_S = 4 * N;       // two S^T buffers of N columns; O^T m-tile mt at mt*N
  // P^T is stored token-major (MN-major B operand): rows of 2N bytes, swizzled
  // with the pattern whose width equals the row (32, 64 or 128 bytes).
  static constexpr int P_CHUNKS = (2 * N) / 16;  // 16-byte chunks per P row
  static constexpr uint32_t P_LAYOUT = (N == 16) ? SMEM_SWIZZLE_32B : (N == 32 ? SMEM_SWIZZLE_64B : SMEM_SWIZZLE_128B);
  // RoPE columns first when a free RoPE slot exists ahead of the current tile
  static constexpr bool ROPE_FIRST = NR >= 2;
  // softmax/epilogue: GR groups of 4 warps, NC columns each (four groups at
  // N = 64 keep a thread's share of a tile at 16 columns)
  static constexpr int GR = N == 64 ? 4 : 2;
  static constexpr int NC = N / GR;
  static constexpr int CW = NC < 16 ? NC : 16;   // TMEM columns per load
  static constexpr int THREADS = 128 + 128 * GR;
};

struct __align__(8) Ctrl {
  uint64_t q_full, q_empty;
  uint64_t pair_full[NP_MAX], pair_empty[NP_MAX];
  uint64_t rope_full[NR_MAX], rope_empty[NR_MAX];
  // by tile parity: S written / S read by the softmax / P written / P.C done
  uint64_t s_full[2], s_free[2], p_full[2], pc_done[2];
  uint64_t o_full, o_empty, mma_final;
  uint32_t tmem_base;
  int abort;
  int vote[4][2][4];
  float m_run[64];
  float alpha[64];
  float red[4][64];
  float lsum[64];
  float linv[64];
  int warp_tot[32];   // one per warp of the CTA (tile_prefix)
};

}  // namespace

template <int N>
__global__ void __launch_bounds__(Cfg<N>::THREADS, 1)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tm_cache,
                       const __grid_constant__ CUtensorMap tm_q, const AttnParams p) {
  using K = Cfg<N>;
  if (threadIdx.x == 0) TRACE_CTA(0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + K::OFF_CTRL);
  const uint32_t s_q = smem_u32(smem);
  const uint32_t s_pair = s_q + K::OFF_PAIR;
  const uint32_t s_rope = s_q + K::OFF_ROPE;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.C;     // unit
  // row group within the unit; with one unit (CTAs in waves) the groups of the
  // latest query tokens, which see the most tiles, are launched first
  const int c = p.U == 1 ? p.C - 1 - blockIdx.x % p.C : blockIdx.x % p.C;
  volatile int* abort = &ctl->abort;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    mbar_init(smem_u32(&ctl->q_empty), 1);
    for (int i = 0; i < K::NP; ++i) {
      mbar_init(smem_u32(&ctl->pair_full[i]), 2);   // one arrival per producer (page)
      mbar_init(smem_u32(&ctl->pair_empty[i]), 1);
    }
    for (int i = 0; i < K::NR; ++i) {
      mbar_init(smem_u32(&ctl->rope_full[i]), 2);
      mbar_init(smem_u32(&ctl->rope_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->s_full[i]), 1);
      mbar_init(smem_u32(&ctl->s_free[i]), 4 * K::GR);
      mbar_init(smem_u32(&ctl->p_full[i]), 4 * K::GR);
      mbar_init(smem_u32(&ctl->pc_done[i]), 1);
    }
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->o_empty), 4 * K::GR);
    mbar_init(smem_u32(&ctl->mma_final), 2);   // both MMA issuers
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_cache);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctl->tmem_base), K::TMEM_COLS);
    tmem_relinquish();
  }
  int* pre = reinterpret_cast<int*>(smem + K::OFF_CTRL + sizeof(Ctrl));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  // The unit's tile range depends only on the sequence lengths, a call input no
  // kernel of this library writes, so it is computed before the wait on the
  // previous kernel; so are L2 prefetch hints for the unit's first tiles, which
  // then stream from HBM while that kernel finishes (a hint cannot change what
  // the loads after the wait read).
  tile_prefix(p, pre, ctl->warp_tot);
  if (threadIdx.x == 0 && c == 0) {
    ItemIter it;
    it.init(p, pre, u, c);
    int b, t0, t1, L;
    long long acc;
    if (it.next(b, t0, t1, L, acc))
      for (int tau = t0; tau < t1 && tau < t0 + 1; ++tau)
        for (int pg = 0; pg < 2; ++pg) {
          const int page = 2 * tau + pg;
          if (page * PAGE >= L) break;
          long long r = -1;
          if (p.paged) {
            const int id = page < p.max_blocks ? p.block_table[(long long)b * p.max_blocks + page] : -1;
            if (id >= 0 && id < p.num_blocks) r = (long long)id * PAGE;
          } else if (L <= p.capacity) {
            r = (long long)b * p.capacity + page * PAGE;
          }
          if (r >= 0)
            prefetch_l2_bulk(p.cache + r * (ROW * 2), static_cast<uint32_t>(min(PAGE, L - page * PAGE) * ROW * 2));
        }
  }
  pdl_wait();
  if (threadIdx.x == 0) TRACE_CTA(1);

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // Two producer threads, one per 64-token page of each tile (warp 0: the
    // first page and the queries, warp 3: the second page). One thread keeps
    // only a few copies moving at a time (about 40 GB/s into one SM with 8 KB
    // boxes, below an SM's share of HBM); two threads double that. Both
    // arrive on every slot's full barrier with the bytes of their own boxes.
    if (lane == 0) {
      const int pg = warp == 0 ? 0 : 1;   // page of the tile this thread loads
      ItemIter it;
      it.init(p, pre, u, c);
      uint32_t pair_i = 0, rope_i = 0, item_i = 0, ptile = 0;
      int b, t0, t1, L;
      long long acc;
      // Tiles read by one CTA only are streamed with an evict-first hint; when
      // C > 1 CTAs read the same tile the later reads should still find it in L2.
      const bool stream_hint = p.C == 1;
      const uint64_t pol_stream = l2_policy_evict_first();
      bool ok = true;
      while (ok && it.next(b, t0, t1, L, acc)) {
        if (pg == 0) {
          const uint32_t qf = smem_u32(&ctl->q_full);
          if (!(ok = mbar_wait(smem_u32(&ctl->q_empty), (item_i & 1) ^ 1, abort, p.status))) break;
          mbar_arrive_expect_tx(qf, K::Q_BYTES);
          for (int kb = 0; kb < 9; ++kb)
            tma_load_2d(s_q + kb * N * 128, &tm_q, qf, 64 * kb, b * p.G + c * N);
        }
        for (int tau = t0; tau < t1 && ok; ++tau) {
          const int page = 2 * tau + pg;
          int row = -1;
          if (page * PAGE < L) {
            if (p.paged) {
              const int id = page < p.max_blocks ? p.block_table[(long long)b * p.max_blocks + page] : -1;
              if (id >= 0 && id < p.num_blocks) row = id * PAGE;
              else atomicOr(p.status, MLA_DEVERR_BOUNDS);
            } else {
              if (L > p.capacity) atomicOr(p.status, MLA_DEVERR_BOUNDS);
              else row = b * p.capacity + page * PAGE;
            }
          }
          const uint32_t nbox = row >= 0 ? 1u : 0u;
          if (pg == 0) TRACE_EV(0, ptile);
          auto load_rope = [&]() -> bool {
            const uint32_t rslot = rope_i % K::NR;
            if (!mbar_wait(smem_u32(&ctl->rope_empty[rslot]), ((rope_i / K::NR) & 1) ^ 1, abort, p.status))
              return false;
            const uint32_t rfull = smem_u32(&ctl->rope_full[rslot]);
            mbar_arrive_expect_tx(rfull, nbox * BOX_BYTES);
            if (row >= 0) {
              const uint32_t dst = s_rope + rslot * HALF_BYTES + pg * BOX_BYTES;
              if (stream_hint) tma_load_2d_hint(dst, &tm_cache, rfull, D_C, row, pol_stream);
              else tma_load_2d(dst, &tm_cache, rfull, D_C, row);
            }
            return true;
          };
          if (K::ROPE_FIRST && !(ok = load_rope())) break;
          for (int pr = 0; pr < 4; ++pr) {
            const uint32_t slot = pair_i % K::NP;
            if (!(ok = mbar_wait(smem_u32(&ctl->pair_empty[slot]), ((pair_i / K::NP) & 1) ^ 1, abort, p.status))) break;
            if (pr == 0 && pg == 0) TRACE_EV(1, ptile);
            const uint32_t full = smem_u32(&ctl->pair_full[slot]);
            mbar_arrive_expect_tx(full, 2 * nbox * BOX_BYTES);
            if (row >= 0)
              for (int half = 0; half < 2; ++half) {
                const uint32_t dst = s_pair + slot * PAIR_BYTES + half * HALF_BYTES + pg * BOX_BYTES;
                if (stream_hint) tma_load_2d_hint(dst, &tm_cache, full, 64 * (2 * pr + half), row, pol_stream);
                else tma_load_2d(dst, &tm_cache, full, 64 * (2 * pr + half), row);
              }
            ++pair_i;
          }
          if (!ok) break;
          if (pg == 0) TRACE_EV(2, ptile);
          if (!K::ROPE_FIRST && !(ok = load_rope())) break;
          if (pg == 0) TRACE_EV(3, ptile);
          ++ptile;
          ++rope_i;
        }
        ++item_i;
      }
      if (!ok) {
        // Let copies already in flight land before the CTA exits (bounded: a
        // phase the other producer never arrived on does not complete).
        for (uint32_t k = 0; k < K::NP && k < pair_i; ++k) {
          const uint32_t i = pair_i - 1 - k;
          mbar_wait_ns(smem_u32(&ctl->pair_full[i % K::NP]), (i / K::NP) & 1, 20000000ull);
        }
        for (uint32_t k = 0; k < K::NR && k < rope_i; ++k) {
          const uint32_t i = rope_i - 1 - k;
          mbar_wait_ns(smem_u32(&ctl->rope_full[i % K::NR]), (i / K::NR) & 1, 20000000ull);
        }
        if (pg == 0 && item_i > 0) mbar_wait_ns(smem_u32(&ctl->q_full), (item_i - 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issues every score MMA (warp 1), another every P.C MMA (warp
    // 2, after the TMEM allocation): a thread issues one MMA per ~90 cycles
    // whatever its size, and a tile takes 68 of them, so with one issuer the
    // tensor-core instructions alone filled most of a tile's time. S is double
    // buffered in TMEM: the scores of tile i+1 go in while the softmax of tile i
    // runs. Each issuer's commits track only its own MMAs.
    if (lane == 0) {
      ItemIter it;
      it.init(p, pre, u, c);
      uint32_t n = 0;       // tile of the unit
      uint32_t item_i = 0;
      int b, t0, t1, L;
      long long acc;
      bool ok = true;
      if (warp == 1) {
        constexpr uint32_t ID_QK = idesc_bf16_f32(128, N, 0, 0);
        while (ok && it.next(b, t0, t1, L, acc)) {
          if (!(ok = mbar_wait(smem_u32(&ctl->q_full), item_i & 1, abort, p.status))) break;
          for (int tau = t0; tau < t1 && ok; ++tau, ++n) {
            // the softmax has read the scores of tile n - 2 from this buffer
            if (n >= 2 && !(ok = mbar_wait(smem_u32(&ctl->s_free[n & 1]), ((n - 2) >> 1) & 1, abort, p.status)))
              break;
            const uint32_t d_s = tmem + K::COL_S + N * (n & 1);
            // S^T = C . Q^T over the 9 column blocks of the tile (RoPE block
            // first when it is loaded first)
            const uint32_t rslot = n % K::NR;
            auto qk_rope = [&](uint32_t accumulate) -> bool {
              if (!mbar_wait(smem_u32(&ctl->rope_full[rslot]), (n / K::NR) & 1, abort, p.status)) return false;
              TRACE_EV(5, n);
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t ad = smem_desc(s_rope + rslot * HALF_BYTES + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
                const uint64_t bd = smem_desc(s_q + 8 * N * 128 + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
                mma_bf16_ss(d_s, ad, bd, ID_QK, (accumulate | k) != 0);
              }
              return true;
            };
            if (K::ROPE_FIRST && !(ok = qk_rope(0))) break;
            for (int pr = 0; pr < 4 && ok; ++pr) {
              const uint32_t i = 4 * n + pr, slot = i % K::NP;
              if (!(ok = mbar_wait(smem_u32(&ctl->pair_full[slot]), (i / K::NP) & 1, abort, p.status))) break;
              if (pr == 0) TRACE_EV(4, n);
              tc_fence_after();
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const int kb = 2 * pr + half;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = smem_desc(s_pair + slot * PAIR_BYTES + half * HALF_BYTES + 32 * k, 16, 1024,
                                                SMEM_SWIZZLE_128B);
                  const uint64_t bd = smem_desc(s_q + kb * N * 128 + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
                  mma_bf16_ss(d_s, ad, bd, ID_QK, K::ROPE_FIRST || (pr | half | k) != 0);
                }
              }
            }
            if (!ok) break;
            if (!K::ROPE_FIRST && !(ok = qk_rope(1))) break;
            mma_commit(smem_u32(&ctl->s_full[n & 1]));
            if (tau == t1 - 1) mma_commit(smem_u32(&ctl->q_empty));
          }
          ++item_i;
        }
      } else {
        constexpr uint32_t ID_PV = idesc_bf16_f32(128, N, 1, 1);
        while (ok && it.next(b, t0, t1, L, acc)) {
          for (int tau = t0; tau < t1 && ok; ++tau, ++n) {
            // O^T += C[:, :512]^T . P^T once the softmax has written P
            if (!(ok = mbar_wait(smem_u32(&ctl->p_full[n & 1]), (n >> 1) & 1, abort, p.status))) break;
            TRACE_EV(8, n);
            if (tau == t0 && item_i > 0)
              if (!(ok = mbar_wait(smem_u32(&ctl->o_empty), (item_i - 1) & 1, abort, p.status))) break;
            tc_fence_after();
            const uint32_t rslot = n % K::NR;
            const uint32_t s_p = s_rope + rslot * HALF_BYTES;
            for (int mt = 0; mt < 4; ++mt) {
              const uint32_t slot = (4 * n + mt) % K::NP;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t ad =
                    smem_desc(s_pair + slot * PAIR_BYTES + k * 2048, HALF_BYTES, 1024, SMEM_SWIZZLE_128B);
                const uint64_t bd = smem_desc(s_p + k * 16 * (2 * N), 16 * (2 * N) * 8, 16 * N, K::P_LAYOUT);
                mma_bf16_ss(tmem + mt * N, ad, bd, ID_PV, !(tau == t0 && k == 0));
              }
              mma_commit(smem_u32(&ctl->pair_empty[slot]));
            }
            mma_commit(smem_u32(&ctl->rope_empty[rslot]));
            mma_commit(smem_u32(&ctl->pc_done[n & 1]));
            TRACE_EV(9, n);
            if (tau == t1 - 1) mma_commit(smem_u32(&ctl->o_full));
          }
          ++item_i;
        }
      }
      // every MMA either thread issued has completed once mma_final flips
      mma_commit(smem_u32(&ctl->mma_final));
      mbar_wait_ns(smem_u32(&ctl->mma_final), 0, 100000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    // K::GR groups of 4 warps; group grp owns the NC columns [cb, cb + NC) of
    // S, P and O (query rows of the CTA); a thread owns one token row.
    constexpr int NC = K::NC, CW = K::CW;
    const int sw = warp & 3;                  // TMEM lane quarter
    const int grp = (warp - 4) >> 2;
    const int cb = grp * NC;
    const uint32_t gbar = 1 + grp;            // named barrier of the group
    const int t = sw * 32 + lane;             // token row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(sw * 32) << 16;
    // column cb + n sees tokens < L - dlim[n / 16] (a query token owns >= 16 columns)
    int dlim[(NC + 15) / 16];
#pragma unroll
    for (int k = 0; k < (NC + 15) / 16; ++k) dlim[k] = p.Hq - 1 - (c * N + cb + 16 * k) / p.H;

    ItemIter it;
    it.init(p, pre, u, c);
    uint32_t pair_i = 0, rope_i = 0, item_i = 0, tile_i = 0;
    int b, t0, t1, L;
    long long acc;
    const long long T = it.T;
    bool ok = true;
    float lrow[NC];
    float* m_run = ctl->m_run + cb;
    float* alpha = ctl->alpha + cb;
    while (ok && it.next(b, t0, t1, L, acc)) {
      if (t < NC) m_run[t] = -INFINITY;
      named_bar_sync(gbar, 128);
#pragma unroll
      for (int n = 0; n < NC; ++n) lrow[n] = 0.f;
      for (int tau = t0; tau < t1; ++tau) {
        if (!(ok = mbar_wait(smem_u32(&ctl->s_full[tile_i & 1]), (tile_i >> 1) & 1, abort, p.status))) break;
        if (t == 0 && grp == 0) TRACE_EV(6, tile_i);
        tc_fence_after();
        float x[NC];
        {
          uint32_t v[NC];
#pragma unroll
          for (int k = 0; k < NC / CW; ++k)
            tmem_ld_w<CW>(tmem + lane_addr + K::COL_S + N * (tile_i & 1) + cb + CW * k, v + CW * k);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < NC / CW; ++k) reg_fence_w<CW>(v + CW * k);
#pragma unroll
          for (int i = 0; i < NC; ++i) x[i] = __uint_as_float(v[i]);
        }
        // this S buffer may take the scores of tile i + 2
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[tile_i & 1]));
        const int tok = tau * TILE + t;
        bool need = false;
#pragma unroll
        for (int n = 0; n < NC; ++n) {
          x[n] = (tok < L - dlim[n / 16]) ? x[n] * p.scale_log2 : -INFINITY;
          need |= x[n] > m_run[n] + RESCALE_LOG2;
        }
        const int vote = __any_sync(0xffffffffu, need);
        if (lane == 0) ctl->vote[grp][tile_i & 1][sw] = vote;
        named_bar_sync(gbar, 128);
        const int* vv = ctl->vote[grp][tile_i & 1];
        if (vv[0] | vv[1] | vv[2] | vv[3]) {
          // new running max per column, rescale l and O by alpha
#pragma unroll
          for (int n = 0; n < NC; ++n) {
            float v = x[n];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) ctl->red[sw][cb + n] = v;
          }
          named_bar_sync(gbar, 128);
          if (t < NC) {
            const int n = cb + t;
            const float mt = fmaxf(fmaxf(ctl->red[0][n], ctl->red[1][n]), fmaxf(ctl->red[2][n], ctl->red[3][n]));
            const float mo = m_run[t];
            const float mn = fmaxf(mo, mt);
            alpha[t] = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
            m_run[t] = mn;
          }
          named_bar_sync(gbar, 128);
#pragma unroll
          for (int n = 0; n < NC; ++n) lrow[n] *= alpha[n];
          if (tau != t0) {
            // the previous tile's P.C products are in O (their issuer is not
            // the one whose commit signalled these scores)
            if (!(ok = mbar_wait(smem_u32(&ctl->pc_done[(tile_i - 1) & 1]), ((tile_i - 1) >> 1) & 1, abort, p.status)))
              break;
            tc_fence_after();
#pragma unroll 1
            for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
              for (int k = 0; k < NC / CW; ++k) {
                uint32_t v[CW];
                const uint32_t ta = tmem + lane_addr + mt * N + cb + CW * k;
                tmem_ld_w<CW>(ta, v);
                tmem_wait_ld();
                reg_fence_w<CW>(v);
#pragma unroll
                for (int i = 0; i < CW; ++i)
                  v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha[CW * k + i]);
                tmem_st_w<CW>(ta, v);
              }
            }
            tmem_wait_st();
          }
        }
        // P = exp2(x - m), rounded to bf16; l accumulates the rounded values
        // P row of this token: N bf16 (2N bytes) in the MN-major swizzled
        // layout the P.C MMA reads (16-byte chunk c of row t at c ^ swz(t));
        // this group writes chunks [cb/8, (cb + NC)/8).
        const uint32_t s_p = s_rope + (rope_i % K::NR) * HALF_BYTES;
        const uint32_t prow = s_p + t * (2 * N);
        const uint32_t pswz = ((t * 2 * N) >> 7) & (K::P_CHUNKS - 1);
#pragma unroll
        for (int c8 = 0; c8 < NC / 8; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n0 = 8 * c8 + 2 * i;
            const float m0 = m_run[n0], m1 = m_run[n0 + 1];
            const float p0 = fast_exp2(x[n0] - (m0 == -INFINITY ? 0.f : m0));
            const float p1 = fast_exp2(x[n0 + 1] - (m1 == -INFINITY ? 0.f : m1));
            w[i] = pack_bf16x2(p0, p1);
            lrow[n0] += __uint_as_float(w[i] << 16);
            lrow[n0 + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
          }
          const uint32_t addr = prow + (((cb / 8 + c8) ^ pswz) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
        if (L - tau * TILE < TILE) {
          // Cache rows past the sequence end may hold anything: zero them so
          // that 0 * garbage cannot reach the P.C product. Every softmax thread
          // takes 16-byte chunks in order (eight consecutive threads fill one
          // 128-byte row segment), so a warp's stores hit distinct banks.
          const int r0 = L - tau * TILE > 0 ? L - tau * TILE : 0;
          const int total = (TILE - r0) * 64;        // 64 chunks per row (8 halves x 8)
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
          for (int idx = grp * 128 + t; idx < total; idx += 128 * K::GR) {
            const int row = r0 + (idx >> 6), h = (idx >> 3) & 7;
            const uint32_t a = s_pair + ((pair_i + (h >> 1)) % K::NP) * PAIR_BYTES + (h & 1) * HALF_BYTES + row * 128 +
                               (idx & 7) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(z.x), "r"(z.y), "r"(z.z), "r"(z.w)
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[tile_i & 1]));
        if (t == 0 && grp == 0) TRACE_EV(7, tile_i);
        pair_i += 4;
        ++rope_i;
        ++tile_i;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait(smem_u32(&ctl->o_full), item_i & 1, abort, p.status))) break;
      tc_fence_after();
#pragma unroll
      for (int n = 0; n < NC; ++n) {
        float v = lrow[n];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ctl->red[sw][cb + n] = v;
      }
      named_bar_sync(gbar, 128);
      if (t < NC) {
        const int n = cb + t;
        const float l = (ctl->red[0][n] + ctl->red[1][n]) + (ctl->red[2][n] + ctl->red[3][n]);
        ctl->lsum[n] = l;
        ctl->linv[n] = l > 0.f ? 1.f / l : 0.f;
      }
      named_bar_sync(gbar, 128);
      const int nt = ntiles(L);
      const bool final_out = unit_of(acc, T, p.U) == unit_of(acc + nt - 1, T, p.U);
      const long long row0 = final_out ? (long long)b * p.G + c * N : ((long long)(b + u)) * p.G + c * N;
      float* obase = (final_out ? p.o_lat : p.ws_o) + (row0 + cb) * D_C;
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t v[NC];
#pragma unroll
        for (int k = 0; k < NC / CW; ++k) tmem_ld_w<CW>(tmem + lane_addr + mt * N + cb + CW * k, v + CW * k);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < NC / CW; ++k) reg_fence_w<CW>(v + CW * k);
#pragma unroll
        for (int n = 0; n < NC; ++n)
          __stcg(obase + (long long)n * D_C + mt * 128 + t, __uint_as_float(v[n]) * ctl->linv[cb + n]);
      }
      if (t < NC) {
        const float l = ctl->lsum[cb + t];
        const float lse = l > 0.f ? (m_run[t] + __log2f(l)) * LN2 : -INFINITY;
        (final_out ? p.lse : p.ws_lse)[row0 + cb + t] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->o_empty));
      named_bar_sync(gbar, 128);
      ++item_i;
    }
  }

  if (threadIdx.x == 128) TRACE_CTA(2);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, K::TMEM_COLS);
  }
  if (threadIdx.x == 64) TRACE_CTA(3);
}

// Merge the partials of sequences that were cut across units:
// lse = log sum_k exp(lse_k), o = sum_k exp(lse_k - lse) o_k.
__global__ void __launch_bounds__(256) combine_kernel(AttnParams p) {
  const int b = blockIdx.x;
  const int g = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  __shared__ long long sums[2][8];
  TRACE_COMB(0);
  pdl_trigger();
  // The tile bookkeeping depends only on the sequence lengths (a call input):
  // T = all tiles, acc = tiles of the sequences before b, computed while the
  // attention kernel finishes.
  long long tot = 0, before = 0;
  for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
    const int n = ntiles(seq_len(p.seq_lens, p.Hq, i));
    tot += n;
    if (i < b) before += n;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
  }
  if (lane == 0) {
    sums[0][threadIdx.x >> 5] = tot;
    sums[1][threadIdx.x >> 5] = before;
  }
  __syncthreads();
  long long T = 0, acc = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    T += sums[0][w];
    acc += sums[1][w];
  }
  const int nt = ntiles(seq_len(p.seq_lens, p.Hq, b));
  pdl_wait();
  TRACE_COMB(1);
  if (g >= p.G) return;
  float4* dst = reinterpret_cast<float4*>(p.o_lat + ((long long)b * p.G + g) * D_C);
  if (nt == 0) {
    // length below the number of query tokens: no attention is defined
    for (int i = lane; i < D_C / 4; i += 32) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) {
      p.lse[(long long)b * p.G + g] = -INFINITY;
      atomicOr(p.status, MLA_DEVERR_LENGTH);
    }
    return;
  }
  const int uf = unit_of(acc, T, p.U), ul = unit_of(acc + nt - 1, T, p.U);
  if (uf == ul) return;
  // Units between uf and ul with an empty tile range (possible when there are
  // more units than tiles) wrote nothing and are skipped.
  auto empty_unit = [&](int k) { return unit_start(k + 1, T, p.U) == unit_start(k, T, p.U); };
  // One pass over the pieces, four at a time with all their loads issued
  // before use: running max m, running sum z and accumulator a are rescaled
  // as the max grows (the same online rule as the attention softmax).
  float m = -INFINITY, z = 0.f;
  float4 a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  int k = uf;
  while (k <= ul) {
    int ks[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      while (k <= ul && empty_unit(k)) ++k;
      ks[j] = k <= ul ? k : -1;
      ++k;
    }
    float lk[4];
    float4 v[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lk[j] = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[j][i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ks[j] >= 0) {
        const long long r = ((long long)(b + ks[j])) * p.G + g;
        lk[j] = __ldcg(p.ws_lse + r);
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + r * D_C);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[j][i] = __ldcg(src + lane + 32 * i);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float mn = fmaxf(m, lk[j]);
      if (mn == -INFINITY) continue;
      const float sc = __expf(m - mn), w = __expf(lk[j] - mn);
      z = z * sc + w;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i].x = a[i].x * sc + w * v[j][i].x;
        a[i].y = a[i].y * sc + w * v[j][i].y;
        a[i].z = a[i].z * sc + w * v[j][i].z;
        a[i].w = a[i].w * sc + w * v[j][i].w;
      }
      m = mn;
    }
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = make_float4(a[i].x * inv, a[i].y * inv, a[i].z * inv, a[i].w * inv);
  if (lane == 0) p.lse[(long long)b * p.G + g] = z > 0.f ? m + __logf(z) : -INFINITY;
  TRACE_COMB(2);
}

size_t attn_smem_bytes(int N) {
  const size_t extra = sizeof(Ctrl) + sizeof(int) * (MAX_SEQS + 1) + 1024;
  switch (N) {
    case 16: return Cfg<16>::OFF_CTRL + extra;
    case 32: return Cfg<32>::OFF_CTRL + extra;
    case 64: return Cfg<64>::OFF_CTRL + extra;
    default: return 0;
  }
}

cudaError_t attn_prepare(int N) {
  const int smem = static_cast<int>(attn_smem_bytes(N));
  switch (N) {
    case 16: return cudaFuncSetAttribute(decode_attn_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 32: return cudaFuncSetAttribute(decode_attn_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 64: return cudaFuncSetAttribute(decode_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_attn(const CUtensorMap& tm_cache, const CUtensorMap& tm_q, const AttnParams& p,
                               cudaStream_t s) {
  if (p.B > MAX_SEQS) return cudaErrorInvalidValue;
  const size_t smem = attn_smem_bytes(p.N);
  const dim3 grid(p.U * p.C);
  switch (p.N) {
    case 16: return launch_pdl(decode_attn_kernel<16>, grid, dim3(Cfg<16>::THREADS), smem, s, tm_cache, tm_q, p);
    case 32: return launch_pdl(decode_attn_kernel<32>, grid, dim3(Cfg<32>::THREADS), smem, s, tm_cache, tm_q, p);
    case 64: return launch_pdl(decode_attn_kernel<64>, grid, dim3(Cfg<64>::THREADS), smem, s, tm_cache, tm_q, p);
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const AttnParams& p, cudaStream_t s) {
  const dim3 grid(p.B, (p.G + 7) / 8);
  return launch_pdl(combine_kernel, grid, dim3(256), 0, s, p);
}

}  // namespace mla
