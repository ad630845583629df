// Absorbed-MLA decode attention for query-row groups of 128 (H = 128, or
// several query tokens per sequence) on CTA pairs: the 2-SM tensor-core path.
//
// What is computed is the same as decode_attn.cu ("DeepSeek MLA 吸收式缓存"
// §2.2-§2.3, §6.1 MQA mode; "80 行 PyTorch 从零写 DeepSeek 的 MLA" §5): per query
// row g, scores s_t = scale * q_abs[g] . row_t over the 576-wide cache rows,
// bottom-right causal softmax, o_lat = sum_t p_t c_kv_t and lse.
//
// Layout of the work. A pair of CTAs (a cluster of two) owns 128 query rows;
// CTA r of the pair holds the 72 KB of queries of its 64 rows and its own
// copy of every 128-token cache tile (the second copy comes from L2).
//  * Scores: one pair MMA per 16 columns, M = 256 (128 tokens in each CTA),
//    N = 128 (64 query rows from each CTA's shared memory). Each CTA's tensor
//    memory receives the scores of all 128 rows for its copy of the tokens; the
//    columns of its own 64 rows are the ones it uses.
//  * Softmax: each CTA on its own 64 rows (four groups of four warps, one token
//    row per thread, fp32, lazy rescale at 2^8), P^T written to its shared
//    memory: the two CTAs' P^T are the two N halves of the next MMA's B.
//  * P.C: pair MMAs with M = 256 over the latent dimension: CTA r supplies the
//    latent blocks {256 j + 128 r, ...} (j = 0, 1) of its tile copy, so CTA r
//    accumulates O^T for those 256 latent columns of all 128 rows (256 TMEM
//    columns), next to the 128 score columns. For this the two copies of a
//    tile sit in shared memory with their 128-column latent blocks swapped in
//    pairs (CTA 1: 1,0,3,2), and each CTA's queries are permuted the same way,
//    so every score column a CTA uses pairs its rows with matching key columns.
//  * The latent blocks a CTA uses only for scores (two of its four) are
//    released right after the score MMAs: the next tile's loads into them
//    overlap the softmax and P.C of the current one.
//  * Rescaling: a row's running max lives in the CTA that owns the row, but its
//    O columns live in both CTAs. Each softmax group sends its 16 factors (1:
//    none) to the peer with st.async (asynchronous stores into the peer's
//    shared memory, counted on the peer's mbarrier); the peer rescales those
//    columns before it lets the next P.C start. The row sums go the same way
//    right after an item's last softmax, so the exchange hides behind the last
//    P.C.
//  * The even CTA of the pair issues every MMA, from two threads (one for the
//    scores, one for P.C); both CTAs' TMA loads count on its mbarriers, and
//    the peer's P-ready and O-drained signals reach them as 4-byte st.async
//    stores (a remote mbarrier arrival stalls the arriving warp for ~1k
//    cycles). MMA completions are multicast to both CTAs' barriers.
//  * A long prompt chunk runs as one unit: when it has more row-group pairs
//    than fit at once, the pairs that fit each walk several of them.
#include "attn_sched.cuh"
#include "launch_once.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase trace (compile with -DMLA_TRACE=1): SM clock stamps of the
// pipeline events of the first tiles of the first CTAs, and per-CTA start and
// end times, read back with mla_pair_trace_read(). Off in normal builds.
#ifndef MLA_TRACE
#define MLA_TRACE 0
#endif
#if MLA_TRACE
#define PT_CTAS 8
#define PT_TILES 32
#define PT_EVENTS 16
__device__ long long g_pair_trace[PT_CTAS][PT_TILES][PT_EVENTS];
__device__ unsigned long long g_pair_cta[1024][4];
#define PTRACE(ev, tile)                                                    \
  do {                                                                      \
    if (blockIdx.x < PT_CTAS && (tile) < PT_TILES)                          \
      g_pair_trace[blockIdx.x][(tile)][(ev)] = clock64();                   \
  } while (0)
#define PTRACE_CTA(ev, v)                                  \
  do {                                                     \
    if (blockIdx.x < 1024) g_pair_cta[blockIdx.x][(ev)] = (v); \
  } while (0)
extern "C" int mla_pair_trace_read(void* trace, size_t tbytes, void* cta, size_t cbytes) {
  if (tbytes > sizeof(g_pair_trace)) tbytes = sizeof(g_pair_trace);
  if (cbytes > sizeof(g_pair_cta)) cbytes = sizeof(g_pair_cta);
  cudaError_t e = cudaMemcpyFromSymbol(trace, g_pair_trace, tbytes);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(cta, g_pair_cta, cbytes);
  return (int)e;
}
#else
#define PTRACE(ev, tile) \
  do {                   \
  } while (0)
#define PTRACE_CTA(ev, v) \
  do {                    \
  } while (0)
#endif

namespace mla {

namespace {

constexpr int PN = 64;                      // query rows per CTA
constexpr int PGR = 4;                      // softmax groups (four warps each)
constexpr int PNC = PN / PGR;               // own columns per group
constexpr int PTHREADS = 128 + 128 * PGR;   // 640
constexpr float P_LN2 = 0.6931471805599453f;
constexpr float P_RESCALE_LOG2 = 8.0f;
constexpr uint32_t P_PAIR_BYTES = 32768;    // 128 tokens x 128 latent columns
constexpr uint32_t P_HALF_BYTES = 16384;    // 128 tokens x 64 columns
constexpr uint32_t P_BOX_BYTES = 8192;      // 64 tokens x 64 columns (one TMA box)
constexpr uint32_t PQ_BYTES = 9u * PN * 128u;
constexpr uint32_t POFF_PAIR = PQ_BYTES;
constexpr uint32_t POFF_ROPE = POFF_PAIR + 4 * P_PAIR_BYTES;
constexpr uint32_t POFF_CTRL = POFF_ROPE + P_HALF_BYTES;
constexpr uint32_t PCOL_S = 256;            // two score buffers (128 columns each); O^T halves at 0 and 128
constexpr uint32_t PTMEM_COLS = 512;
constexpr uint16_t BOTH = 3;                // multicast mask: both CTAs of the pair

struct __align__(16) PairCtrl {
  uint64_t q_full, q_empty;
  uint64_t pair_full[4], pair_empty[4];
  uint64_t rope_full, rope_empty;
  uint64_t s_full, o_full, o_empty, mma_final;
  uint64_t p_full[2], pc_done[2];   // by tile parity: P written (both CTAs) / P.C done
  uint64_t xch_full[2], l_full[2];
  uint32_t tmem_base;
  int abort;
  int vote[PGR][2][4];
  alignas(16) float xalpha[2][PN];   // written by the peer: its rows' rescale factors (1: none)
  float xl[2][PN];          // written by the peer: its rows' softmax sums (by item parity;
                            // the peer can be one item ahead)
  float lsum[PN];           // this CTA's rows' softmax sums
  uint32_t sink[2][4 * PGR];   // landing words of the peer's P-ready / O-drained signals (leader)
  float m_run[PN];
  float alpha[PN];
  float red[4][PN];
  float linv[2 * PN];       // by pair column (128 rows)
  int warp_tot[32];
};
static_assert(POFF_CTRL % 1024 == 0, "control block after the swizzled slots");

// Latent block (of four, 128 columns each) held in slot s by CTA r of the pair.
MLA_DEV int slot_block(int r, int s) { return r ? (s ^ 1) : s; }
// Order in which a tile's latent slots are filled and consumed by the scores:
// the score-only slots 1 and 3 first (they are free earliest), then the P.C
// slots 0 and 2.
MLA_DEV int slot_order(int si) { return si < 2 ? 2 * si + 1 : 2 * si - 4; }

// The items a pair walks, with the row group c of each. Normally the pair's
// one row group (both CTAs walk the tiles of its later row group's causal
// limit). With one unit launched on p.slots pairs (a long prompt chunk with
// more row-group pairs than fit at once), pair k takes the row-group pairs of
// the latest query tokens first, k, k + slots, k + 2 slots, ... in that order,
// so the epilogue of one overlaps the loads and scores of the next.
struct PairWalk {
  ItemIter it;
  const AttnParams* pp;
  const int* pre;
  int u, r, c, j, jstep, npairs;
  bool many, have;
  MLA_DEV void init(const AttnParams& p, const int* pre_, int u_, int r_, int c_fixed) {
    pp = &p;
    pre = pre_;
    u = u_;
    r = r_;
    many = p.U == 1 && p.slots > 0;
    npairs = p.C / 2;
    if (many) {
      j = blockIdx.x / 2;
      jstep = gridDim.x / 2;
      have = j < npairs;
      c = 2 * (npairs - 1 - j) + r;
    } else {
      have = true;
      c = c_fixed;
    }
    if (have) it.init(p, pre, u, c | 1);
  }
  MLA_DEV bool next(int& b, int& t0, int& t1, int& L, long long& acc) {
    while (have) {
      if (it.next(b, t0, t1, L, acc)) return true;
      if (!many) return false;
      j += jstep;
      have = j < npairs;
      if (!have) return false;
      c = 2 * (npairs - 1 - j) + r;
      it.init(*pp, pre, u, c | 1);
    }
    return false;
  }
};

}  // namespace

__global__ void __launch_bounds__(PTHREADS, 1)
    decode_attn_pair_kernel(const __grid_constant__ CUtensorMap tm_cache, const __grid_constant__ CUtensorMap tm_q,
                            const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  PairCtrl* ctl = reinterpret_cast<PairCtrl*>(smem + POFF_CTRL);
  int* pre = reinterpret_cast<int*>(smem + POFF_CTRL + sizeof(PairCtrl));
  const uint32_t s_q = smem_u32(smem);
  const uint32_t s_pair = s_q + POFF_PAIR;
  const uint32_t s_rope = s_q + POFF_ROPE;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.C;        // unit
  // 64-row group within the unit. With one unit (a long prompt chunk, its
  // pairs in waves) the pairs of the latest query tokens, which see the most
  // tiles, are launched first: longest first packs the waves.
  const int c_launch = blockIdx.x % p.C;
  const int c = p.U == 1 ? (p.C - 2 - (c_launch & ~1)) + (c_launch & 1) : c_launch;
  const int r = static_cast<int>(cluster_ctarank());   // == c & 1
  const int peer = r ^ 1;
  volatile int* abort = &ctl->abort;
  auto at_leader = [&](const void* x) { return mapa_shared(smem_u32(x), 0); };
  auto at_peer = [&](const void* x) { return mapa_shared(smem_u32(x), peer); };

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_full), 1);
    mbar_init(smem_u32(&ctl->q_empty), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(smem_u32(&ctl->pair_full[i]), 2);   // the leader's two producers (one per page)
      mbar_init(smem_u32(&ctl->pair_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctl->rope_full), 2);
    mbar_init(smem_u32(&ctl->rope_empty), 1);
    mbar_init(smem_u32(&ctl->s_full), 1);
    // P-ready / O-drained: one arrival per warp of the leader's softmax groups,
    // and 4 bytes (st.async) per warp of the peer's
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->p_full[i]), 4 * PGR);
      mbar_init(smem_u32(&ctl->pc_done[i]), 1);
    }
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->o_empty), 4 * PGR);
    mbar_init(smem_u32(&ctl->mma_final), 2);   // the leader's two MMA issuers
    mbar_init(smem_u32(&ctl->xch_full[0]), PGR);
    mbar_init(smem_u32(&ctl->xch_full[1]), PGR);
    mbar_init(smem_u32(&ctl->l_full[0]), PGR);
    mbar_init(smem_u32(&ctl->l_full[1]), PGR);
    ctl->abort = 0;
    fence_mbar_init();
    // each softmax group expects its 16 factors (64 bytes) from the peer per use
    for (int g = 0; g < PGR; ++g) {
      mbar_arrive_expect_tx(smem_u32(&ctl->xch_full[0]), 4 * PNC);
      mbar_arrive_expect_tx(smem_u32(&ctl->xch_full[1]), 4 * PNC);
      mbar_arrive_expect_tx(smem_u32(&ctl->l_full[0]), 4 * PNC);   // and its 16 softmax sums per item
      mbar_arrive_expect_tx(smem_u32(&ctl->l_full[1]), 4 * PNC);
    }
    tma_prefetch_desc(&tm_cache);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(&ctl->tmem_base), PTMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either CTA signals the other's
  cluster_sync();
  if (threadIdx.x == 0) {
    PTRACE_CTA(0, (unsigned long long)clock64());
    PTRACE_CTA(1, globaltimer());
  }
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  tile_prefix(p, pre, ctl->warp_tot);
  pdl_wait();


  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers (each CTA, its own copy)
    // One thread per 64-token page of each tile (warp 0: the first page and
    // the queries, warp 3: the second page): one issuing thread keeps too few
    // 8 KB boxes moving to fill an SM at its share of the bandwidth. The
    // leader's two producers each expect their page's bytes of both CTAs.
    if (lane == 0) {
      const int pg = warp == 0 ? 0 : 1;
      PairWalk it;
      it.init(p, pre, u, r, c);
      uint32_t item_i = 0, ptile = 0;
      int b, t0, t1, L;
      long long acc;
      bool ok = true;
      const uint32_t qf = at_leader(&ctl->q_full);
      while (ok && it.next(b, t0, t1, L, acc)) {
        if (pg == 0) {
          if (!(ok = mbar_wait(smem_u32(&ctl->q_empty), (item_i & 1) ^ 1, abort, p.status))) break;
          if (r == 0) mbar_arrive_expect_tx(smem_u32(&ctl->q_full), 2 * PQ_BYTES);
          for (int kp = 0; kp < 9; ++kp) {
            const int kb = kp < 8 ? 2 * slot_block(r, kp >> 1) + (kp & 1) : 8;
            tma_load_2d_pair(s_q + kp * PN * 128, &tm_q, qf, 64 * kb, b * p.G + it.c * PN);
          }
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
          const uint32_t par = (ptile & 1) ^ 1;
          for (int si = 0; si < 4 && ok; ++si) {
            const int slot = slot_order(si);
            if (!(ok = mbar_wait(smem_u32(&ctl->pair_empty[slot]), par, abort, p.status))) break;
            if (r == 0) mbar_arrive_expect_tx(smem_u32(&ctl->pair_full[slot]), 2 * 2 * nbox * P_BOX_BYTES);
            const uint32_t full = at_leader(&ctl->pair_full[slot]);
            const int blk = slot_block(r, slot);
            if (row >= 0)
              for (int half = 0; half < 2; ++half)
                tma_load_2d_pair(s_pair + slot * P_PAIR_BYTES + half * P_HALF_BYTES + pg * P_BOX_BYTES, &tm_cache,
                                 full, 64 * (2 * blk + half), row);
          }
          if (!ok) break;
          if (!(ok = mbar_wait(smem_u32(&ctl->rope_empty), par, abort, p.status))) break;
          if (r == 0) mbar_arrive_expect_tx(smem_u32(&ctl->rope_full), 2 * nbox * P_BOX_BYTES);
          const uint32_t rfull = at_leader(&ctl->rope_full);
          if (row >= 0) tma_load_2d_pair(s_rope + pg * P_BOX_BYTES, &tm_cache, rfull, D_C, row);
          ++ptile;
        }
        ++item_i;
      }
      if (!ok) {
        // copies in flight count on the leader's barriers: give them time to land
        const uint64_t t_0 = globaltimer();
        while (globaltimer() - t_0 < 2000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers (the pair's even CTA)
    // Warp 1 issues the score MMAs, warp 2 (after the TMEM allocation) the P.C
    // MMAs: a thread issues one tcgen05.mma per ~90 cycles, so with one issuer
    // a tile's scores and the previous tile's P.C queued behind each other.
    // The scores of a tile go to TMEM buffer n & 1 once both CTAs' softmax has
    // signalled P of tile n - 2 (it had read those scores before).
    if (lane == 0 && r == 0) {
      PairWalk it;
      it.init(p, pre, u, r, c);
      uint32_t n = 0, item_i = 0;
      int b, t0, t1, L;
      long long acc;
      bool ok = true;
      if (warp == 1) {
        constexpr uint32_t ID_S = idesc_bf16_f32(256, 128, 0, 0);
        while (ok && it.next(b, t0, t1, L, acc)) {
          if (!(ok = mbar_wait(smem_u32(&ctl->q_full), item_i & 1, abort, p.status))) break;
          for (int tau = t0; tau < t1 && ok; ++tau, ++n) {
            const uint32_t par = n & 1;
            if (n >= 2 && !(ok = mbar_wait_cluster(smem_u32(&ctl->p_full[par]), ((n - 2) >> 1) & 1, abort, p.status)))
              break;
            const uint32_t d_s = tmem + PCOL_S + 128 * par;
            // the score-only slots 1 and 3 (released as soon as their MMAs
            // complete), then the P.C slots 0 and 2 and the RoPE block
            for (int si = 0; si < 4 && ok; ++si) {
              const int slot = slot_order(si);
              if (!(ok = mbar_wait(smem_u32(&ctl->pair_full[slot]), par, abort, p.status))) break;
              if (si == 0) PTRACE(0, n);
              if (si == 2) PTRACE(11, n);
              tc_fence_after();
#pragma unroll
              for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = smem_desc(s_pair + slot * P_PAIR_BYTES + half * P_HALF_BYTES + 32 * k, 16, 1024,
                                                SMEM_SWIZZLE_128B);
                  const uint64_t bd =
                      smem_desc(s_q + (2 * slot + half) * PN * 128 + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
                  mma_bf16_ss_pair(d_s, ad, bd, ID_S, (si == 0 && half == 0 && k == 0) ? 0u : 1u);
                }
              if (si < 2) mma_commit_pair(smem_u32(&ctl->pair_empty[slot]), BOTH);
            }
            if (!ok) break;
            if (!(ok = mbar_wait(smem_u32(&ctl->rope_full), par, abort, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc(s_rope + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
              const uint64_t bd = smem_desc(s_q + 8 * PN * 128 + 32 * k, 16, 1024, SMEM_SWIZZLE_128B);
              mma_bf16_ss_pair(d_s, ad, bd, ID_S, 1u);
            }
            mma_commit_pair(smem_u32(&ctl->s_full), BOTH);
            PTRACE(1, n);
            if (tau == t1 - 1) mma_commit_pair(smem_u32(&ctl->q_empty), BOTH);
          }
          ++item_i;
        }
      } else {
        constexpr uint32_t ID_PV = idesc_bf16_f32(256, 128, 1, 1);
        while (ok && it.next(b, t0, t1, L, acc)) {
          for (int tau = t0; tau < t1 && ok; ++tau, ++n) {
            // O^T += C[:, latent blocks]^T . P^T once both CTAs have written P
            if (!(ok = mbar_wait_cluster(smem_u32(&ctl->p_full[n & 1]), (n >> 1) & 1, abort, p.status))) break;
            PTRACE(2, n);
            if (tau == t0 && item_i > 0)
              if (!(ok = mbar_wait_cluster(smem_u32(&ctl->o_empty), (item_i - 1) & 1, abort, p.status))) break;
            tc_fence_after();
            for (int j = 0; j < 2; ++j) {
              const int slot = 2 * j;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t ad =
                    smem_desc(s_pair + slot * P_PAIR_BYTES + k * 2048, P_HALF_BYTES, 1024, SMEM_SWIZZLE_128B);
                const uint64_t bd = smem_desc(s_rope + k * 16 * 128, 16 * 128 * 8, 16 * PN, SMEM_SWIZZLE_128B);
                mma_bf16_ss_pair(tmem + 128 * j, ad, bd, ID_PV, (tau == t0 && k == 0) ? 0u : 1u);
              }
              mma_commit_pair(smem_u32(&ctl->pair_empty[slot]), BOTH);
            }
            mma_commit_pair(smem_u32(&ctl->rope_empty), BOTH);
            mma_commit_pair(smem_u32(&ctl->pc_done[n & 1]), BOTH);
            if (tau == t1 - 1) mma_commit_pair(smem_u32(&ctl->o_full), BOTH);
            PTRACE(3, n);
          }
          ++item_i;
        }
      }
      // every MMA either thread issued has completed once mma_final flips
      mma_commit_pair(smem_u32(&ctl->mma_final), 1);
      mbar_wait_ns(smem_u32(&ctl->mma_final), 0, 100000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue (each CTA, own rows)
    const int sw = warp & 3;                 // TMEM lane quarter
    const int grp = (warp - 4) >> 2;
    const int cb = grp * PNC;                // own columns [cb, cb + 16)
    const uint32_t gbar = 1 + grp;
    const int t = sw * 32 + lane;            // token row of the tile / latent row of O^T
    const uint32_t lane_addr = static_cast<uint32_t>(sw * 32) << 16;
    const uint32_t col_own = 64 * r + cb;    // pair column of this group's own rows
    const uint32_t col_peer = 64 * peer + cb;
    const uint32_t p_full_l[2] = {at_leader(&ctl->p_full[0]), at_leader(&ctl->p_full[1])};
    const uint32_t o_empty_l = at_leader(&ctl->o_empty);
    const int wi = warp - 4;   // softmax warp index (0..15)
    // Signal of one softmax warp to the leader's barrier `bar` (index kind of
    // the landing words): a local arrival in the leader (the first warp also
    // announces the peer's 64 bytes), a 4-byte st.async from the peer.
    auto signal_leader = [&](uint64_t* bar, uint32_t bar_l, int kind) {
      if (r == 0) {
        if (wi == 0) mbar_arrive_expect_tx(smem_u32(bar), 4 * 4 * PGR);
        else mbar_arrive(smem_u32(bar));
      } else {
        st_async_u32(at_leader(&ctl->sink[kind][wi]), bar_l, 1u);
      }
    };

    PairWalk it;
    it.init(p, pre, u, r, c);
    uint32_t item_i = 0, tile_i = 0;
    int b, t0, t1, L;
    long long acc;
    const long long T = it.it.T;
    bool ok = true;
    float lrow[PNC];
    float* m_run = ctl->m_run + cb;
    float* alpha = ctl->alpha + cb;
    // O holds the previous tile's P.C products (issued by a thread other than
    // the one whose commit signalled the scores) before it is rescaled
    auto wait_pc = [&]() -> bool {
      if (!mbar_wait(smem_u32(&ctl->pc_done[(tile_i - 1) & 1]), ((tile_i - 1) >> 1) & 1, abort, p.status)) return false;
      tc_fence_after();
      return true;
    };
    while (ok && it.next(b, t0, t1, L, acc)) {
      const int dlim = p.Hq - 1 - (it.c * PN + cb) / p.H;   // a query token owns >= 16 rows
      if (t < PNC) m_run[t] = -INFINITY;
      named_bar_sync(gbar, 128);
#pragma unroll
      for (int n = 0; n < PNC; ++n) lrow[n] = 0.f;
      for (int tau = t0; tau < t1; ++tau) {
        const uint32_t k2 = tile_i & 1;
        bool pc_seen = false;
        if (!(ok = mbar_wait(smem_u32(&ctl->s_full), k2, abort, p.status))) break;
        if (grp == 0 && t == 0) PTRACE(7, tile_i);
        tc_fence_after();
        float x[PNC];
        {
          uint32_t v[PNC];
          tmem_ld16(tmem + lane_addr + PCOL_S + 128 * k2 + col_own, *reinterpret_cast<uint32_t(*)[16]>(v));
          tmem_wait_ld();
          reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v));
#pragma unroll
          for (int i = 0; i < PNC; ++i) x[i] = __uint_as_float(v[i]);
        }
        if (grp == 0 && t == 0) PTRACE(4, tile_i);
        const int tok = tau * TILE + t;
        const bool live = tok < L - dlim;
        float mr[PNC];   // the running max as it stands
        bool need = false;
#pragma unroll
        for (int n = 0; n < PNC; ++n) {
          mr[n] = m_run[n];
          x[n] = live ? x[n] * p.scale_log2 : -INFINITY;
          need |= x[n] > mr[n] + P_RESCALE_LOG2;
        }
        const int vote = __any_sync(0xffffffffu, need);
        if (lane == 0) ctl->vote[grp][k2][sw] = vote;
        // P = exp2(x - m) in bf16 (ls sums the rounded values), written as the
        // 128-byte rows of P^T (16-byte chunk q of row t at q ^ (t & 7))
        const uint32_t prow = s_rope + t * 128;
        const uint32_t pswz = t & 7;
        float ls[PNC];
        auto write_p = [&]() {
#pragma unroll
          for (int c8 = 0; c8 < PNC / 8; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int n0 = 8 * c8 + 2 * i;
              const float m0 = mr[n0], m1 = mr[n0 + 1];
              const float p0 = fast_exp2(x[n0] - (m0 == -INFINITY ? 0.f : m0));
              const float p1 = fast_exp2(x[n0 + 1] - (m1 == -INFINITY ? 0.f : m1));
              w[i] = pack_bf16x2(p0, p1);
              ls[n0] = __uint_as_float(w[i] << 16);
              ls[n0 + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
            const uint32_t addr = prow + ((((uint32_t)cb / 8 + c8) ^ pswz) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                         : "memory");
          }
        };
        named_bar_sync(gbar, 128);
        const int* vv = ctl->vote[grp][k2];
        const int gvote = vv[0] | vv[1] | vv[2] | vv[3];
        if (grp == 0 && t == 0) PTRACE(5, tile_i);
        if (gvote) {
#pragma unroll
          for (int n = 0; n < PNC; ++n) {
            float v = x[n];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) ctl->red[sw][cb + n] = v;
          }
          named_bar_sync(gbar, 128);
          if (t < PNC) {
            const int n = cb + t;
            const float mt = fmaxf(fmaxf(ctl->red[0][n], ctl->red[1][n]), fmaxf(ctl->red[2][n], ctl->red[3][n]));
            const float mo = m_run[t];
            const float mn = fmaxf(mo, mt);
            alpha[t] = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
            m_run[t] = mn;
          }
          named_bar_sync(gbar, 128);
#pragma unroll
          for (int n = 0; n < PNC; ++n) {
            lrow[n] *= alpha[n];
            mr[n] = m_run[n];
          }
        }
        // publish this group's rescale factors (1: none) to the peer CTA, which
        // holds the other latent half of these rows' O columns: as soon as they
        // are known, so that they travel while P is computed here
        if (sw == 0 && lane < PNC / 4) {
          uint32_t a[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = __float_as_uint(gvote ? alpha[4 * lane + i] : 1.f);
          st_async_v4(at_peer(&ctl->xalpha[k2][cb + 4 * lane]), at_peer(&ctl->xch_full[k2]), a[0], a[1], a[2], a[3]);
        }
        if (gvote) {
          if (tau != t0) {
            if (!(ok = wait_pc())) break;
            pc_seen = true;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t v[16];
              const uint32_t ta = tmem + lane_addr + 128 * j + col_own;
              tmem_ld16(ta, v);
              tmem_wait_ld();
              reg_fence16(v);
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha[i]);
              tmem_st16(ta, v);
            }
            tmem_wait_st();
          }
        }
        write_p();
#pragma unroll
        for (int n = 0; n < PNC; ++n) lrow[n] += ls[n];
        if (grp == 0 && t == 0) PTRACE(8, tile_i);
        if (grp == 0 && t == 0) PTRACE(6, tile_i);
        if (L - tau * TILE < TILE) {
          // rows past the sequence end in the two P.C slots: zero, so that
          // 0 * garbage cannot reach O (32 chunks of 16 bytes per row)
          const int r0 = L - tau * TILE > 0 ? L - tau * TILE : 0;
          const int total = (TILE - r0) * 32;
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
          for (int idx = grp * 128 + t; idx < total; idx += 128 * PGR) {
            const int row = r0 + (idx >> 5), h4 = (idx >> 3) & 3;
            const uint32_t a = s_pair + (h4 >> 1) * 2 * P_PAIR_BYTES + (h4 & 1) * P_HALF_BYTES + row * 128 + (idx & 7) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(z.x), "r"(z.y), "r"(z.z), "r"(z.w)
                         : "memory");
          }
        }
        // P (and any zeroed rows) visible to the tensor core before the signal;
        // issued here, its latency overlaps the wait for the peer's factors
        fence_proxy_async_smem();
        // the peer's vote for the same tile: rescale its rows' O columns here
        if (!(ok = mbar_wait_cluster(smem_u32(&ctl->xch_full[k2]), (tile_i >> 1) & 1, abort, p.status))) break;
        if (grp == 0 && t == 0) PTRACE(9, tile_i);
        float pa[PNC];
        bool peer_rescale = false;
#pragma unroll
        for (int i = 0; i < PNC; ++i) {
          pa[i] = ctl->xalpha[k2][cb + i];
          peer_rescale |= pa[i] != 1.f;
        }
        // arm the barrier's next use (two tiles on): the peer cannot send that
        // tile's factors before this CTA has passed the next tile
        if (t == 0) mbar_arrive_expect_tx(smem_u32(&ctl->xch_full[k2]), 4 * PNC);
        if (peer_rescale && tau != t0) {
          if (!pc_seen && !(ok = wait_pc())) break;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t v[16];
            const uint32_t ta = tmem + lane_addr + 128 * j + col_peer;
            tmem_ld16(ta, v);
            tmem_wait_ld();
            reg_fence16(v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * pa[i]);
            tmem_st16(ta, v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) signal_leader(&ctl->p_full[k2], p_full_l[k2], 0);
        if (grp == 0 && t == 0) PTRACE(10, tile_i);
        if (tau == t1 - 1) {
          // the item's softmax sums are final: reduce them and send them to the
          // peer now, while the last P.C runs
#pragma unroll
          for (int n = 0; n < PNC; ++n) {
            float v = lrow[n];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) ctl->red[sw][cb + n] = v;
          }
          named_bar_sync(gbar, 128);
          if (t < PNC) {
            const int n = cb + t;
            const float l = (ctl->red[0][n] + ctl->red[1][n]) + (ctl->red[2][n] + ctl->red[3][n]);
            ctl->lsum[n] = l;
            st_async_u32(at_peer(&ctl->xl[item_i & 1][n]), at_peer(&ctl->l_full[item_i & 1]), __float_as_uint(l));
          }
        }
        ++tile_i;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait(smem_u32(&ctl->o_full), item_i & 1, abort, p.status))) break;
      if (grp == 0 && t == 0) PTRACE(12, tile_i - 1);
      tc_fence_after();
      if (!(ok = mbar_wait_cluster(smem_u32(&ctl->l_full[item_i & 1]), (item_i >> 1) & 1, abort, p.status))) break;
      const float l_own = t < PNC ? ctl->lsum[cb + t] : 0.f;
      if (t < PNC) {
        ctl->linv[col_own + t] = l_own > 0.f ? 1.f / l_own : 0.f;
        const float lp = ctl->xl[item_i & 1][cb + t];
        ctl->linv[col_peer + t] = lp > 0.f ? 1.f / lp : 0.f;
      }
      named_bar_sync(gbar, 128);
      if (t == 0) mbar_arrive_expect_tx(smem_u32(&ctl->l_full[item_i & 1]), 4 * PNC);   // arm its next use
      if (grp == 0 && t == 0) PTRACE(13, tile_i - 1);
      const int nt = ntiles(L);
      const bool final_out = unit_of(acc, T, p.U) == unit_of(acc + nt - 1, T, p.U);
      const long long row0 = (final_out ? (long long)b * p.G : ((long long)(b + u)) * p.G) + (it.c & ~1) * PN;
      float* obase = final_out ? p.o_lat : p.ws_o;
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        const int lat = 256 * j + 128 * r + t;
#pragma unroll
        for (int side = 0; side < 2; ++side) {
          const uint32_t col = side ? col_peer : col_own;
          uint32_t v[16];
          tmem_ld16(tmem + lane_addr + 128 * j + col, v);
          tmem_wait_ld();
          reg_fence16(v);
#pragma unroll
          for (int n = 0; n < 16; ++n)
            __stcg(obase + (row0 + col + n) * D_C + lat, __uint_as_float(v[n]) * ctl->linv[col + n]);
        }
      }
      if (grp == 0 && t == 0) PTRACE(14, tile_i - 1);
      if (t < PNC) {
        const float lse = l_own > 0.f ? (m_run[t] + __log2f(l_own)) * P_LN2 : -INFINITY;
        (final_out ? p.lse : p.ws_lse)[row0 + col_own + t] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) signal_leader(&ctl->o_empty, o_empty_l, 1);
      if (grp == 0 && t == 0) PTRACE(15, tile_i - 1);
      named_bar_sync(gbar, 128);
      ++item_i;
    }
  }

  __syncwarp();
  if (threadIdx.x == 128) PTRACE_CTA(2, globaltimer());
  tc_fence_before();
  // neither CTA leaves while the other may still touch its shared or tensor
  // memory (remote arrivals, the pair MMAs)
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, PTMEM_COLS);
  }
}

size_t attn_pair_smem_bytes() { return POFF_CTRL + sizeof(PairCtrl) + sizeof(int) * (MAX_SEQS + 1) + 1024; }

// Sets the shared-memory attribute once per device and returns how many CTA
// pairs fit on the GPU at once (the persistent grid's size).
cudaError_t attn_pair_prepare(int* max_pairs) {
  static DeviceFlags attr;
  const int smem = static_cast<int>(attn_pair_smem_bytes());
  cudaError_t e = once_per_device(attr, [smem] {
    return cudaFuncSetAttribute(decode_attn_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PTHREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_pairs, decode_attn_pair_kernel, &cfg);
}

cudaError_t launch_decode_attn_pair(const CUtensorMap& tm_cache, const CUtensorMap& tm_q, const AttnParams& p,
                                    cudaStream_t s) {
  if (p.B > MAX_SEQS || p.N != PN || p.C % 2) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.U == 1 && p.slots > 0 ? 2 * p.slots : p.U * p.C);
  cfg.blockDim = dim3(PTHREADS);
  cfg.dynamicSmemBytes = attn_pair_smem_bytes();
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_attn_pair_kernel, tm_cache, tm_q, p);
}

}  // namespace mla
