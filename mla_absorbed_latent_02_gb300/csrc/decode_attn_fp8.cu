// Decode attention over the FP8 latent cache ("DeepSeek MLA 吸收式缓存" §6.1:
// FlashMLA's decoding kernels that read an FP8 KV cache in MQA mode, a 576-wide
// key and a 512-wide value). Cache row (656 bytes): e4m3 codes of c_kv / sigma |
// the bf16 RoPE'd key | sigma (float32, a power of two) | padding.
//
// Same unit split, warp roles and split-KV output as the bf16 kernel; what
// changes is the operand precision of the two tile contractions and the way
// the MMA warp schedules them:
//  * Scores. The latent part runs as e4m3 x e4m3 tensor-core MMAs
//    (kind::f8f6f4, K = 32): the cache codes against the latent query, which
//    warps 2-3 split per query row into e4m3 hi + lo parts of q / sigma_q
//    (sigma_q the row's power-of-two scale; the lo part stored scaled by 2^4;
//    hi + lo carry about as many bits as bf16). The two parts are stacked on the MMA's N axis (N' = 2N), so each
//    MMA reads its cache slice once for both. The RoPE part stays bf16
//    (kind::f16) in its own TMEM columns.
//  * Softmax. The thread of token t forms the log2-domain logit
//    x = scale*log2(e) * (sigma_t sigma_q (S_hi + S_lo) + S_rope) and runs the
//    online softmax on x' = x + log2 sigma_t, so that P' = 2^(x' - m + 8)
//    = p_t sigma_t times a per-row factor: O accumulates P' . codes directly and
//    the normaliser l accumulates P' / sigma_t (the same softmax scaled by
//    2^(8-m)). The running max m is raised as soon as a logit exceeds it by
//    2^0.5, so P' <= 2^8.5 < 448. P' values far below the running max fall in
//    e4m3's subnormal range, where a code is exact to 2^-10 (in P' units): with
//    N <= 32 the remainder part is stored scaled by 2^4 (its own accumulator
//    columns, summed in the epilogue), which carries every P' to within 2^-22
//    of the running max and drops smaller ones; with N = 64 the two parts
//    share an accumulator and the bound is 2^-18. The normaliser sums the
//    weights as represented, so the output is a convex combination of rows.
//  * P.C. P' is split into e4m3 hi + lo and written K-major (one 128-byte row of
//    token bytes per query row, hi rows then lo rows, 128-byte swizzle; a 4-lane
//    byte transpose turns the thread-per-token values into 4-token words); the
//    A operand is the same cache tile read MN-major (token rows of 128 latent
//    codes). With N <= 32 the hi and lo rows are one N' = 2N operand and O^T has
//    hi and lo columns; with N = 64 (TMEM is short) they are two MMAs into one
//    accumulator.
//  * Scheduling. The MMA warp polls both contractions' operands and issues
//    whatever is ready: the next tile's scores (into a second TMEM buffer) group
//    by group as its cache columns land, and the current tile's P.C products as
//    soon as its P' is written.
// Per 128-token tile (N <= 32): 4 RoPE + 16 latent score MMAs and 16 P.C MMAs
// over 82 KB of cache (the bf16 kernel: 68 MMAs over 147 KB).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "attn_sched.cuh"
#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

// Optional phase trace (compile with -DMLA_TRACE=1): SM clock stamps of the
// pipeline events of the first tiles of the first CTAs, read back with
// mla_trace8_read(). Off in normal builds.
#ifndef MLA_TRACE
#define MLA_TRACE 0
#endif
#if MLA_TRACE
#define T8_CTAS 8
#define T8_TILES 32
#define T8_EVENTS 12
__device__ long long g_mla_trace8[T8_CTAS][T8_TILES][T8_EVENTS];
#define T8(ev, tile)                                                      \
  do {                                                                    \
    if (blockIdx.x < T8_CTAS && (tile) < T8_TILES)                        \
      g_mla_trace8[blockIdx.x][(tile)][(ev)] = clock64();                 \
  } while (0)
extern "C" int mla_trace8_read(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace8)) bytes = sizeof(g_mla_trace8);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace8, bytes);
}
__device__ unsigned long long g_mla_trace8_cta[1024][4];
#define T8CTA(ev)                                                               \
  do {                                                                          \
    if (blockIdx.x < 1024) g_mla_trace8_cta[blockIdx.x][(ev)] = globaltimer();  \
  } while (0)
extern "C" int mla_trace8_read_cta(void* host, size_t bytes) {
  if (bytes > sizeof(g_mla_trace8_cta)) bytes = sizeof(g_mla_trace8_cta);
  return (int)cudaMemcpyFromSymbol(host, g_mla_trace8_cta, bytes);
}
#else
#define T8(ev, tile) \
  do {               \
  } while (0)
#define T8CTA(ev) \
  do {            \
  } while (0)
#endif

namespace mla {

namespace {

constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE8_LOG2 = 0.5f;   // raise the running max past this margin (log2 units)
// Scale of the e4m3 remainder parts that land in accumulator columns of their
// own (the query's lo part of the scores; the weights' lo part when hi and lo
// are stacked on the MMA's N): 2^4 is the largest that cannot overflow e4m3.
constexpr float LO_SCALE = 16.0f;
constexpr float P_SHIFT = 8.0f;         // P' = 2^(x' - m + P_SHIFT)
constexpr uint32_t G_BYTES = 16384;     // 128 tokens x 128 latent codes
constexpr uint32_t R_BYTES = 16384;     // 128 tokens x 64 bf16 RoPE key (with N = 64: then P'^T hi | lo)
constexpr uint32_t SC_BYTES = 2048;     // 128 tokens x 16 bytes (sigma + padding)
constexpr uint32_t BOX8 = 8192;         // one TMA box: 64 rows x 128 bytes
constexpr uint32_t SCBOX = 1024;        // 64 rows x 16 bytes
constexpr int NG_MAX = 9, NR8 = 2;

struct __align__(8) Ctrl8 {
  uint64_t q_empty, qr_full, q8_full, q8_free;
  uint64_t g_full[NG_MAX], g_empty[NG_MAX];
  uint64_t r_full[NR8], r_empty[NR8];
  uint64_t s_full[2], p_full[2], pc_done, o_full, o_empty, mma_final;
  uint32_t tmem_base;
  int abort;
  int vote[4][2][4];
  float qsig[2][64];   // sigma_q of each query row, by item parity
  float m_run[64];
  float alpha[64];
  float red[4][64];
  float lsum[64];
  float linv[64];
  int warp_tot[32];   // one per warp of the CTA (tile_prefix)
};

template <int N>
struct Cfg8 {
  static constexpr int NG = (N == 16) ? 9 : (N == 32 ? 8 : 6);   // latent group slots
  static constexpr uint32_t QG = N * 128u;      // one 128-column group of a query part: N rows x 128 bytes
  // P'^T (hi | lo, 2 QG) in its own buffer per tile parity, so that the RoPE
  // slot is free once the scores are done; with N = 64 shared memory is short
  // and P'^T takes the tile's RoPE slot instead (freed by its P.C products)
  static constexpr bool P_SEP = N <= 32;
  // hi and lo are stacked on the MMA's N axis (N' = 2N): one MMA reads each
  // cache slice once for both parts (at these N an MMA costs what streaming its
  // 128-row A slice out of shared memory costs). The scores are always
  // stacked (hi | lo | RoPE columns); O^T is stacked (hi | lo per m-tile) when
  // TMEM has room, N <= 32: with N = 64 the P.C products stay two MMAs into one
  // accumulator.
  static constexpr bool STACK_O = N <= 32;
  // query group g: hi rows at q_hi(g), lo rows right below (N x 128 bytes each),
  // so that rows 0..2N-1 form one operand
  __host__ __device__ static constexpr uint32_t q_hi(int g) { return 2 * g * QG; }
  __host__ __device__ static constexpr uint32_t q_lo(int g) { return (2 * g + 1) * QG; }
  static constexpr uint32_t OFF_QR = 8 * QG;    // bf16 RoPE query block
  static constexpr uint32_t OFF_P = 9 * QG;     // P'^T buffers (P_SEP)
  static constexpr uint32_t OFF_G = OFF_P + (P_SEP ? 4 * QG : 0);
  static constexpr uint32_t OFF_R = OFF_G + NG * G_BYTES;
  static constexpr uint32_t OFF_SC = OFF_R + NR8 * R_BYTES;
  static constexpr uint32_t OFF_CTRL = OFF_SC + NR8 * SC_BYTES;
  static constexpr uint32_t SMEM = OFF_CTRL + sizeof(Ctrl8) + sizeof(int) * (MAX_SEQS + 1) + 1024;
  // TMEM: O^T m-tile mt at mt*OW (stacked: hi columns, then lo); two score
  // buffers of SB columns from COL_S: latent scores (stacked: hi, lo) then RoPE
  static constexpr uint32_t OW = STACK_O ? 2 * N : N;
  static constexpr uint32_t SB = 3 * N;
  static constexpr uint32_t COL_S = 4 * OW;
  static constexpr uint32_t COL_R = 2 * N;              // RoPE scores within a buffer
  // the scores of tile i+1 go to the second buffer only when issued ahead
  static constexpr uint32_t NSB = (NG >= 8) ? 2 : 1;
  static constexpr uint32_t TMEM_NEED = COL_S + NSB * SB;
  static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 128 ? 128u : (TMEM_NEED <= 256 ? 256u : 512u);
  // The scores of tile i+1 are issued before the P.C MMAs of tile i when the
  // latent slots hold both tiles (the tensor pipe then works through tile i's
  // softmax); otherwise the issue order is S(i), P.C(i), S(i+1).
  static constexpr bool AHEAD = NSB == 2;
  // softmax/epilogue: GR groups of 4 warps, NC query rows (columns) each; four
  // groups at N = 64 keep a thread's share of a tile at 16 columns
  static constexpr int GR = N == 64 ? 4 : 2;
  static constexpr int NC = N / GR;
  static constexpr int CW = NC < 16 ? NC : 16;
  static constexpr int THREADS = 128 + 128 * GR;
  static_assert(OFF_P % 1024 == 0 && OFF_G % 1024 == 0 && OFF_R % 1024 == 0, "swizzled operands need 1 KB alignment");
  static_assert(2 * QG <= R_BYTES, "P'^T hi and lo fit in a RoPE slot");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(TMEM_NEED <= 512, "tensor memory per CTA");
};

// Token scale exponent of a row maximum: the smallest e >= FP8_SCALE_EXP_MIN
// with amax / 2^e <= 448 = 1.75 * 2^8 (the cache writer's rule).
MLA_DEV int scale_exp(float amax) {
  const uint32_t ab = __float_as_uint(amax);
  const int ef = static_cast<int>(ab >> 23);
  const int e = ef == 0 ? FP8_SCALE_EXP_MIN : ef - 127 - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return max(e, FP8_SCALE_EXP_MIN);
}

// Two values as e4m3 pairs (byte 0 from a, byte 1 from b): hi = e4m3(x) and lo = e4m3((x - hi) * lo_scale),
// nearest-even both. Returns the values the pair stands for, hi + lo / lo_scale.
// A remainder is at most half an e4m3 step of hi (2^-4 of |x|, and 16 for
// |x| <= 448), so lo_scale = LO_SCALE keeps it finite while lifting small
// remainders out of the subnormal range; lo_scale = 1 when hi and lo are summed
// by the tensor core into one accumulator.
MLA_DEV float2 split_e4m3x2(float a, float b, uint32_t& hi, uint32_t& lo, float lo_scale) {
  const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
  const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(
      make_float2((a - hf.x) * lo_scale, (b - hf.y) * lo_scale), __NV_SATFINITE, __NV_E4M3);
  const float2 lf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(l, __NV_E4M3)));
  hi = h;
  lo = l;
  const float inv = 1.f / lo_scale;   // a power of two: exact
  return make_float2(hf.x + lf.x * inv, hf.y + lf.y * inv);
}

// 4 x 4 byte transpose across the lanes of a quad: lane i holds byte k = value
// (token i, column k); afterwards lane i holds byte k = value (token k, column i).
MLA_DEV uint32_t quad_transpose(uint32_t w, int i) {
  uint32_t y = __shfl_xor_sync(0xffffffffu, w, 2);
  const uint32_t x = (i < 2) ? __byte_perm(w, y, 0x5410) : __byte_perm(w, y, 0x3276);
  y = __shfl_xor_sync(0xffffffffu, x, 1);
  return (i & 1) ? __byte_perm(x, y, 0x3715) : __byte_perm(x, y, 0x6240);
}

}  // namespace

template <int N>
__global__ void __launch_bounds__(Cfg8<N>::THREADS, 1)
    decode_attn_fp8_kernel(const __grid_constant__ CUtensorMap tm_c8, const __grid_constant__ CUtensorMap tm_sc,
                           const __grid_constant__ CUtensorMap tm_qr, const AttnParams p) {
  using K = Cfg8<N>;
  if (threadIdx.x == 0) T8CTA(0);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctrl8* ctl = reinterpret_cast<Ctrl8*>(smem + K::OFF_CTRL);
  const uint32_t s_q8 = smem_u32(smem);
  const uint32_t s_qr = s_q8 + K::OFF_QR;
  const uint32_t s_g = s_q8 + K::OFF_G;
  const uint32_t s_pb = s_q8 + K::OFF_P;
  const uint32_t s_r = s_q8 + K::OFF_R;
  const uint32_t s_sc = s_q8 + K::OFF_SC;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x / p.C;     // unit
  const int c = blockIdx.x % p.C;     // row group within the unit
  volatile int* abort = &ctl->abort;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->q_empty), 1);
    mbar_init(smem_u32(&ctl->qr_full), 1);
    mbar_init(smem_u32(&ctl->q8_full), 2);
    mbar_init(smem_u32(&ctl->q8_free), 4 * K::GR);
    for (int i = 0; i < K::NG; ++i) {
      mbar_init(smem_u32(&ctl->g_full[i]), 1);
      mbar_init(smem_u32(&ctl->g_empty[i]), 1);
    }
    for (int i = 0; i < NR8; ++i) {
      mbar_init(smem_u32(&ctl->r_full[i]), 1);
      // released by the softmax warps once they have read the scales (P_SEP),
      // else by the tile's P.C products
      mbar_init(smem_u32(&ctl->r_empty[i]), K::P_SEP ? 4 * K::GR : 1);
    }
    mbar_init(smem_u32(&ctl->pc_done), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->s_full[i]), 1);
      mbar_init(smem_u32(&ctl->p_full[i]), 4 * K::GR);
    }
    mbar_init(smem_u32(&ctl->o_full), 1);
    mbar_init(smem_u32(&ctl->o_empty), 4 * K::GR);
    mbar_init(smem_u32(&ctl->mma_final), 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_c8);
    tma_prefetch_desc(&tm_sc);
    tma_prefetch_desc(&tm_qr);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctl->tmem_base), K::TMEM_COLS);
    tmem_relinquish();
  }
  int* pre = reinterpret_cast<int*>(smem + K::OFF_CTRL + sizeof(Ctrl8));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  // the unit's tile range depends only on the sequence lengths (a call input)
  tile_prefix(p, pre, ctl->warp_tot);
  pdl_wait();
  if (threadIdx.x == 0) T8CTA(1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ItemIter it;
      it.init(p, pre, u, c);
      uint32_t g_i = 0, rope_i = 0, qr_issued = 0;
      int b, t0, t1, L;
      long long acc;
      const bool stream_hint = p.C == 1;
      const uint64_t pol_stream = l2_policy_evict_first();
      bool ok = true;
      auto load = [&](const CUtensorMap* m, uint32_t dst, uint32_t bar, int x, int y) {
        if (stream_hint) tma_load_2d_hint(dst, m, bar, x, y, pol_stream);
        else tma_load_2d(dst, m, bar, x, y);
      };
      while (ok && it.next(b, t0, t1, L, acc)) {
        // the item's RoPE query rows, once the previous item's score MMAs are done
        const uint32_t qf = smem_u32(&ctl->qr_full);
        if (!(ok = mbar_wait(smem_u32(&ctl->q_empty), (qr_issued & 1) ^ 1, abort, p.status))) break;
        mbar_arrive_expect_tx(qf, K::QG);
        tma_load_2d(s_qr, &tm_qr, qf, D_C, b * p.G + c * N);
        ++qr_issued;
        for (int tau = t0; tau < t1 && ok; ++tau) {
          int row[2];
          uint32_t nbox = 0;
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            const int page = 2 * tau + pg;
            row[pg] = -1;
            if (page * PAGE >= L) continue;
            if (p.paged) {
              const int id = page < p.max_blocks ? p.block_table[(long long)b * p.max_blocks + page] : -1;
              if (id >= 0 && id < p.num_blocks) row[pg] = id * PAGE;
              else atomicOr(p.status, MLA_DEVERR_BOUNDS);
            } else {
              if (L > p.capacity) atomicOr(p.status, MLA_DEVERR_BOUNDS);
              else row[pg] = b * p.capacity + page * PAGE;
            }
            if (row[pg] >= 0) ++nbox;
          }
          // RoPE key and scales of the tile
          const uint32_t rslot = rope_i % NR8;
          if (!(ok = mbar_wait(smem_u32(&ctl->r_empty[rslot]), ((rope_i / NR8) & 1) ^ 1, abort, p.status))) break;
          T8(0, rope_i);
          const uint32_t rfull = smem_u32(&ctl->r_full[rslot]);
          mbar_arrive_expect_tx(rfull, nbox * (BOX8 + SCBOX));
          for (int pg = 0; pg < 2; ++pg)
            if (row[pg] >= 0) {
              load(&tm_c8, s_r + rslot * R_BYTES + pg * BOX8, rfull, ROW8_ROPE, row[pg]);
              load(&tm_sc, s_sc + rslot * SC_BYTES + pg * SCBOX, rfull, ROW8_SCALE, row[pg]);
            }
          ++rope_i;
          // the four 128-column groups of latent codes
          for (int gq = 0; gq < 4; ++gq) {
            const uint32_t slot = g_i % K::NG;
            if (!(ok = mbar_wait(smem_u32(&ctl->g_empty[slot]), ((g_i / K::NG) & 1) ^ 1, abort, p.status))) break;
            const uint32_t full = smem_u32(&ctl->g_full[slot]);
            mbar_arrive_expect_tx(full, nbox * BOX8);
            for (int pg = 0; pg < 2; ++pg)
              if (row[pg] >= 0) load(&tm_c8, s_g + slot * G_BYTES + pg * BOX8, full, 128 * gq, row[pg]);
            ++g_i;
          }
          T8(1, rope_i - 1);
        }
      }
      if (!ok) {
        // Let copies already in flight land before the CTA exits.
        for (uint32_t k = 0; k < K::NG && k < g_i; ++k) {
          const uint32_t i = g_i - 1 - k;
          mbar_wait_ns(smem_u32(&ctl->g_full[i % K::NG]), (i / K::NG) & 1, 20000000ull);
        }
        for (uint32_t k = 0; k < NR8 && k < rope_i; ++k) {
          const uint32_t i = rope_i - 1 - k;
          mbar_wait_ns(smem_u32(&ctl->r_full[i % NR8]), (i / NR8) & 1, 20000000ull);
        }
        if (qr_issued > 0) mbar_wait_ns(smem_u32(&ctl->qr_full), (qr_issued - 1) & 1, 20000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Two cursors walk the unit's tiles in order: one issues the scores, the
    // other the P.C products (one tile behind when K::AHEAD).
    if (lane == 0) {
      struct Cursor {
        ItemIter it;
        bool valid;
        int b, t0, t1, L, tau;
        long long acc;
        uint32_t item, tile, g, r;   // item and tile counts, latent and RoPE slot counts
        MLA_DEV void start(const AttnParams& p, const int* pre, int u, int c) {
          it.init(p, pre, u, c);
          valid = it.next(b, t0, t1, L, acc);
          tau = t0;
          item = tile = g = r = 0;
        }
        MLA_DEV void advance() {
          ++tile;
          g += 4;
          ++r;
          if (++tau >= t1) {
            valid = it.next(b, t0, t1, L, acc);
            tau = t0;
            ++item;
          }
        }
      };
      constexpr uint32_t ID_QR = idesc_bf16_f32(128, N, 0, 0);
      constexpr uint32_t ID_QL = idesc_e4m3_f32(128, 2 * N, 0, 0);
      constexpr uint32_t ID_PV = idesc_e4m3_f32(128, K::STACK_O ? 2 * N : N, 1, 0);
      Cursor cs, cp;
      cs.start(p, pre, u, c);
      cp.start(p, pre, u, c);
      bool ok = true;
      // O^T += codes^T . (P'_hi + P'_lo)^T of tile k (P' written, O free)
      auto issue_pv = [&](Cursor& k) {
        tc_fence_after();
        T8(6, k.tile);
        const uint32_t rslot = k.r % NR8;
        const uint32_t s_p = K::P_SEP ? s_pb + (k.tile & 1) * 2 * K::QG : s_r + rslot * R_BYTES;
        for (int mt = 0; mt < 4; ++mt) {
          const uint32_t slot = (k.g + mt) % K::NG;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(s_g + slot * G_BYTES + kk * 4096, 16384, 1024, SMEM_SWIZZLE_128B);
            const uint32_t bp = s_p + 32 * kk;
            // P'^T rows: hi 0..N-1, lo N..2N-1
            mma_e4m3_ss(tmem + mt * K::OW, ad, smem_desc(bp, 16, 1024, SMEM_SWIZZLE_128B), ID_PV,
                        !(k.tau == k.t0 && kk == 0));
            if (!K::STACK_O)
              mma_e4m3_ss(tmem + mt * N, ad, smem_desc(bp + K::QG, 16, 1024, SMEM_SWIZZLE_128B), ID_PV, 1);
          }
          mma_commit(smem_u32(&ctl->g_empty[slot]));
        }
        if (!K::P_SEP) mma_commit(smem_u32(&ctl->r_empty[rslot]));
        mma_commit(smem_u32(&ctl->pc_done));
        T8(7, k.tile);
        if (k.tau == k.t1 - 1) mma_commit(smem_u32(&ctl->o_full));
      };
      // The issue loop polls the operands of both contractions and issues
      // whatever is ready: the scores of tile cs group by group as its cache
      // columns land (S_rope = C_rope . Q_rope^T in bf16, then S_lat = codes .
      // (Q_hi + Q_lo)^T in e4m3, one 128-column group at a time), and the P.C
      // products of tile cp as soon as its P' is written. Scores run at most
      // one tile ahead of the next P.C (their TMEM buffer is then free: the
      // softmax of the tile two back has been consumed); without K::AHEAD they
      // wait for the previous tile's P.C. A stall longer than the wait limit
      // aborts the CTA like any other bounded wait.
      int s_stage = 0;   // tile cs: 0 query operands, 1 RoPE block, 2 + gq latent group gq, 6 done
      uint64_t t_idle = globaltimer();
      while (ok && cp.valid) {
        bool progress = false;
        if (cs.valid && cs.tile <= cp.tile + (K::AHEAD ? 1u : 0u)) {
          const uint32_t sb = cs.tile & 1;
          const uint32_t d_sl = tmem + K::COL_S + K::SB * (sb % K::NSB), d_sr = d_sl + K::COL_R;
          while (true) {
            if (s_stage == 0) {
              if (cs.tau == cs.t0 && !(mbar_probe(smem_u32(&ctl->qr_full), cs.item & 1) &&
                                       mbar_probe(smem_u32(&ctl->q8_full), cs.item & 1)))
                break;
              s_stage = 1;
            }
            if (s_stage == 1) {
              const uint32_t rslot = cs.r % NR8;
              if (!mbar_probe(smem_u32(&ctl->r_full[rslot]), (cs.r / NR8) & 1)) break;
              T8(2, cs.tile);
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16_ss(d_sr, smem_desc(s_r + rslot * R_BYTES + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B),
                            smem_desc(s_qr + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B), ID_QR, kk != 0);
              s_stage = 2;
              progress = true;
            }
            if (s_stage < 6) {
              const int gq = s_stage - 2;
              const uint32_t i = cs.g + gq, slot = i % K::NG;
              if (!mbar_probe(smem_u32(&ctl->g_full[slot]), (i / K::NG) & 1)) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc(s_g + slot * G_BYTES + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B);
                mma_e4m3_ss(d_sl, ad, smem_desc(s_q8 + K::q_hi(gq) + 32 * kk, 16, 1024, SMEM_SWIZZLE_128B), ID_QL,
                            (gq | kk) != 0);
              }
              progress = true;
              if (++s_stage < 6) continue;
            }
            mma_commit(smem_u32(&ctl->s_full[sb]));
            T8(3, cs.tile);
            if (cs.tau == cs.t1 - 1) mma_commit(smem_u32(&ctl->q_empty));
            cs.advance();
            s_stage = 0;
            break;
          }
        }
        if (cp.tile < cs.tile) {
          bool ready = mbar_probe(smem_u32(&ctl->p_full[cp.tile & 1]), (cp.tile >> 1) & 1);
          if (ready && cp.tau == cp.t0 && cp.item > 0) ready = mbar_probe(smem_u32(&ctl->o_empty), (cp.item - 1) & 1);
          if (ready) {
            issue_pv(cp);
            cp.advance();
            progress = true;
          }
        }
        if (progress) {
          t_idle = globaltimer();
        } else if (*abort) {
          ok = false;
        } else if (globaltimer() - t_idle > MLA_WAIT_TIMEOUT_NS) {
          *abort = 1;
          atomicOr(p.status, MLA_DEVERR_TIMEOUT);
          ok = false;
        }
      }
      // every MMA this thread issued has completed once mma_final flips
      mma_commit(smem_u32(&ctl->mma_final));
      mbar_wait_ns(smem_u32(&ctl->mma_final), 0, 100000000ull);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ query converter (warps 2-3)
    // Row r of the CTA's N query rows: lane j owns latent columns 16j .. 16j+15
    // (group j/8, 16-byte chunk j%8). sigma_q = 2^e by the cache writer's scale
    // rule; hi = e4m3(q / sigma_q), lo = e4m3(q / sigma_q - hi), written K-major
    // with the 128-byte swizzle (chunk j of row r at j ^ (r % 8)).
    const int wq = warp - 2;
    constexpr int RW = N / 2;              // rows per converter warp: wq, wq + 2, ...
    constexpr int CH = RW < 8 ? RW : (K::GR == 4 ? 4 : 8);   // rows whose loads are in flight together
    ItemIter it;
    it.init(p, pre, u, c);
    uint32_t item_i = 0;
    int b, t0, t1, L;
    long long acc;
    bool ok = true;
    const int g = lane >> 3, j = lane & 7;
    uint4 buf[CH][2];
    auto load_rows = [&](int r0) {
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int r = wq + 2 * (r0 + i);
        const uint4* src =
            reinterpret_cast<const uint4*>(p.q_abs + ((long long)b * p.G + c * N + r) * ROW + 16 * lane);
        buf[i][0] = __ldcg(src);
        buf[i][1] = __ldcg(src + 1);
      }
    };
    bool have = it.next(b, t0, t1, L, acc);
    if (have) load_rows(0);
    while (ok && have) {
      // the query buffers are free once the previous item's score MMAs are done;
      // the sigma_q slot (item parity) once the softmax has started the item before
      if (!(ok = mbar_wait(smem_u32(&ctl->q_empty), (item_i & 1) ^ 1, abort, p.status))) break;
      if (item_i > 0 && !(ok = mbar_wait(smem_u32(&ctl->q8_free), (item_i - 1) & 1, abort, p.status))) break;
      float* qs = ctl->qsig[item_i & 1];
      if (lane == 0 && wq == 0) T8(8, item_i);
#pragma unroll 1
      for (int r0 = 0; r0 < RW; r0 += CH) {
        if (r0 > 0) load_rows(r0);
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          const int r = wq + 2 * (r0 + i);
          const uint32_t w[8] = {buf[i][0].x, buf[i][0].y, buf[i][0].z, buf[i][0].w,
                                 buf[i][1].x, buf[i][1].y, buf[i][1].z, buf[i][1].w};
          float v[16];
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            amax = fmaxf(amax, fmaxf(fabsf(v[2 * k]), fabsf(v[2 * k + 1])));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const int e = scale_exp(amax);
          const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t h0, l0, h1, l1;
            split_e4m3x2(v[4 * k] * inv, v[4 * k + 1] * inv, h0, l0, LO_SCALE);
            split_e4m3x2(v[4 * k + 2] * inv, v[4 * k + 3] * inv, h1, l1, LO_SCALE);
            hi[k] = h0 | (h1 << 16);
            lo[k] = l0 | (l1 << 16);
          }
          const uint32_t rw = r * 128 + ((j ^ (r & 7)) << 4);
          const uint32_t a = s_q8 + K::q_hi(g) + rw, a_lo = s_q8 + K::q_lo(g) + rw;
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                       "r"(hi[3])
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a_lo), "r"(lo[0]), "r"(lo[1]),
                       "r"(lo[2]), "r"(lo[3])
                       : "memory");
          if (lane == 0) qs[r] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->q8_full));
      if (lane == 0 && wq == 0) T8(9, item_i);
      ++item_i;
      // the next item's first rows are loaded before waiting for its buffers
      have = it.next(b, t0, t1, L, acc);
      if (have) load_rows(0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // K::GR groups of 4 warps; group grp owns the NC columns [cb, cb + NC) of
    // S, P' and O (query rows of the CTA); a thread owns one token row.
    constexpr int NC = K::NC, CW = K::CW;
    const int sw = warp & 3;                  // TMEM lane quarter
    const int grp = (warp - 4) >> 2;
    const int cb = grp * NC;
    const uint32_t gbar = 1 + grp;            // named barrier of the group
    const int t = sw * 32 + lane;             // token row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(sw * 32) << 16;
    const int qi = lane & 3;                  // lane within its quad
    const int tq = sw * 32 + (lane & ~3);     // first token of the quad
    // column cb + n sees tokens < L - dlim[n / 16] (a query token owns >= 16 columns)
    int dlim[(NC + 15) / 16];
#pragma unroll
    for (int k = 0; k < (NC + 15) / 16; ++k) dlim[k] = p.Hq - 1 - (c * N + cb + 16 * k) / p.H;

    ItemIter it;
    it.init(p, pre, u, c);
    uint32_t g_i = 0, rope_i = 0, item_i = 0, tile_i = 0;
    int b, t0, t1, L;
    long long acc;
    const long long T = it.T;
    bool ok = true;
    float lrow[NC];
    float* m_run = ctl->m_run + cb;
    float* alpha = ctl->alpha + cb;
    while (ok && it.next(b, t0, t1, L, acc)) {
      if (!(ok = mbar_wait(smem_u32(&ctl->q8_full), item_i & 1, abort, p.status))) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->q8_free));
      const float* qs = ctl->qsig[item_i & 1] + cb;
      if (t < NC) m_run[t] = -INFINITY;
      named_bar_sync(gbar, 128);
#pragma unroll
      for (int n = 0; n < NC; ++n) lrow[n] = 0.f;
      for (int tau = t0; tau < t1; ++tau) {
        const uint32_t rslot = rope_i % NR8;
        const uint32_t sb = tile_i & 1;
        if (!(ok = mbar_wait(smem_u32(&ctl->s_full[sb]), (tile_i >> 1) & 1, abort, p.status))) break;
        // the scales come from the tile's TMA copies
        if (!(ok = mbar_wait(smem_u32(&ctl->r_full[rslot]), (rope_i / NR8) & 1, abort, p.status))) break;
        if (t == 0 && grp == 0) T8(4, tile_i);
        tc_fence_after();
        const int tok = tau * TILE + t;
        float x[NC];
        float inv_sig;
        {
          uint32_t vl[NC], vr[NC], vh[NC];
          const uint32_t sbase = tmem + lane_addr + K::COL_S + K::SB * (sb % K::NSB) + cb;
#pragma unroll
          for (int k = 0; k < NC / CW; ++k) {
            tmem_ld_w<CW>(sbase + CW * k, vl + CW * k);
            tmem_ld_w<CW>(sbase + N + CW * k, vh + CW * k);
            tmem_ld_w<CW>(sbase + K::COL_R + CW * k, vr + CW * k);
          }
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < NC / CW; ++k) {
            reg_fence_w<CW>(vl + CW * k);
            reg_fence_w<CW>(vh + CW * k);
            reg_fence_w<CW>(vr + CW * k);
          }
          // S_lat = S_hi + S_lo / LO_SCALE (the query's lo part is stored scaled)
#pragma unroll
          for (int n = 0; n < NC; ++n)
            vl[n] = __float_as_uint(__uint_as_float(vl[n]) + __uint_as_float(vh[n]) * (1.f / LO_SCALE));
          uint32_t sb;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sb) : "r"(s_sc + rslot * SC_BYTES + t * 16));
          // sigma_t = 2^(ef - 127); rows past the sequence end hold anything, so
          // the exponent is clamped into the range the cache writer produces
          const int ef = min(max(static_cast<int>((sb >> 23) & 0xFFu), 127 + FP8_SCALE_EXP_MIN), 247);
          const float sig = __uint_as_float(static_cast<uint32_t>(ef) << 23);
          inv_sig = __uint_as_float(static_cast<uint32_t>(254 - ef) << 23);
          const float et = static_cast<float>(ef - 127);
          // x' = scale*log2(e) * (sigma_t sigma_q S_lat + S_rope) + log2 sigma_t
#pragma unroll
          for (int n = 0; n < NC; ++n) {
            const float s = fmaf(__uint_as_float(vl[n]) * sig, qs[n], __uint_as_float(vr[n]));
            x[n] = (tok < L - dlim[n / 16]) ? fmaf(s, p.scale_log2, et) : -INFINITY;
          }
        }
        if (K::P_SEP) {
          // the scores are done with the RoPE slot and the scales are read
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->r_empty[rslot]));
        }
        bool need = false;
#pragma unroll
        for (int n = 0; n < NC; ++n) need |= x[n] > m_run[n] + RESCALE8_LOG2;
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
            // the previous tile's P.C products (issued after this tile's
            // scores) accumulate into O: wait for them before rescaling it
            if (!(ok = mbar_wait(smem_u32(&ctl->pc_done), (tile_i - 1) & 1, abort, p.status))) break;
            tc_fence_after();
#pragma unroll 1
            for (int mh = 0; mh < (K::STACK_O ? 8 : 4); ++mh) {
              // m-tile mh (or, stacked, half mh & 1 of m-tile mh / 2)
              const uint32_t ocol = K::STACK_O ? (mh >> 1) * K::OW + (mh & 1) * N : mh * N;
#pragma unroll
              for (int k = 0; k < NC / CW; ++k) {
                uint32_t v[CW];
                const uint32_t ta = tmem + lane_addr + ocol + cb + CW * k;
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
        // P' = 2^(x' - m + 8) as e4m3 hi + lo; l accumulates P' / sigma_t. Row
        // cb + n of P'^T holds the 128 token bytes of query row cb + n (hi at
        // s_p, lo at s_p + QG), chunk q of row r at q ^ (r % 8).
        const uint32_t s_p = K::P_SEP ? s_pb + (tile_i & 1) * 2 * K::QG : s_r + rslot * R_BYTES;
#pragma unroll
        for (int c4 = 0; c4 < NC / 4; ++c4) {
          float pv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int n = 4 * c4 + k;
            const float m = m_run[n];
            pv[k] = fast_exp2(x[n] - (m == -INFINITY ? 0.f : m - P_SHIFT));
          }
          uint32_t h0, l0, h1, l1;
          constexpr float PLO = K::STACK_O ? LO_SCALE : 1.f;
          const float2 r0 = split_e4m3x2(pv[0], pv[1], h0, l0, PLO);
          const float2 r1 = split_e4m3x2(pv[2], pv[3], h1, l1, PLO);
          // the normaliser sums the weights the e4m3 parts stand for, so the
          // output is a convex combination of the tile's rows
          lrow[4 * c4] += r0.x * inv_sig;
          lrow[4 * c4 + 1] += r0.y * inv_sig;
          lrow[4 * c4 + 2] += r1.x * inv_sig;
          lrow[4 * c4 + 3] += r1.y * inv_sig;
          const uint32_t whi = quad_transpose(h0 | (h1 << 16), qi);
          const uint32_t wlo = quad_transpose(l0 | (l1 << 16), qi);
          const int nr = cb + 4 * c4 + qi;
          const uint32_t a = s_p + nr * 128 + ((((tq >> 4) ^ nr) & 7) << 4) + (tq & 15);
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(whi) : "memory");
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(a + K::QG), "r"(wlo) : "memory");
        }
        if (L - tau * TILE < TILE) {
          // Cache rows past the sequence end may hold anything (NaN codes
          // included): zero them so that 0 * garbage cannot reach P'.C. Every
          // softmax thread takes 16-byte chunks in order (eight consecutive
          // threads fill one 128-byte row), so a warp's stores hit distinct banks.
          const int r0 = L - tau * TILE > 0 ? L - tau * TILE : 0;
          const int total = (TILE - r0) * 32;        // 32 chunks per row (4 groups x 8)
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
          for (int idx = grp * 128 + t; idx < total; idx += 128 * K::GR) {
            const int row = r0 + (idx >> 5), mt = (idx >> 3) & 3;
            const uint32_t a = s_g + ((g_i + mt) % K::NG) * G_BYTES + row * 128 + (idx & 7) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(z.x), "r"(z.y), "r"(z.z), "r"(z.w)
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[sb]));
        if (t == 0 && grp == 0) T8(5, tile_i);
        if (lane == 0 && grp == 1 && sw == 0) T8(10, tile_i);
        if (lane == 0 && grp == 0 && sw == 3) T8(11, tile_i);
        g_i += 4;
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
        uint32_t v[NC], vh[K::STACK_O ? NC : 1];
        const uint32_t obuf = tmem + lane_addr + mt * K::OW + cb;
#pragma unroll
        for (int k = 0; k < NC / CW; ++k) {
          tmem_ld_w<CW>(obuf + CW * k, v + CW * k);
          if (K::STACK_O) tmem_ld_w<CW>(obuf + N + CW * k, vh + CW * k);
        }
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < NC / CW; ++k) {
          reg_fence_w<CW>(v + CW * k);
          if (K::STACK_O) reg_fence_w<CW>(vh + CW * k);
        }
#pragma unroll
        for (int n = 0; n < NC; ++n) {
          const float o = K::STACK_O ? __uint_as_float(v[n]) + __uint_as_float(vh[n]) * (1.f / LO_SCALE)
                                     : __uint_as_float(v[n]);
          __stcg(obase + (long long)n * D_C + mt * 128 + t, o * ctl->linv[cb + n]);
        }
      }
      if (t < NC) {
        // l = 2^(8 - m) sum_t 2^x_t (x in log2 units), so log2 sum = m - 8 + log2 l
        const float l = ctl->lsum[cb + t];
        const float lse = l > 0.f ? (m_run[t] - P_SHIFT + __log2f(l)) * LN2 : -INFINITY;
        (final_out ? p.lse : p.ws_lse)[row0 + cb + t] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->o_empty));
      named_bar_sync(gbar, 128);
      ++item_i;
    }
  }

  if (threadIdx.x == 128) T8CTA(2);
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, K::TMEM_COLS);
  }
  if (threadIdx.x == 64) T8CTA(3);
}

size_t attn8_smem_bytes(int N) {
  switch (N) {
    case 16: return Cfg8<16>::SMEM;
    case 32: return Cfg8<32>::SMEM;
    case 64: return Cfg8<64>::SMEM;
    default: return 0;
  }
}

cudaError_t attn8_prepare(int N) {
  const int smem = static_cast<int>(attn8_smem_bytes(N));
  switch (N) {
    case 16: return cudaFuncSetAttribute(decode_attn_fp8_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 32: return cudaFuncSetAttribute(decode_attn_fp8_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 64: return cudaFuncSetAttribute(decode_attn_fp8_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_attn_fp8(const CUtensorMap& tm_c8, const CUtensorMap& tm_sc, const CUtensorMap& tm_qr,
                                   const AttnParams& p, cudaStream_t s) {
  if (p.B > MAX_SEQS) return cudaErrorInvalidValue;
  const size_t smem = attn8_smem_bytes(p.N);
  const dim3 grid(p.U * p.C);
  switch (p.N) {
    case 16:
      return launch_pdl(decode_attn_fp8_kernel<16>, grid, dim3(Cfg8<16>::THREADS), smem, s, tm_c8, tm_sc, tm_qr, p);
    case 32:
      return launch_pdl(decode_attn_fp8_kernel<32>, grid, dim3(Cfg8<32>::THREADS), smem, s, tm_c8, tm_sc, tm_qr, p);
    case 64:
      return launch_pdl(decode_attn_fp8_kernel<64>, grid, dim3(Cfg8<64>::THREADS), smem, s, tm_c8, tm_sc, tm_qr, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
