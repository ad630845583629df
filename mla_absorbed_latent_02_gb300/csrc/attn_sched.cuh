// Split-KV scheduling shared by the decode attention kernels (bf16 and FP8
// caches): the flattened list of (sequence, 128-token tile) pairs is cut into U
// equal contiguous ranges, one per unit; every role of a CTA walks its unit's
// (sequence, tile range) items in the same order.
#pragma once

#include "mla_kernels.cuh"
#include "mla_ptx.cuh"

namespace mla {

MLA_DEV int seq_len(const int32_t* lens, int Hq, int b) {
  const int L = lens[b];
  return L >= Hq ? L : 0;   // lengths below Hq are rejected (combine flags them)
}
MLA_DEV int ntiles(int L) { return L > 0 ? (L + TILE - 1) / TILE : 0; }

// Units: T tiles cut into U contiguous ranges of q = T / U tiles, the first
// r = T % U of them one tile longer. The longer ranges go to the lowest unit
// numbers, i.e. to the CTAs that are launched (and start) first.
MLA_DEV long long unit_start(long long u, long long T, int U) {
  const long long q = T / U, r = T % U;
  return u * q + (u < r ? u : r);
}

// Unit whose tile range [unit_start(u), unit_start(u + 1)) holds global tile x (x < T).
MLA_DEV int unit_of(long long x, long long T, int U) {
  const long long q = T / U, r = T % U;
  const long long big = r * (q + 1);
  return static_cast<int>(x < big ? x / (q + 1) : r + (x - big) / q);
}

// Tile prefix over the sequences, computed once per CTA by all its threads:
// pre[b] = sum_{i<b} ntiles(L_i), pre[B] = T. The loads of the lengths are
// independent (one latency for the whole CTA, not one per sequence).
MLA_DEV void tile_prefix(const AttnParams& p, int* pre, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (p.B + blockDim.x - 1) / blockDim.x;   // <= MAX_SEQS / 256
  int n[MAX_SEQS / 256];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < MAX_SEQS / 256; ++i) {
    const int b = tid * per + i;
    n[i] = (i < per && b < p.B) ? ntiles(seq_len(p.seq_lens, p.Hq, b)) : 0;
    sum += n[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < w; ++i) base += warp_tot[i];
  int run = base + incl - sum;   // exclusive prefix of this thread's first sequence
  if (tid == 0) pre[0] = 0;
#pragma unroll
  for (int i = 0; i < MAX_SEQS / 256; ++i) {
    const int b = tid * per + i;
    if (i < per && b < p.B) {
      run += n[i];
      pre[b + 1] = run;
    }
  }
  __syncthreads();
}

// Walks the (sequence, tile range) items of one unit, in order. With a single
// unit (nothing split) the tile range of row group c stops at the last tile its
// latest query token attends: sequence positions below L - dlim (bottom-right
// causal), so a CTA of early prompt tokens skips the tiles no row of it sees.
struct ItemIter {
  const int* pre;
  const int32_t* lens;
  int B, Hq;
  long long T, s, e;
  int b;
  int dlim;   // -1: the whole range
  MLA_DEV void init(const AttnParams& p, const int* pre_, int u, int c) {
    pre = pre_;
    lens = p.seq_lens;
    B = p.B;
    Hq = p.Hq;
    T = pre[B];
    s = unit_start(u, T, p.U);
    e = unit_start(u + 1, T, p.U);
    dlim = -1;
    if (p.U == 1) {
      const int jmax = min(p.Hq - 1, (c * p.N + p.N - 1) / p.H);
      dlim = p.Hq - 1 - jmax;
    }
    // first sequence with pre[b+1] > s
    int lo = 0, hi = B;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid + 1] > s) hi = mid;
      else lo = mid + 1;
    }
    b = lo;
  }
  // item: sequence ob (length L), tiles [t0, t1); global tile index of ob's first tile is oacc
  MLA_DEV bool next(int& ob, int& t0, int& t1, int& L, long long& oacc) {
    if (s >= e) return false;
    while (b < B && pre[b + 1] <= s) ++b;
    if (b >= B) return false;
    L = seq_len(lens, Hq, b);
    const long long end = min(e, (long long)pre[b + 1]);
    ob = b;
    t0 = static_cast<int>(s - pre[b]);
    t1 = static_cast<int>(end - pre[b]);
    if (dlim >= 0) t1 = min(t1, ntiles(L - dlim));   // >= 1 = t0 + 1: L >= Hq > dlim
    oacc = pre[b];
    s = end;
    return true;
  }
};


}  // namespace mla
