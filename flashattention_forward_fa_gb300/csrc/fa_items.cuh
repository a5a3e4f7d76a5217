// Work decomposition of the prefill kernel, shared with host-side checks: per-sequence geometry,
// the K/V tiles a 128-row Q tile sees, the work items (two Q tiles that read one K/V head) and
// their order over the persistent CTAs.  Plain integer arithmetic, callable on host and device.
#pragma once

#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

struct SeqInfo {
  int q_row0, Lq, rows_out, k_row0, Lk;
  long long lse_row0;  // LSE index of row 0 of this (sequence, head)
};

__host__ __device__ __forceinline__ SeqInfo seq_info(const PrefillParams& p, int b, int h) {
  SeqInfo s;
  if (p.cu_q) {
    int q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    // cu_seqlens that disagree with the totals and maxima the launch was sized for would send the
    // plain stores (LSE, ragged rows) past the outputs: report it and skip the sequence.
    if (!(0 <= q0 && q0 <= q1 && q1 <= p.total_q && q1 - q0 <= p.Nq && 0 <= k0 && k0 <= k1 &&
          k1 <= p.total_k && k1 - k0 <= p.Nk)) {
#ifdef __CUDA_ARCH__
      atomicOr(p.err, kDevErrBounds);
#endif
      q0 = q1 = k0 = k1 = 0;
    }
    s.q_row0 = q0;
    s.Lq = q1 - q0;
    s.k_row0 = k0;
    s.Lk = k1 - k0;
    s.rows_out = s.Lq;
    s.lse_row0 = (long long)h * p.total_q + s.q_row0;
  } else {
    s.q_row0 = b * p.Nq;
    s.k_row0 = b * p.Nk;
    s.Lq = p.seqlens_q ? min(max(p.seqlens_q[b], 0), p.Nq) : p.Nq;
    s.Lk = p.seqlens_k ? min(max(p.seqlens_k[b], 0), p.Nk) : p.Nk;
    s.rows_out = p.Nq;
    s.lse_row0 = ((long long)b * p.Hq + h) * p.Nq;
  }
  return s;
}

// The K/V tiles one 128-row Q tile can see.
struct QTileRange {
  int q0;                // first row (within the sequence)
  int rows_valid;        // rows < Lq in this tile
  int pos_min, pos_max;  // absolute positions of its first / last valid row
  int t0, t1;            // visible K/V tiles [t0, t1); empty when t0 >= t1
};

template <int BM, int BN>
__host__ __device__ __forceinline__ QTileRange qtile_range(const SeqInfo& s, int q0, int causal, int window) {
  QTileRange r;
  r.q0 = q0;
  r.rows_valid = max(0, min(BM, s.Lq - q0));
  r.pos_min = q0 + s.Lk - s.Lq;
  r.pos_max = q0 + r.rows_valid - 1 + s.Lk - s.Lq;
  int lo = 0, hi = s.Lk;
  if (causal) hi = min(hi, r.pos_max + 1);
  if (window > 0) {
    lo = max(lo, r.pos_min - window + 1);
    if (!causal) hi = min(hi, r.pos_max + window);
  }
  if (r.rows_valid > 0 && hi > lo) {
    r.t0 = lo / BN;
    r.t1 = (hi + BN - 1) / BN;
  } else {
    r.t0 = r.t1 = 0;
  }
  return r;
}

// Does K/V tile [k0, k0 + BN) hold a key that some valid row of the tile may not see?
template <int BN>
__host__ __device__ __forceinline__ bool tile_needs_mask(const QTileRange& r, int k0, int Lk, int causal, int window) {
  bool m = (k0 + BN > Lk);
  if (causal) m |= (k0 + BN - 1 > r.pos_min);
  if (window > 0) {
    m |= (k0 < r.pos_max - window + 1);
    if (!causal) m |= (k0 + BN - 1 > r.pos_min + window - 1);
  }
  return m;
}

// The keys row position `pos` may see form one interval [lo, hi): causal keeps j <= pos, a
// window keeps j > pos - window (and, without causal, j < pos + window), every row keeps j < Lk.
__host__ __device__ __forceinline__ void visible_keys(int pos, int Lk, int causal, int window, int& lo, int& hi) {
  lo = 0;
  hi = Lk;
  if (causal) hi = min(hi, pos + 1);
  if (window > 0) {
    lo = max(lo, pos - window + 1);
    if (!causal) hi = min(hi, pos + window);
  }
}

// One work item: two 128-row Q tiles of one sequence that read the same K/V head.  Without
// grouping (one query head per KV head) they are consecutive row tiles of one query head; with an
// even number of query heads per KV head they are the same rows of two query heads of one group,
// whose K/V ranges and masks are then identical (no step of the walk feeds only one tile).
struct WorkItem {
  int h, q0;       // tile A: query head, first row (tile B: item_head / item_row0)
  SeqInfo s;       // lse_row0 for tile A's head
  QTileRange ra, rb;
  int u0, u1;  // union of the two tiles' K/V tile ranges (contiguous: tile B's rows equal or
               // follow tile A's, so B's first visible key is at most one past A's last); empty if u0 >= u1
  bool live;   // the block holds output rows (q0 < rows_out)
};

// Item w: head (pair) fastest, then sequence, then row block; masked problems (causal or window)
// take the blocks latest-first, which is heaviest-first for causal.
template <int BM, int BN>
__host__ __device__ __forceinline__ WorkItem work_item(const PrefillParams& p, int w) {
  WorkItem it;
  const bool hp = p.pair_heads != 0;
  const int nh = hp ? p.Hq / 2 : p.Hq;
  const int hh = w % nh;
  const int rest = w / nh;
  const int b = rest % p.B;
  const int j = rest / p.B;
  const int qblk = (p.causal || p.window > 0) ? p.n_qblk - 1 - j : j;
  it.h = hp ? 2 * hh : hh;
  it.q0 = qblk * (hp ? BM : 2 * BM);
  it.s = seq_info(p, b, it.h);
  it.live = it.q0 >= 0 && it.q0 < it.s.rows_out;  // never a block outside the rows
  it.ra = qtile_range<BM, BN>(it.s, it.q0, p.causal, p.window);
  it.rb = qtile_range<BM, BN>(it.s, hp ? it.q0 : it.q0 + BM, p.causal, p.window);
  const bool act_a = it.ra.t1 > it.ra.t0, act_b = it.rb.t1 > it.rb.t0;
  it.u0 = act_a ? (act_b ? min(it.ra.t0, it.rb.t0) : it.ra.t0) : (act_b ? it.rb.t0 : 0);
  it.u1 = act_a ? (act_b ? max(it.ra.t1, it.rb.t1) : it.ra.t1) : (act_b ? it.rb.t1 : 0);
  return it;
}

// Tile X's query head and first row (tile B: the next head of the pair, or the next row tile).
template <int BM>
__host__ __device__ __forceinline__ int item_head(const PrefillParams& p, const WorkItem& it, int X) {
  return it.h + (X && p.pair_heads ? 1 : 0);
}
template <int BM>
__host__ __device__ __forceinline__ int item_row0(const PrefillParams& p, const WorkItem& it, int X) {
  return it.q0 + (X && !p.pair_heads ? BM : 0);
}

// The k-th item of CTA c of G: a snake over the resident CTAs (round k runs forward for even k,
// backward for odd k), which evens out the decreasing costs of heaviest-first items.  -1 when
// round k has no item for this CTA.
__host__ __device__ __forceinline__ int snake_item_of(int k, int n_items, long long G, long long c) {
  const long long w = (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
  return w < n_items ? (int)w : -1;
}

// P handoffs of tile X over this CTA's items: one per K/V tile of the tile's walk.  The softmax
// warps of tile X and the MMA issuer both make exactly this many (named barrier 1 + X).
template <int BM, int BN>
__host__ __device__ __forceinline__ uint32_t handoffs_total_of(const PrefillParams& p, int X, int n_rounds, int n_items,
                                                               long long G, long long c) {
  uint32_t n = 0;
  for (int k = 0; k < n_rounds; ++k) {
    const int w = snake_item_of(k, n_items, G, c);
    if (w < 0) continue;
    const WorkItem it = work_item<BM, BN>(p, w);
    if (!it.live) continue;
    const QTileRange r = X ? it.rb : it.ra;
    if (r.t1 > r.t0) n += (uint32_t)(r.t1 - r.t0);
  }
  return n;
}

}  // namespace fa
