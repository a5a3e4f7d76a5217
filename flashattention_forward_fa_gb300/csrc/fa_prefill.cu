// Fused attention forward (prefill / encoder) for sm_103a.
//
// What it computes: O = softmax(Q K^T * scale + mask) V and the row LSE, with the
// running-max / running-sum softmax, so scores never leave the SM — the fused
// tiled evaluation of the jsqmd page "CANN Transformer算子库ops-transformer深度实践",
// §二 "FlashAttention的融合计算思想" (Q split by rows, K/V by columns, every Q block
// sweeps all K/V blocks on chip) with the max-subtracted fp32 softmax of the
// hwcomputing.csdn.net page, §2.2 "数值稳定性优化" (the page carries the row maximum from one
// block to the next; here that is a running max whose changes rescale the accumulator).
//
// How (GB300-first; the pages' Cube/Vector double buffer is only prior art):
//   persistent: one CTA per SM walks its share of the work items (a snake over the
//   CTAs of the heaviest-first item list); one item = two 128-row Q tiles (A, B) of
//   one sequence that read the same K/V: consecutive row tiles of one query head, or,
//   with an even number of query heads per KV head, the same rows of two heads of one
//   group (identical K/V ranges and masks).  The K/V rings and every barrier phase run on across
//   items, so the next item's Q load (each tile's Q as soon as that tile's last S of the
//   current item has run), K/V loads and first S overlap the current item's last P V and
//   epilogue instead of a CTA launch, TMEM allocation and pipeline fill per item.  12 warps:
//     warps 0-3   softmax of tile A: thread r owns score row r (TMEM lane r)
//     warps 4-7   softmax of tile B
//     warp  8     TMA producer for Q (each tile's Q once per item) and the K ring
//     warp  9     TMA producer for the V ring
//     warp  10    TMEM allocator and tcgen05.mma issuer
//     warp  11    idle (gives its registers to the softmax warpgroups)
//   TMEM holds S_A, S_B (128 fp32 columns each) and O_A, O_B (d columns each).
//   The tensor core ping-pongs between the tiles in the order
//       PV_A(t), S_A(t+1), PV_B(t), S_B(t+1), PV_A(t+1), ...
//   so while one warpgroup exponentiates its scores the tensor core runs the
//   other tile's two GEMMs.  P_X(t) (bf16) is written back over S_X(t) in TMEM
//   and read from there as the A operand of PV_X(t); O accumulates in TMEM.
//   Because S_X(t+1) is issued after PV_X(t), the completion of S_X(t+1) also
//   means O_X already holds PV_X(t): the softmax may rescale O_X without a wait.
//   The rescale is rare: O is divided by the sum of the very (bf16) weights P V used,
//   so the exponent base only has to keep the weights finite.  A row's base is set
//   from its first tile's max; later tiles are exponentiated against it without
//   reducing their max, unless their weights would sum past 2^57, in which case the
//   tile's max is taken, O rescaled and the tile exponentiated again.
//   Per step the issuer waits for the step's V and next K first, then for each P in
//   turn, so no wait sits between a P and its P V.  A P reaches the issuer through a
//   named barrier shared by the tile's four softmax warps and the issuer warp, not an
//   mbarrier: barrier-unit traffic does not queue behind the S GEMMs' shared-memory
//   operand reads, which held an mbarrier handoff back by ~450 cycles per tile.  A
//   named barrier has no time limit, so both sides count their handoffs and, after an
//   abort, complete the rest without work (handoffs_total).  The epilogue stages a tile's O
//   in shared memory (64 columns at a time, in the TMA layout) and writes it with
//   TMA stores; a ragged tile stores row by row.
//   With ALiBi (jsqmd page, §三 "ALiBi位置编码的线性偏置") each score gets
//   -m_h |p - j| (p the query's absolute position) right after masking, folded into
//   the same fused multiply-add that applies the softmax scale.
//   With RoPE (jsqmd page, §三 "融合位置编码的Attention计算") the softmax warps rotate
//   the next item's Q tile in shared memory as soon as it lands (rotate_q_tile), before
//   its first S_X; K arrives rotated (a K tile is read by every CTA of its head, so it is
//   rotated once, not per CTA).
//   Each Q tile visits only the K/V tiles its rows can see (causal / window
//   tiles that are fully masked are never loaded or multiplied).  With ALiBi
//   the walk starts at the last tile: the diagonal, where ALiBi scores peak,
//   sets the running max early, so later tiles rarely move it and O is rarely
//   rescaled; otherwise it starts at the first, so the CTAs of one head stream
//   the same early K/V tiles at about the same time and share them in L2.  Only
//   tiles crossing a mask edge or the ragged tail evaluate the mask.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_internal.h"
#include "fa_items.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// TMA load with an L2 eviction-priority hint (a policy from createpolicy).
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                                 int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5}], "
      "[%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy(bool keep) {
  uint64_t p;
  if (keep) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// The producers' loads: with ALiBi (items walk their tiles last to first) K and V are marked to
// stay in L2 and Q to leave it first (measured 2.7 % faster there; neutral to 1 % slower on
// forward walks, which keep the plain loads).
template <bool HINT>
__device__ __forceinline__ void tma_load_3d_walk(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  if (HINT) tma_load_3d_hint(dst, map, bar, c0, c1, c2, policy);
  else tma_load_3d(dst, map, bar, c0, c1, c2);
}

// Threads at a P handoff (named barrier 1 + X): tile X's four softmax warps and the MMA issuer warp.
constexpr uint32_t kNamedBarThreads = 5 * 32;

// Named barrier `id` (1-15) for `count` threads (a multiple of 32), whole warps converged.
// Unlike the bounded mbarrier waits it has no time limit: it is used only where every party
// makes the same number of calls on every path, aborts included.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;  // query rows per Q tile (one TMEM lane each)
  static constexpr int NQT = 2;   // Q tiles per CTA
  static constexpr int BN = 128;  // keys per K/V tile
  static constexpr int KST = (D == 128) ? 2 : 3;
  static constexpr int VST = (D == 128) ? 2 : 3;
  static constexpr int CHUNK = 128 * 128;  // bytes of one 64-column swizzled slab of a 128-row tile
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  // O staging, one buffer per tile: a 64-column box of its 128 rows in the layout TMA stores from
  static constexpr int OFF_OST = OFF_V + VST * KV_BYTES;
  static constexpr int O_BOX = BM * 64 * 2;
  static constexpr int OFF_BAR = OFF_OST + NQT * O_BOX;
  // barriers: q[2], k_full[KST], k_empty[KST], v_full[VST], v_empty[VST],
  //           s_full[2], o_final[2], mma_done, q_ready[2], q_empty[2], o_free[2], o_staged[2]
  static constexpr int NBAR = 2 + 2 * KST + 2 * VST + 2 + 2 + 1 + 2 + 2 + 2 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;     // S_X at COL_S + 128 X
  static constexpr uint32_t COL_O = 256;   // O_X at COL_O + D X
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 0, 1);   // P K-major (TMEM), V MN-major
  // Registers per thread after the split (setmaxnreg): the softmax warpgroups grow, the
  // producer warpgroup shrinks.  Chosen so that neither side spills for either head dim (at
  // d=128, 216/72 measured 0.7 % faster than 200/96 without options, 1.7 % with ALiBi).
  static constexpr int REGS_SOFTMAX = (D == 128) ? 216 : 208;
  static constexpr int REGS_PRODUCER = 72;
  static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_PRODUCER <= THREADS * (65536 / THREADS / 8 * 8),
                "register split exceeds the launch allocation");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

template <int D>
__device__ __forceinline__ void store_row_zero(const PrefillParams& p, const SeqInfo& s, int h, int i) {
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)(s.q_row0 + i) * p.Hq + h) * D;
  uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
  if (p.lse) p.lse[s.lse_row0 + i] = -INFINITY;
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// This CTA's k-th item, and its P handoffs of tile X (see snake_item_of, handoffs_total_of).
__device__ __forceinline__ int snake_item(int k, int n_items) { return snake_item_of(k, n_items, gridDim.x, blockIdx.x); }
template <int BM, int BN>
__device__ __forceinline__ uint32_t handoffs_total(const PrefillParams& p, int X, int n_rounds, int n_items) {
  return handoffs_total_of<BM, BN>(p, X, n_rounds, n_items, gridDim.x, blockIdx.x);
}

// RoPE: rotate Q_X of item `iq` in place once its Q has landed (bar_q phase `ph`) — 16-byte
// chunks of the 128-byte swizzled rows the TMA wrote, four adjacent pairs per chunk — and tell the
// MMA issuer (q_ready[X]).  Warp w of the warpgroup takes rows 32 (w & 3) .. 32 (w & 3) + 31, two
// per step: lanes 0-15 the chunks of one row, lanes 16-31 those of the next, so that a warp's
// table load reads 512 contiguous bytes (a table row holds rope_dim / 8 float4 of cos, the same of
// sin).  Four steps' loads are issued before their stores (Q is reached through a generic pointer,
// so the compiler never moves a load above an earlier store); a lane with nothing to rotate loads
// table entry 0 and stores nothing.  Returns false if the wait gave up.
template <int D>
__device__ __forceinline__ bool rotate_q_tile(const PrefillParams& p, const WorkItem& iq, uint32_t ph, int X, int warp,
                                              int lane, uint8_t* sQ, uint64_t* bar_q, uint64_t* q_ready,
                                              volatile int* abort_flag) {
  using C = PrefillCfg<D>;
  const bool good = __all_sync(0xffffffffu, mbar_wait(bar_q, ph & 1, abort_flag, p.err));
  if (good) {
    const QTileRange rq = X ? iq.rb : iq.ra;
    const int nch = p.rope_dim / 8;  // chunks per row to rotate (at most D / 8 <= 16)
    const int c = lane & 15;
    const int shift = iq.s.Lk - iq.s.Lq;
    const float4* cos4 = reinterpret_cast<const float4*>(p.rope_cos);
    const float4* sin4 = reinterpret_cast<const float4*>(p.rope_sin);
    uint8_t* qt = sQ + X * C::Q_BYTES;
#pragma unroll 1
    for (int kb = 0; kb < 16; kb += 4) {
      float4 cv[4], sv[4];
      uint32_t qoff[4];
      uint32_t live = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = (warp & 3) * 32 + 2 * (kb + u) + (lane >> 4);  // row within the tile
        const int i = rq.q0 + row, pos = i + shift;
        const bool in = c < nch && i < iq.s.Lq;
        const bool okp = in && pos >= 0 && pos < p.rope_rows;
        if (in && !okp) atomicOr(p.err, kDevErrBounds);  // no table row for this position
        const size_t tix = okp ? (size_t)pos * nch + c : 0;
        cv[u] = __ldg(cos4 + tix);
        sv[u] = __ldg(sin4 + tix);
        qoff[u] = (uint32_t)((c >> 3) * C::CHUNK + row * 128 + (((c & 7) ^ (row & 7)) << 4));
        live |= (okp ? 1u : 0u) << u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((live >> u) & 1u) {
          uint4* ch = reinterpret_cast<uint4*>(qt + qoff[u]);
          *ch = rope_rotate4(*ch, cv[u], sv[u]);
        }
    }
  }
  fence_async_smem();  // the MMA reads Q through the async proxy
  __syncwarp();
  if (lane == 0) mbar_arrive(&q_ready[X]);
  return good;
}

// PADK: padded layout with per-sequence key lengths, where K/V rows past a sequence's keys are
// in-bounds caller memory (see the zeroing of V below); other layouts compile without that code.
template <int D, bool ALIBI, bool ROPE, bool PADK>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const PrefillParams p) {
  using C = PrefillCfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = (p.pair_heads ? p.Hq / 2 : p.Hq) * p.B * p.n_qblk;  // as the launcher counts them
  const int n_rounds = (int)(((long long)n_items + gridDim.x - 1) / gridDim.x);
  constexpr bool rev = ALIBI;  // walk each item's K/V tiles last to first
  constexpr int REGS_S = C::REGS_SOFTMAX, REGS_P = C::REGS_PRODUCER;  // register split after setmaxnreg
  static_assert(2 * 128 * REGS_S + 128 * REGS_P <= C::THREADS * (65536 / C::THREADS / 8 * 8), "register split");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_q = bars;               // [2]: Q_X of an item landed
  uint64_t* k_full = bar_q + 2;
  uint64_t* k_empty = k_full + C::KST;
  uint64_t* v_full = k_empty + C::KST;
  uint64_t* v_empty = v_full + C::VST;
  uint64_t* s_full = v_empty + C::VST;  // [2]: one completion per S of tile X
  uint64_t* o_final = s_full + 2;       // [2]: one completion per item, the last PV of tile X
  uint64_t* mma_done = o_final + 2;
  uint64_t* q_ready = mma_done + 1;     // [2]: four warp arrivals once Q_X is rotated (RoPE only)
  uint64_t* q_empty = q_ready + 2;      // [2]: every S of tile X in an item has run: Q_X may be overwritten
  uint64_t* o_free = q_empty + 2;       // [2]: tile X's last O store has read its staging buffer
  uint64_t* o_staged = o_free + 2;      // [2]: four warp arrivals once a box of tile X's O rows is staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(&bar_q[0], 1);
    mbar_init(&bar_q[1], 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&o_final[i], 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(&q_ready[0], 4);
    mbar_init(&q_ready[1], 4);
    mbar_init(&q_empty[0], 1);
    mbar_init(&q_empty[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_free[i], 1);
      mbar_init(&o_staged[i], 4);
    }
    fence_barrier_init();
  }
  if (warp == 10) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Every role walks the same item sequence and derives the same per-item facts, so the
  // barrier phases below are running counts that continue from one item to the next.
  if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    setmaxnreg_inc<REGS_S>();
    const int X = warp >> 2;               // 0: tile A, 1: tile B
    const int rg = tid & 127;              // row within the tile = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t colS = C::COL_S + 128u * X, colO = C::COL_O + (uint32_t)D * X;
    // scores are scaled into log2 units by sl2; with ALiBi the scale is applied together with
    // the bias below and everything after works on already-scaled scores (xs = 1)
    const float sl2 = p.scale_log2;
    const float xs = ALIBI ? 1.0f : sl2;
    uint32_t n_sx = 0;  // S tiles of this warpgroup so far (s_full phase; P handoffs made)
    uint32_t n_ox = 0;  // items in which this tile was active (o_final phase)
    uint32_t n_q = 0;   // items that loaded Q (bar_q[X] phase)
    uint32_t v_next = 0;  // V ring index of the next item's first tile
    uint32_t n_box = 0;   // O boxes of this tile staged and stored so far (o_staged / o_free phase)
    int rot_k = -1;     // RoPE: the round whose item already has this tile's Q rotated
    bool ok = true;
    // RoPE rotation of Q_X (rotate_q_tile).  bar_q phases are waited strictly in order (a parity
    // wait more than one phase ahead would pass early), so a tile with no rows in an item still
    // waits its phase.
    auto rotate_q = [&](const WorkItem& iq, uint32_t ph) -> bool {
      return rotate_q_tile<D>(p, iq, ph, X, warp, lane, sQ, bar_q + X, q_ready, abort_flag);
    };
    for (int k = 0; ok && k < n_rounds; ++k) {
      const int w = snake_item(k, n_items);
      if (w < 0) continue;
      const WorkItem it = work_item<C::BM, C::BN>(p, w);
      if (!it.live) continue;
      SeqInfo s = it.s;
      if (X && p.pair_heads) s.lse_row0 += p.cu_q ? (long long)p.total_q : (long long)p.Nq;  // the next head
      const QTileRange r = X ? it.rb : it.ra;
      const int h = item_head<C::BM>(p, it, X);
      const int i = r.q0 + rg;
      if (it.u1 > it.u0) ++n_q;
      const uint32_t v_first = v_next;  // V ring index of this item's first tile
      if (it.u1 > it.u0) v_next += (uint32_t)(it.u1 - it.u0);
      if (r.t1 <= r.t0) {  // this tile's rows see no key: O = 0, LSE = -inf (and zero padding rows)
        if (ROPE && it.u1 > it.u0) ok = __all_sync(0xffffffffu, mbar_wait(bar_q + X, (n_q - 1) & 1, abort_flag, p.err));
        if (ok && i < s.rows_out) store_row_zero<D>(p, s, h, i);
        continue;
      }
      const int pos = i + s.Lk - s.Lq;
      int row_lo, row_hi;  // this row's visible keys [row_lo, row_hi)
      visible_keys(pos, s.Lk, p.causal, p.window, row_lo, row_hi);
      const float slope2 = ALIBI ? p.alibi[h] * 1.4426950408889634f : 0.f;  // m_h in log2 units
      float m = -INFINITY;  // running max used for exponentiation (log2 units)
      float l = 0.f;        // running sum of exp2(score*sl2 - m) in fp32 (gives the LSE)
      float lr = 0.f;       // running sum of the same weights rounded to bf16 (normalises O)
      if (ROPE && rot_k != k) ok = rotate_q(it, n_q - 1);
      for (int t = rev ? r.t1 - 1 : r.t0; ok && (rev ? t >= r.t0 : t < r.t1); t += rev ? -1 : 1, ++n_sx) {
        const int n = rev ? r.t1 - 1 - t : t - r.t0;  // position of tile t in the walk
        ok = mbar_wait(&s_full[X], n_sx & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sc[C::BN];
        const int k0 = t * C::BN;
        const bool edge = tile_needs_mask<C::BN>(r, k0, s.Lk, p.causal, p.window);
        // Scores of the tile from TMEM, masked (S stays in TMEM until P is stored over it).
        auto load_s = [&]() {
          uint32_t r0[32], r1[32], r2[32], r3[32];
          tmem_ld32(t_lane + colS + 0, r0);
          tmem_ld32(t_lane + colS + 32, r1);
          tmem_ld32(t_lane + colS + 64, r2);
          tmem_ld32(t_lane + colS + 96, r3);
          tmem_ld_wait(r0);
          tmem_ld_wait(r1);
          tmem_ld_wait(r2);
          tmem_ld_wait(r3);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sc[j] = __uint_as_float(r0[j]);
            sc[32 + j] = __uint_as_float(r1[j]);
            sc[64 + j] = __uint_as_float(r2[j]);
            sc[96 + j] = __uint_as_float(r3[j]);
          }
          if (edge) {
            // keep column j iff k0 + j lies in the row's visible interval: one unsigned compare per key
            const uint32_t lo = (uint32_t)(row_lo - k0);
            const uint32_t span = (uint32_t)max(row_hi - row_lo, 0);
#pragma unroll
            for (int j = 0; j < C::BN; ++j)
              if ((uint32_t)j - lo >= span) sc[j] = -INFINITY;
          }
        };
        load_s();
        if (edge) {
          if (PADK && k0 + C::BN > s.Lk) {
            // The tile crosses the end of the sequence's keys: the V rows past it are in-bounds
            // memory the caller may leave as anything, and 0 * NaN is NaN in P V.  Zero them (whole
            // 128-byte rows of each slab, so the swizzle does not matter) once V has landed; the
            // P handoff below orders this before the first P V that reads the tile.  Both
            // warpgroups may do it for the same tile; writing zeros over zeros changes nothing.
            const uint32_t g = v_first + (uint32_t)(rev ? it.u1 - 1 - t : t - it.u0);
            ok = __all_sync(0xffffffffu, mbar_wait(&v_full[g % C::VST], (g / C::VST) & 1, abort_flag, p.err));
            if (ok) {
              uint8_t* vt = sV + (g % C::VST) * C::KV_BYTES;
              const int nvalid = s.Lk - k0;
              for (int idx = rg; idx < (C::BN - nvalid) * (D / 8); idx += 128) {
                const int row = nvalid + idx / (D / 8), c16 = idx % (D / 8);
                *reinterpret_cast<uint4*>(vt + (c16 >> 3) * C::CHUNK + row * 128 + ((c16 & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
              fence_async_smem();  // the MMA reads V through the async proxy
            }
          }
        }
        bool lin = false;           // ALiBi bias added in the exponent
        float ba = 0.f, bc = 0.f;   // b_j = ba j + bc (log2 units)
        float xs_t = xs;            // scale applied in the exponent's FMA
        // P V runs on bf16-rounded weights, so O is normalised by the sum of those same rounded
        // weights (lr): O is then an exact convex combination of V rows, and a rounding error of a
        // weight moves O only by its share times |v_j - O| (a row that sees one key returns that
        // V row exactly).  Normalising by the unrounded sum instead measured up to 1.5e-2 off on
        // rows dominated by two or three keys with |O| ~ 2.  The LSE uses the fp32 sum of the
        // unrounded weights (l): from the rounded sum it would be up to 2.7e-3 off.
        // Exponentiate the tile against base mb into P (bf16 pairs written over S in TMEM, 32 scores
        // at a time); return the fp32 sum of the unrounded weights and add the sum of the rounded
        // ones to *tlr.  Two lanes of fp32 per instruction (fma/add .f32x2) for the scale-and-shift
        // and the sum (two accumulators for short chains).  The scores stay in registers: a tile
        // exponentiated against a base that turns out too low is done again from them.
        auto exp_tile = [&](float mb, float* tlr) -> float {
          const uint64_t sl2x2 = f2_pack(xs_t, xs_t), negm2 = f2_pack(-mb, -mb);
          // ALiBi: exponent addend b_j - m per key pair, eight chains stepping 16 keys
          uint64_t bm[8];
          const uint64_t bstep = f2_pack(16.f * ba, 16.f * ba);
          if (ALIBI) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              bm[u] = f2_pack(fmaf(ba, (float)(2 * u), bc) - mb, fmaf(ba, (float)(2 * u + 1), bc) - mb);
          }
          uint64_t ls[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
          float lr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < C::BN / 32; ++c) {  // 32 scores -> 16 packed columns, stored at once
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(sc[32 * c + 2 * j], sc[32 * c + 2 * j + 1]), sl2x2, ALIBI ? bm[j & 7] : negm2),
                        x0, x1);
              if (ALIBI) bm[j & 7] = f2_add(bm[j & 7], bstep);
              const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
              ls[j & 1] = f2_add(ls[j & 1], f2_pack(e0, e1));
              pk[j] = pack_bf16x2(e0, e1);
              bf16x2_accumulate(lr4[2 * (j & 1)], lr4[2 * (j & 1) + 1], pk[j]);
            }
            tmem_st16(t_lane + colS + 16 * c, pk);
          }
          *tlr = (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]);
          float a0, a1;
          f2_unpack(f2_add(ls[0], ls[1]), a0, a1);
          return a0 + a1;
        };
        // The exponent base m moves only when a tile would otherwise carry weights near the top
        // of the fp32 range.  Because O is divided by the sum of the very weights P V used, the
        // base only has to keep them finite: with the row's first base set from a tile max, later
        // tiles are exponentiated against m without reducing their max first, and only a tile
        // whose weights sum past 2^57 (some score > ~50 log2 units above m; weights, their sums
        // and O stay far below 2^127 for any row length the launch accepts), or a row still
        // without a base, goes through the path below: tile max, O rescaled by 2^(m - m_new),
        // exponentiated again.  The decision is per warp (the TMEM rescale is warp-collective).
        float ts = 0.f, tlr = 0.f;  // this tile's sums of unrounded and of rounded weights
        bool done = false;
        if (!ALIBI && __all_sync(0xffffffffu, m != -INFINITY)) {
          ts = exp_tile(m, &tlr);
          done = __all_sync(0xffffffffu, ts <= 0x1p57f);  // false for inf / NaN too
        }
        if constexpr (ALIBI) {
          // ALiBi (bias -m_h |p - j|, log2 units).  When every key of the tile lies on one side of
          // p — always for causal rows, whose later keys are masked — the bias is linear in the
          // key, b_j = ba j + bc: it is added inside the exponent's FMA by eight chains of paired
          // adds, and a max, where one is taken, is bounded per 16-key chunk (scaled raw chunk max
          // plus the chunk's largest bias).  The bound exceeds the biased max by at most 15 |ba|
          // (below 19 for the steepest slope), which only lowers every weight of the tile by a
          // common factor, and it keeps the bias off the max's critical path.  A tile that p
          // splits (non-causal only) takes |.| per key before the max.  Linear tiles of a row
          // with a base go first without a max, as above: the walk starts at the diagonal, whose
          // tile sets the base, so later tiles rarely need one (3-4 % faster).  One
          // exponentiation site, in a loop of at most two passes (a second copy spilled); the
          // generic path below is then skipped.
          const int dk = pos - k0;
          bool quick = __all_sync(0xffffffffu, (p.causal || dk >= C::BN - 1 || dk <= 0) && m != -INFINITY);
#pragma unroll 1
          for (;;) {
            float mx;
            lin = p.causal || dk >= C::BN - 1 || dk <= 0;
            if (lin) {
              ba = (p.causal || dk > 0) ? slope2 : -slope2;
              bc = -ba * (float)dk;
              xs_t = sl2;
            }
            if (!quick) {
              if (lin) {
                const float jtop = ba >= 0.f ? 15.f : 0.f;  // key of a chunk's largest bias
                float c8[C::BN / 16];
#pragma unroll
                for (int q = 0; q < C::BN / 16; ++q) {
                  const float* v = sc + 16 * q;
                  const float c16 = fmax3(fmax3(fmax3(v[0], v[1], v[2]), fmax3(v[3], v[4], v[5]), fmax3(v[6], v[7], v[8])),
                                          fmax3(v[9], v[10], v[11]), fmax3(fmax3(v[12], v[13], v[14]), v[15], v[15]));
                  c8[q] = fmaf(c16, sl2, fmaf(ba, (float)(16 * q) + jtop, bc));
                }
                mx = fmax3(fmax3(c8[0], c8[1], c8[2]), fmax3(c8[3], c8[4], c8[5]), fmaxf(c8[6], c8[7]));
              } else {
                const float dpos = (float)dk;
#pragma unroll
                for (int j = 0; j < C::BN; ++j) sc[j] = fmaf(sc[j], sl2, -slope2 * fabsf(dpos - (float)j));
                float t8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) t8[u] = fmax3(sc[u], sc[8 + u], sc[16 + u]);
#pragma unroll
                for (int j = 24; j < C::BN - 8; j += 16)
#pragma unroll
                  for (int u = 0; u < 8; ++u) t8[u] = fmax3(t8[u], sc[j + u], sc[j + 8 + u]);
#pragma unroll
                for (int u = 0; u < 8; ++u) t8[u] = fmaxf(t8[u], sc[C::BN - 8 + u]);
                mx = fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7]));
              }
              const float m_new = fmaxf(m, mx);
              const bool need = m_new > m + 8.0f;
              const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
              const bool o_live = need && (n > 0) && (m != -INFINITY);
              if (__any_sync(0xffffffffu, o_live)) {
                const float f = o_live ? alpha : 1.0f;
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                  uint32_t ov[16];
                  tmem_ld16(t_lane + colO + c, ov);
                  tmem_ld_wait(ov);
#pragma unroll
                  for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
                  tmem_st16(t_lane + colO + c, ov);
                }
              }
              if (need) {
                l *= alpha;
                lr *= alpha;
                m = m_new;
              }
            }
            ts = exp_tile((m == -INFINITY) ? 0.f : m, &tlr);
            if (!quick || __all_sync(0xffffffffu, ts <= 0x1p57f)) break;
            quick = false;
          }
          done = true;
        }
        if (!done) {
          float mx;
          {  // row max: eight independent chains of three-input max
            float t8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = fmax3(sc[u], sc[8 + u], sc[16 + u]);
#pragma unroll
            for (int j = 24; j < C::BN - 8; j += 16)
#pragma unroll
              for (int u = 0; u < 8; ++u) t8[u] = fmax3(t8[u], sc[j + u], sc[j + 8 + u]);
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = fmaxf(t8[u], sc[C::BN - 8 + u]);
            mx = fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]), fmaxf(t8[6], t8[7])) * xs;
          }
          const float m_new = fmaxf(m, mx);
          const bool need = m_new > m + 8.0f;  // -inf + 8 = -inf: the first finite max always moves m
          const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
          const bool o_live = need && (n > 0) && (m != -INFINITY);  // O row holds data to rescale
          if (__any_sync(0xffffffffu, o_live)) {
            // S_X(t) was issued after PV_X(t-1), so O_X is current: rescale it in place.
            const float f = o_live ? alpha : 1.0f;
#pragma unroll
            for (int c = 0; c < D; c += 16) {
              uint32_t ov[16];
              tmem_ld16(t_lane + colO + c, ov);
              tmem_ld_wait(ov);
#pragma unroll
              for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
              tmem_st16(t_lane + colO + c, ov);
            }
          }
          if (need) {
            l *= alpha;
            lr *= alpha;
            m = m_new;
          }
          ts = exp_tile((m == -INFINITY) ? 0.f : m, &tlr);
        }
        l += ts;
        lr += tlr;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        named_bar_sync(1 + X, kNamedBarThreads);  // hand P_X(t) to the issuer
      }
      if (ROPE && ok) {
        // Look ahead: when the next item with any work has rows in this tile, rotate its Q now
        // (it lands once this item's last S has run), so the next item's first S can run while
        // this item's epilogue does.
        for (int k2 = k + 1; k2 < n_rounds; ++k2) {
          const int w2 = snake_item(k2, n_items);
          if (w2 < 0) continue;
          const WorkItem it2 = work_item<C::BM, C::BN>(p, w2);
          if (!it2.live || it2.u1 <= it2.u0) continue;
          const QTileRange r2 = X ? it2.rb : it2.ra;
          if (r2.t1 > r2.t0) {
            ok = rotate_q(it2, n_q);
            rot_k = k2;
          }
          break;
        }
      }
      if (ok) {
        ok = mbar_wait(&o_final[X], n_ox & 1, abort_flag, p.err);  // the last PV of this tile finished
        ok = __all_sync(0xffffffffu, ok);
      }
      ++n_ox;
      if (ok) {
        tc_fence_after();
        const bool store = i < s.Lq;
        const float inv = lr > 0.f ? 1.0f / lr : 0.f;
        if (store && p.lse) p.lse[s.lse_row0 + i] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        // 64 columns of this row of O_X (box bx), normalised and packed to bf16 pairs
        auto load_box = [&](int bx, uint32_t (&ow)[32]) {
          uint32_t ov0[32], ov1[32];
          tmem_ld32(t_lane + colO + 64 * bx, ov0);
          tmem_ld32(t_lane + colO + 64 * bx + 32, ov1);
          tmem_ld_wait(ov0);
          tmem_ld_wait(ov1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            ow[j] = pack_bf16x2(__uint_as_float(ov0[2 * j]) * inv, __uint_as_float(ov0[2 * j + 1]) * inv);
            ow[16 + j] = pack_bf16x2(__uint_as_float(ov1[2 * j]) * inv, __uint_as_float(ov1[2 * j + 1]) * inv);
          }
        };
        if (r.q0 + C::BM <= s.Lq) {
          // Every row of the tile lies inside the sequence: stage its O in shared memory, one
          // 64-column box at a time, in the 128-byte swizzled layout of the O tensor map, and write
          // each box with one TMA store (whole lines, instead of one 16-byte piece of 32 rows per
          // store instruction).  The buffer is this tile's own; a box may be staged once the
          // previous box's store has read it (o_free; the wait for the last box of an epilogue is
          // left to the next one).
          uint8_t* stg = sm + C::OFF_OST + X * C::O_BOX;
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx) {
            uint32_t ow[32];
            load_box(bx, ow);
            if (n_box > 0) {
              if (bx == 0 && rg == 0) {
                bulk_wait_read();
                mbar_arrive(&o_free[X]);
              }
              ok = __all_sync(0xffffffffu, mbar_wait(&o_free[X], (n_box - 1) & 1, abort_flag, p.err));
            }
            if (ok) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4*>(stg + rg * 128 + ((q ^ (rg & 7)) << 4)) =
                    make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
              fence_async_smem();  // the TMA store reads the staged rows through the async proxy
              __syncwarp();
              if (lane == 0) mbar_arrive(&o_staged[X]);
              if (rg == 0) {
                ok = mbar_wait(&o_staged[X], n_box & 1, abort_flag, p.err);  // all four warps' rows
                if (ok) {
                  tma_store_3d(&tm_o, stg, bx * 64, h, s.q_row0 + r.q0);
                  bulk_commit();
                  if (bx + 1 < D / 64) {
                    bulk_wait_read();
                    mbar_arrive(&o_free[X]);
                  }
                }
              }
              ok = __all_sync(0xffffffffu, ok);
            }
            ++n_box;
            if (!ok) break;
          }
        } else {
          // A ragged tile stores row by row: its rows past the sequence belong to the next
          // sequence or are padding.
          __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)(s.q_row0 + i) * p.Hq + h) * D;
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx) {
            uint32_t ow[32];
            load_box(bx, ow);  // TMEM loads are warp-wide: every lane takes part, stored or not
            if (store) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                reinterpret_cast<uint4*>(orow)[8 * bx + q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
            }
          }
          if (!store && i < s.rows_out) store_row_zero<D>(p, s, h, i);
        }
      }
    }
    if (!ok) {
      // Aborted (a wait gave up): the issuer may still be at a P handoff of this tile, and a named
      // barrier cannot time out, so make the remaining ones without work.
      const uint32_t total = handoffs_total<C::BM, C::BN>(p, X, n_rounds, n_items);
      for (; n_sx < total; ++n_sx) {
        __syncwarp();
        named_bar_sync(1 + X, kNamedBarThreads);
      }
    }
    if (rg == 0) bulk_wait_all();  // this thread's O stores are complete before the CTA exits
  } else if (warp == 8) {
    // ------------------------------------------------------------ Q + K producer
    setmaxnreg_dec<REGS_P>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      const uint64_t pol_kv = ALIBI ? l2_policy(true) : 0, pol_q = ALIBI ? l2_policy(false) : 0;
      uint32_t gk = 0;   // K tiles issued (ring index)
      uint32_t n_q = 0;  // items whose Q was loaded
      bool ok = true;
      for (int k = 0; ok && k < n_rounds; ++k) {
        const int w = snake_item(k, n_items);
        if (w < 0) continue;
        const WorkItem it = work_item<C::BM, C::BN>(p, w);
        if (!it.live || it.u1 <= it.u0) continue;
#pragma unroll
        for (int X = 0; X < C::NQT; ++X) {
          // Q_X of the previous item is in use until tile X's last S has run
          if (n_q > 0 && !mbar_wait(&q_empty[X], (n_q - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_q[X], C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_walk<ALIBI>(sQ + X * C::Q_BYTES + c * C::CHUNK, &tm_q, &bar_q[X], c * 64,
                                    item_head<C::BM>(p, it, X), it.s.q_row0 + item_row0<C::BM>(p, it, X), pol_q);
        }
        if (!ok) break;
        ++n_q;
        const int hkv = it.h / p.group;
        // ALiBi walks each item's tiles last to first: bring the next item's Q and first K tiles
        // into L2 now (measured 2.7 % faster there).  For forward walks the prefetch changed
        // nothing on llama7b_causal and cost 1 % on gqa_window (its bookkeeping delays the next
        // item's first K load), and with RoPE it measured slower, so only the ALiBi walk takes it.
        for (int k2 = k + 1; ALIBI && !ROPE && k2 < n_rounds; ++k2) {
          const int w2 = snake_item(k2, n_items);
          if (w2 < 0) continue;
          const WorkItem nx = work_item<C::BM, C::BN>(p, w2);
          if (!nx.live || nx.u1 <= nx.u0) continue;
#pragma unroll
          for (int X = 0; X < C::NQT; ++X)
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_prefetch_l2_3d(&tm_q, c * 64, item_head<C::BM>(p, nx, X), nx.s.q_row0 + item_row0<C::BM>(p, nx, X));
          for (int j = 0; j < C::KST && j < nx.u1 - nx.u0; ++j) {
            const int t2 = rev ? nx.u1 - 1 - j : nx.u0 + j;
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_prefetch_l2_3d(&tm_k, c * 64, nx.h / p.group, nx.s.k_row0 + t2 * C::BN);
          }
          break;
        }
        for (int t = rev ? it.u1 - 1 : it.u0; rev ? t >= it.u0 : t < it.u1; t += rev ? -1 : 1, ++gk) {
          const uint32_t st = gk % C::KST;
          if (gk >= (uint32_t)C::KST && !mbar_wait(&k_empty[st], ((gk / C::KST) + 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
          uint8_t* dst = sK + st * C::KV_BYTES;
          const int row = it.s.k_row0 + t * C::BN;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_walk<ALIBI>(dst + c * C::CHUNK, &tm_k, &k_full[st], c * 64, hkv, row, pol_kv);
        }
      }
      // drain: every issued load has landed before the CTA may exit
      if (n_q > 0) {
        mbar_wait_drain(&bar_q[0], (n_q - 1) & 1);
        mbar_wait_drain(&bar_q[1], (n_q - 1) & 1);
      }
      for (uint32_t st = 0; st < (uint32_t)C::KST && st < gk; ++st) {
        const uint32_t last = st + ((gk - 1 - st) / C::KST) * C::KST;
        mbar_wait_drain(&k_full[st], (last / C::KST) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ V producer
    setmaxnreg_dec<REGS_P>();
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_kv = ALIBI ? l2_policy(true) : 0;
      uint32_t gv = 0;  // V tiles issued (ring index)
      bool ok = true;
      for (int k = 0; ok && k < n_rounds; ++k) {
        const int w = snake_item(k, n_items);
        if (w < 0) continue;
        const WorkItem it = work_item<C::BM, C::BN>(p, w);
        if (!it.live || it.u1 <= it.u0) continue;
        const int hkv = it.h / p.group;
        for (int t = rev ? it.u1 - 1 : it.u0; rev ? t >= it.u0 : t < it.u1; t += rev ? -1 : 1, ++gv) {
          const uint32_t st = gv % C::VST;
          if (gv >= (uint32_t)C::VST && !mbar_wait(&v_empty[st], ((gv / C::VST) + 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          if (p.v_load_cap > 0 && gv >= (uint32_t)p.v_load_cap) {  // abort self-test: V stops coming
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
          uint8_t* dst = sV + st * C::KV_BYTES;
          const int row = it.s.k_row0 + t * C::BN;
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_walk<ALIBI>(dst + c * C::CHUNK, &tm_v, &v_full[st], c * 64, hkv, row, pol_kv);
        }
      }
      for (uint32_t st = 0; st < (uint32_t)C::VST && st < gv; ++st) {
        const uint32_t last = st + ((gv - 1 - st) / C::VST) * C::VST;
        mbar_wait_drain(&v_full[st], (last / C::VST) & 1);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged; one elected lane issues each instruction.
    setmaxnreg_dec<REGS_P>();
    const uint32_t leader = elect_one_sync() ? 1u : 0u;
    // Descriptors are built once; per MMA only the start-address field (bits 0..13, in 16-byte
    // units) moves, by an offset that is a compile-time constant after unrolling.
    const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(sV), C::CHUNK, 1024);
    // S_X = Q_X K^T with K from ring slot g % KST
    auto issue_s = [&](int X, uint32_t g) {
      const uint64_t kd = k_desc + (uint64_t)(((g % C::KST) * C::KV_BYTES) >> 4);
      const uint64_t qd = q_desc + (uint64_t)((X * C::Q_BYTES) >> 4);
      const uint32_t d_cols = tmem + C::COL_S + 128u * X;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)((((kk >> 2) * C::CHUNK) + (kk & 3) * 32) >> 4);
        umma_ss_by(leader, d_cols, qd + off, kd + off, C::IDESC_S, kk > 0 ? 1u : 0u);
      }
      umma_commit_by(leader, &s_full[X]);
    };
    // O_X (+)= P_X V with V from ring slot g % VST, P_X read from TMEM where the softmax left it.
    // The first P V of an item overwrites O_X: the softmax warps read the previous item's O_X
    // before they handed over P for this item's first tile, which this issue waited for.
    auto issue_pv = [&](int X, int t, uint32_t g, const QTileRange& r) {
      const uint64_t vd = v_desc + (uint64_t)(((g % C::VST) * C::KV_BYTES) >> 4);
      const uint32_t p_cols = tmem + C::COL_S + 128u * X;
      const uint32_t d_cols = tmem + C::COL_O + (uint32_t)D * X;
      const uint32_t acc0 = (rev ? t < r.t1 - 1 : t > r.t0) ? 1u : 0u;  // the walk's first P V overwrites O_X
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        umma_ts_by(leader, d_cols, p_cols + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4), C::IDESC_O,
                   kk > 0 ? 1u : acc0);
      if (t == (rev ? r.t0 : r.t1 - 1)) umma_commit_by(leader, &o_final[X]);
    };
    uint32_t gk = 0, gv = 0;              // K / V tiles consumed (ring indices)
    uint32_t n_q = 0;                     // items (bar_q[X] phase)
    uint32_t n_p[2] = {0, 0};             // P handoffs of tile X so far
    uint32_t n_r[2] = {0, 0};             // items with tile X active (q_ready phase)
    bool ok = true;
    for (int k = 0; ok && k < n_rounds; ++k) {
      const int w = snake_item(k, n_items);
      if (w < 0) continue;
      const WorkItem it = work_item<C::BM, C::BN>(p, w);
      if (!it.live || it.u1 <= it.u0) continue;
      const bool act_a = it.ra.t1 > it.ra.t0, act_b = it.rb.t1 > it.rb.t0;
      ok = mbar_wait(&k_full[gk % C::KST], (gk / C::KST) & 1, abort_flag, p.err);
      const uint32_t qph = n_q & 1;
      ++n_q;
      // Tile A's first S as soon as Q_A (and its rotation) is there, then tile B's.  Tile X's Q
      // buffer is free once its last S of the item has run; an inactive tile's once its load of
      // this item has landed (an earlier release would let the next load overlap this one).
#pragma unroll
      for (int X = 0; X < C::NQT; ++X) {
        const bool act = X ? act_b : act_a;
        const QTileRange& rx = X ? it.rb : it.ra;
        ok = ok && mbar_wait(&bar_q[X], qph, abort_flag, p.err);
        if (ROPE && act) ok = ok && mbar_wait(&q_ready[X], n_r[X] & 1, abort_flag, p.err);
        if (ROPE && act) ++n_r[X];
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (!act) {
          umma_commit_by(leader, &q_empty[X]);
        } else if (rev ? rx.t1 == it.u1 : rx.t0 == it.u0) {
          issue_s(X, gk);
          if (rx.t1 - rx.t0 == 1) umma_commit_by(leader, &q_empty[X]);
        }
      }
      if (!ok) break;
      umma_commit_by(leader, &k_empty[gk % C::KST]);
      for (int t = rev ? it.u1 - 1 : it.u0; ok && (rev ? t >= it.u0 : t < it.u1); t += rev ? -1 : 1) {
        const int j = rev ? it.u1 - 1 - t : t - it.u0;  // position of tile t in the walk
        const int tn = rev ? t - 1 : t + 1;             // the next tile of the walk
        const uint32_t gki = gk + (uint32_t)j, gvi = gv + (uint32_t)j;
        const bool nxt = rev ? tn >= it.u0 : tn < it.u1;
        // This step's operands first: V(t) for its P V and K(t+1) for the next S.  They have
        // normally landed long before; waiting for them here, while the softmax still works on
        // P(t), keeps both waits off the path from P(t) to the tensor core.
        const bool pv_a = t >= it.ra.t0 && t < it.ra.t1, pv_b = t >= it.rb.t0 && t < it.rb.t1;
        const bool s_a = nxt && tn >= it.ra.t0 && tn < it.ra.t1, s_b = nxt && tn >= it.rb.t0 && tn < it.rb.t1;
        // Both are normally complete: probe the two together (their shared-memory round trips
        // overlap; one after the other they cost ~150-280 cycles each with the tensor core idle),
        // and wait for them one by one only if either is not.
        if (!(nxt && mbar_test2(&v_full[gvi % C::VST], (gvi / C::VST) & 1, &k_full[(gki + 1) % C::KST],
                                ((gki + 1) / C::KST) & 1))) {
          if (pv_a || pv_b)
            ok = __all_sync(0xffffffffu, mbar_wait(&v_full[gvi % C::VST], (gvi / C::VST) & 1, abort_flag, p.err));
          if (ok && (s_a || s_b))
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&k_full[(gki + 1) % C::KST], ((gki + 1) / C::KST) & 1, abort_flag, p.err));
        }
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int X = 0; X < C::NQT; ++X) {
          if (X ? pv_b : pv_a) {
            __syncwarp();
            named_bar_sync(1 + X, kNamedBarThreads);  // P_X(t) from the tile's four softmax warps
            ++n_p[X];
            tc_fence_after();
            issue_pv(X, t, gvi, X ? it.rb : it.ra);
          }
          if (X ? s_b : s_a) {
            issue_s(X, gki + 1);
            const QTileRange& rx = X ? it.rb : it.ra;
            if (rev ? tn == rx.t0 : tn == rx.t1 - 1) umma_commit_by(leader, &q_empty[X]);  // tile X's last S
          }
        }
        if (!ok) break;
        umma_commit_by(leader, &v_empty[gvi % C::VST]);
        if (nxt) umma_commit_by(leader, &k_empty[(gki + 1) % C::KST]);
      }
      gk += (uint32_t)(it.u1 - it.u0);
      gv += (uint32_t)(it.u1 - it.u0);
    }
    if (!ok) {  // aborted: complete the P handoffs the softmax warps still make (see handoffs_total)
      const uint32_t ta = handoffs_total<C::BM, C::BN>(p, 0, n_rounds, n_items);
      const uint32_t tb = handoffs_total<C::BM, C::BN>(p, 1, n_rounds, n_items);
      for (; n_p[0] < ta; ++n_p[0]) named_bar_sync(1, kNamedBarThreads);
      for (; n_p[1] < tb; ++n_p[1]) named_bar_sync(2, kNamedBarThreads);
    }
    umma_commit_by(leader, mma_done);  // every MMA issued above has completed once this fires
    mbar_wait_drain(mma_done, 0);
    __syncwarp();
  } else {
    setmaxnreg_dec<REGS_P>();  // warp 11: idle, its registers go to the softmax warps
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool ALIBI, bool ROPE, bool PADK>
static cudaError_t launch_prefill_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                    const PrefillParams& p, int max_rows, int sm_count, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  // The shared-memory opt-in is a per-device function attribute: set it once per device.  The
  // register split (setmaxnreg) must fit in the registers the block is launched with: a split
  // above them would make the softmax warps wait for registers forever, so a build whose launch
  // register count came out lower than the split needs is refused here instead of launched.
  static int attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_prefill_kernel<D, ALIBI, ROPE, PADK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, fa_prefill_kernel<D, ALIBI, ROPE, PADK>);
    if (e != cudaSuccess) return e;
    if ((long long)fa.numRegs * C::THREADS < 2LL * 128 * C::REGS_SOFTMAX + 128LL * C::REGS_PRODUCER)
      return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  // Persistent (one CTA per SM walks its share of the items) when every sequence has the same
  // lengths, so that the static order balances; with per-sequence lengths the item costs are
  // unknown here, and one CTA per item lets the hardware scheduler balance them.
  PrefillParams q = p;
  // an even number of query heads per KV head: pair heads (same rows, same K/V), else row tiles
  q.pair_heads = (p.group % 2 == 0) ? 1 : 0;
  const int rows_per_item = q.pair_heads ? C::BM : C::NQT * C::BM;
  q.n_qblk = (max_rows + rows_per_item - 1) / rows_per_item;
  const long long n_items = (long long)(q.pair_heads ? q.Hq / 2 : q.Hq) * q.B * q.n_qblk;
  if (n_items <= 0) return cudaSuccess;
  if (n_items >= (1LL << 31)) return cudaErrorInvalidConfiguration;
  const bool uniform = !p.cu_q && !p.seqlens_q && !p.seqlens_k;
  const unsigned grid = (unsigned)(uniform && n_items > sm_count ? sm_count : n_items);
  fa_prefill_kernel<D, ALIBI, ROPE, PADK><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, to, q);
  return cudaGetLastError();
}

template <int D, bool ALIBI, bool ROPE>
static cudaError_t launch_prefill_p(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                    const PrefillParams& p, int max_rows, int sm, cudaStream_t stream) {
  const bool padk = p.seqlens_k != nullptr && p.cu_q == nullptr;
  return padk ? launch_prefill_d<D, ALIBI, ROPE, true>(tq, tk, tv, to, p, max_rows, sm, stream)
              : launch_prefill_d<D, ALIBI, ROPE, false>(tq, tk, tv, to, p, max_rows, sm, stream);
}

template <int D>
static cudaError_t launch_prefill_dd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                                     const PrefillParams& p, int max_rows, int sm, cudaStream_t stream) {
  const bool alibi = p.alibi != nullptr, rope = p.rope_cos != nullptr;
  if (alibi) return rope ? launch_prefill_p<D, true, true>(tq, tk, tv, to, p, max_rows, sm, stream)
                         : launch_prefill_p<D, true, false>(tq, tk, tv, to, p, max_rows, sm, stream);
  return rope ? launch_prefill_p<D, false, true>(tq, tk, tv, to, p, max_rows, sm, stream)
              : launch_prefill_p<D, false, false>(tq, tk, tv, to, p, max_rows, sm, stream);
}

cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                           const PrefillParams& p, int max_rows, int sm_count, cudaStream_t stream) {
  return d == 64 ? launch_prefill_dd<64>(tq, tk, tv, to, p, max_rows, sm_count, stream)
                 : launch_prefill_dd<128>(tq, tk, tv, to, p, max_rows, sm_count, stream);
}

int prefill_box_rows() { return PrefillCfg<128>::BM; }

}  // namespace fa
