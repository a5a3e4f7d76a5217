// Fused attention forward (prefill / encoder) for sm_103a.
//
// What it computes: O = softmax(Q K^T * scale + mask) V and the row LSE, with the
// running-max / running-sum softmax, so scores never leave the SM — the fused
// tiled evaluation of the jsqmd page "CANN Transformer算子库ops-transformer深度实践",
// §二 "FlashAttention的融合计算思想" (Q split by rows, K/V by columns, every Q block
// sweeps all K/V blocks on chip) with the max-subtracted fp32 softmax of the
// hwcomputing.csdn.net page, §2.2 "数值稳定性优化" (its "two-stage max propagation"
// realised as a running max whose changes rescale the accumulator).
//
// How (GB300-first; the pages' Cube/Vector double buffer is only prior art):
//   one CTA = one 128-row Q tile of one (sequence, query head); 7 warps:
//     warps 0-3  softmax: thread r owns score row r (TMEM lane r)
//     warp  4    TMA producer for Q (once) and the K ring
//     warp  5    TMA producer for the V ring
//     warp  6    TMEM allocator and tcgen05.mma issuer
//   S_t = Q K_t^T runs on the tensor cores into one of two TMEM score buffers
//   while the softmax warps work on the other; P_t (bf16) is written back over
//   its own scores in TMEM and consumed straight from there by O += P_t V_t
//   (A operand in TMEM), O accumulating in TMEM in fp32.
//   The O rescale is lazy: the running max used for exponentiation only moves
//   when the tile max exceeds it by more than 2^8, so most tiles touch O never;
//   the final O / l uses the same max, so the result is exact.
//   Causal / window tiles that are fully masked are never loaded; only tiles
//   crossing a mask boundary (or the ragged tail) evaluate the mask.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;  // query rows per CTA
  static constexpr int BN = 128;  // keys per tile
  static constexpr int KST = (D == 128) ? 3 : 4;
  static constexpr int VST = (D == 128) ? 2 : 4;
  static constexpr int CHUNK_Q = BM * 128;  // bytes of one 64-column swizzled slab of a Q tile
  static constexpr int CHUNK_KV = BN * 128;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * KV_BYTES;
  // barriers: q, k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2], p_full[2], o_done,
  // o_final, mma_done
  static constexpr int NBAR = 1 + 2 * KST + 2 * VST + 2 + 2 + 1 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem slot (4 B) + abort flag (4 B)
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 224;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);  // Q, K both K-major
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 0, 1);   // P K-major (TMEM), V MN-major
};

struct SeqInfo {
  int q_row0, Lq, rows_out, k_row0, Lk;
  long long lse_row0;  // LSE index of row 0 of this (sequence, head)
};

__device__ __forceinline__ SeqInfo seq_info(const PrefillParams& p, int b, int h) {
  SeqInfo s;
  if (p.cu_q) {
    s.q_row0 = p.cu_q[b];
    s.Lq = p.cu_q[b + 1] - s.q_row0;
    s.k_row0 = p.cu_k[b];
    s.Lk = p.cu_k[b + 1] - s.k_row0;
    s.rows_out = s.Lq;
    const int total_q = p.cu_q[p.B];
    s.lse_row0 = (long long)h * total_q + s.q_row0;
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

__device__ __forceinline__ bool key_visible(int key, int pos, int Lk, int causal, int window) {
  bool ok = key < Lk;
  if (causal) {
    ok = ok && key <= pos;
    if (window > 0) ok = ok && key > pos - window;
  } else if (window > 0) {
    ok = ok && key > pos - window && key < pos + window;
  }
  return ok;
}

template <int D>
__device__ __forceinline__ void store_row_zero(const PrefillParams& p, const SeqInfo& s, int h, int i) {
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)(s.q_row0 + i) * p.Hq + h) * D;
  uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
  if (p.lse) p.lse[s.lse_row0 + i] = -INFINITY;
}

template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using C = PrefillCfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int b = blockIdx.z;
  const int qtile = (p.causal || p.window > 0) ? (int)(gridDim.y - 1 - blockIdx.y) : (int)blockIdx.y;
  const int q0 = qtile * C::BM;
  const SeqInfo s = seq_info(p, b, h);
  if (q0 >= s.rows_out) return;  // whole tile past the (padded) end
  const int hkv = h / p.group;

  // KV tile range [t_begin, t_begin + T) visible to the valid rows of this tile.
  const int rows_valid = max(0, min(C::BM, s.Lq - q0));
  const int pos_min = q0 + s.Lk - s.Lq;
  const int pos_max = q0 + rows_valid - 1 + s.Lk - s.Lq;
  int lo = 0, hi = s.Lk;
  if (p.causal) hi = min(hi, pos_max + 1);
  if (p.window > 0) {
    lo = max(lo, pos_min - p.window + 1);
    if (!p.causal) hi = min(hi, pos_max + p.window);
  }
  const int T = (rows_valid > 0 && hi > lo) ? ((hi + C::BN - 1) / C::BN - lo / C::BN) : 0;
  const int t_begin = lo / C::BN;

  if (T == 0) {  // no key visible to any row: O = 0, LSE = -inf (and zero padding rows)
    for (int r = tid; r < C::BM; r += blockDim.x)
      if (q0 + r < s.rows_out) store_row_zero<D>(p, s, h, q0 + r);
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* bar_q = bars;
  uint64_t* k_full = bar_q + 1;
  uint64_t* k_empty = k_full + C::KST;
  uint64_t* v_full = k_empty + C::KST;
  uint64_t* v_empty = v_full + C::VST;
  uint64_t* s_full = v_empty + C::VST;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;   // one completion per PV (phase gap to any waiter is at most one)
  uint64_t* o_final = o_done + 1;  // single completion: the last PV of this tile
  uint64_t* mma_done = o_final + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);

  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_q, 1);
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
      mbar_init(&p_full[i], 4);  // one arrival per softmax warp
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    mbar_init(mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 6) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ softmax warps
    const int r = tid;
    const int i = q0 + r;
    const int pos = i + s.Lk - s.Lq;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max used for exponentiation (log2 units)
    float l = 0.f;        // running sum of exp2(score*sl2 - m) in fp32 (gives the LSE)
    float lr = 0.f;       // running sum of the same weights rounded to bf16 (normalises O)
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int sb = t & 1;
      ok = mbar_wait(&s_full[sb], (t >> 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sc[C::BN];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        const uint32_t a = t_lane + (sb ? C::COL_S1 : C::COL_S0);
        tmem_ld32(a + 0, r0);
        tmem_ld32(a + 32, r1);
        tmem_ld32(a + 64, r2);
        tmem_ld32(a + 96, r3);
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
      }
      const int k0 = (t_begin + t) * C::BN;
      bool need_mask = (k0 + C::BN > s.Lk);
      if (p.causal) need_mask |= (k0 + C::BN - 1 > pos_min);
      if (p.window > 0) {
        need_mask |= (k0 < pos_max - p.window + 1);
        if (!p.causal) need_mask |= (k0 + C::BN - 1 > pos_min + p.window - 1);
      }
      if (need_mask) {
#pragma unroll
        for (int j = 0; j < C::BN; ++j)
          if (!key_visible(k0 + j, pos, s.Lk, p.causal, p.window)) sc[j] = -INFINITY;
      }
      float mx;
      {
        float t4[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t4[u] = sc[u];
#pragma unroll
        for (int j = 8; j < C::BN; j += 8)
#pragma unroll
          for (int u = 0; u < 8; ++u) t4[u] = fmaxf(t4[u], sc[j + u]);
        mx = fmaxf(fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3])), fmaxf(fmaxf(t4[4], t4[5]), fmaxf(t4[6], t4[7])));
      }
      mx *= sl2;
      const float m_new = fmaxf(m, mx);
      const bool need = m_new > m + 8.0f;  // -inf + 8 = -inf: the first finite max always moves m
      const float alpha = need ? ex2_approx(m - m_new) : 1.0f;
      const bool o_live = need && (t > 0) && (m != -INFINITY);  // O row holds data to rescale
      if (__any_sync(0xffffffffu, o_live)) {
        ok = mbar_wait(o_done, (t - 1) & 1, abort_flag, p.err);  // PV_{t-1} finished
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = o_live ? alpha : 1.0f;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld32(t_lane + C::COL_O + c, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
          tmem_st32(t_lane + C::COL_O + c, ov);
        }
      }
      if (need) {
        l *= alpha;
        lr *= alpha;
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // P V runs on bf16-rounded weights; normalising O by the sum of those same rounded
      // weights keeps O an exact convex combination of V rows (the bf16 rounding of P then
      // only perturbs the weights, never their total), while the LSE uses the fp32 sum.
      float rs0 = 0.f, rs1 = 0.f, rr0 = 0.f, rr1 = 0.f;
      uint32_t pk0[32], pk1[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float e0 = ex2_approx(fmaf(sc[2 * j], sl2, -m_use));
        const float e1 = ex2_approx(fmaf(sc[2 * j + 1], sl2, -m_use));
        rs0 += e0;
        rs1 += e1;
        pk0[j] = pack_bf16x2(e0, e1);
        rr0 += __uint_as_float(pk0[j] << 16);
        rr1 += __uint_as_float(pk0[j] & 0xffff0000u);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float e0 = ex2_approx(fmaf(sc[64 + 2 * j], sl2, -m_use));
        const float e1 = ex2_approx(fmaf(sc[64 + 2 * j + 1], sl2, -m_use));
        rs0 += e0;
        rs1 += e1;
        pk1[j] = pack_bf16x2(e0, e1);
        rr0 += __uint_as_float(pk1[j] << 16);
        rr1 += __uint_as_float(pk1[j] & 0xffff0000u);
      }
      l += rs0 + rs1;
      lr += rr0 + rr1;
      const uint32_t pa = t_lane + (sb ? C::COL_S1 : C::COL_S0);
      tmem_st32(pa + 0, pk0);
      tmem_st32(pa + 32, pk1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    if (ok) {
      // A fast warp can get here while PV_{T-2} is still pending, two phases behind o_done, so the
      // last PV signals its own single-phase barrier.
      ok = mbar_wait(o_final, 0, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const bool store = i < s.Lq;
      const float inv = lr > 0.f ? 1.0f / lr : 0.f;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)(s.q_row0 + i) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t ov[32];
        tmem_ld32(t_lane + C::COL_O + c, ov);
        tmem_ld_wait(ov);
        if (store) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack_bf16x2(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (store && p.lse) p.lse[s.lse_row0 + i] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (!store && i < s.rows_out) store_row_zero<D>(p, s, h, i);
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ Q + K producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * C::CHUNK_Q, &tm_q, bar_q, c * 64, h, s.q_row0 + q0);
      int t = 0;
      for (; t < T; ++t) {
        const int st = t % C::KST;
        if (t >= C::KST && !mbar_wait(&k_empty[st], ((t / C::KST) + 1) & 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
        uint8_t* dst = sK + st * C::KV_BYTES;
        const int row = s.k_row0 + (t_begin + t) * C::BN;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * C::CHUNK_KV, &tm_k, &k_full[st], c * 64, hkv, row);
      }
      // drain: every issued load has landed before the CTA may exit
      mbar_wait(bar_q, 0, abort_flag, nullptr);
      for (int st = 0; st < C::KST && st < t; ++st) {
        const int last = st + ((t - 1 - st) / C::KST) * C::KST;
        mbar_wait(&k_full[st], (last / C::KST) & 1, abort_flag, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      int t = 0;
      for (; t < T; ++t) {
        const int st = t % C::VST;
        if (t >= C::VST && !mbar_wait(&v_empty[st], ((t / C::VST) + 1) & 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
        uint8_t* dst = sV + st * C::KV_BYTES;
        const int row = s.k_row0 + (t_begin + t) * C::BN;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * C::CHUNK_KV, &tm_v, &v_full[st], c * 64, hkv, row);
      }
      for (int st = 0; st < C::VST && st < t; ++st) {
        const int last = st + ((t - 1 - st) / C::VST) * C::VST;
        mbar_wait(&v_full[st], (last / C::VST) & 1, abort_flag, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
      auto issue_pv = [&](int u, bool last) -> bool {
        const int vs = u % C::VST;
        if (!mbar_wait(&p_full[u & 1], (u >> 1) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(&v_full[vs], (u / C::VST) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t p_cols = tmem + ((u & 1) ? C::COL_S1 : C::COL_S0);
        const uint32_t vb = v_base + vs * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(vb + kk * 16 * 128, C::CHUNK_KV, 1024);
          umma_ts(tmem + C::COL_O, p_cols + kk * 8, bdesc, C::IDESC_O, (u > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&v_empty[vs]);
        umma_commit(o_done);
        if (last) umma_commit(o_final);
        return true;
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.err);
      for (int t = 0; ok && t < T; ++t) {
        const int ks = t % C::KST;
        if (!mbar_wait(&k_full[ks], (t / C::KST) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_cols = tmem + ((t & 1) ? C::COL_S1 : C::COL_S0);
        const uint32_t kb = k_base + ks * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_Q + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * C::CHUNK_KV + (kk & 3) * 32;
          const uint64_t adesc = sdesc_sw128(q_base + off, 16, 1024);
          const uint64_t bdesc = sdesc_sw128(kb + offk, 16, 1024);
          umma_ss(s_cols, adesc, bdesc, C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        umma_commit(&k_empty[ks]);
        umma_commit(&s_full[t & 1]);
        if (t >= 1) ok = issue_pv(t - 1, false);
      }
      if (ok) issue_pv(T - 1, true);
      umma_commit(mma_done);  // every MMA issued above has completed once this fires
      mbar_wait(mma_done, 0, abort_flag, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
static cudaError_t launch_prefill_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const PrefillParams& p, int n_qtiles, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(fa_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.Hq, n_qtiles, p.B);
  fa_prefill_kernel<D><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int n_qtiles, cudaStream_t stream) {
  if (d == 64) return launch_prefill_d<64>(tq, tk, tv, p, n_qtiles, stream);
  return launch_prefill_d<128>(tq, tk, tv, p, n_qtiles, stream);
}

int prefill_block_m() { return PrefillCfg<128>::BM; }

}  // namespace fa
