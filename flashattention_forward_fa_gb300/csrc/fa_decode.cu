// Incremental decode over a KV cache, split along the key axis, for sm_103a.
//
// What it computes: for every sequence b and query head h, the attention of the
// new token over the cached keys 0 .. len_b-1 (the incremental mode of the
// agent.csdn.net BERT walkthrough, 结尾: the new token attends to all cached K/V
// and the old K/V are not recomputed, so cost is linear in the cache length).
// With nq > 1 new tokens per sequence (speculative drafts, a chunk of a prompt)
// they are the last nq cache slots: token t sits at position len_b - nq + t and
// sees the keys up to its own position (bottom-right causal alignment).
// The key range is cut into chunks; each chunk yields a partial (O_s, lse_s)
// and a combine kernel merges them with the log-sum-exp identity
//     LSE = log sum_s exp(lse_s),   O = sum_s exp(lse_s - LSE) O_s,
// which is the running-max/running-sum softmax of the hwcomputing.csdn.net page,
// §2.2 "数值稳定性优化" applied across chunks instead of across tiles.
//
// How: the kernel is bound by HBM bandwidth (each cached byte is read once per
// KV head group), so the design is about bytes in flight, not MMA width:
//   one CTA = one (sequence, KV head, chunk); warp 4 streams 64-key K and V
//   tiles through a TMA + mbarrier ring; warps 0-3 each take 16 keys of a tile
//   and run Q K^T and P V on the tensor cores with mma.sync m16n8k16 (the
//   nq x G (token, query head) rows of the group are the M rows, 16 per CTA;
//   a few rows are below the tcgen05 minimum M of 64), keeping a private running
//   max/sum; the four warps merge in shared memory at the end of the chunk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

template <int D>
struct DecodeCfg {
  static constexpr int BN = 64;                   // keys per pipeline tile
  static constexpr int ST = 3;                    // ring stages
  static constexpr int SLAB = BN * 128;           // one 64-column swizzled slab (bytes)
  static constexpr int TILE = BN * D * 2;         // K or V tile (bytes)
  static constexpr int STAGE = 2 * TILE;          // K + V
  static constexpr int OFF_BAR = ST * STAGE;
  static constexpr int MERGE_BYTES = 4 * 16 * D * 4 + 3 * 4 * 16 * 4;  // per-warp O, m, l, lr
  static_assert(MERGE_BYTES <= ST * STAGE, "merge area reuses the ring");
  static constexpr int SMEM_BYTES = OFF_BAR + 2 * ST * 8 + 16 + 1024;
  static constexpr int THREADS = 160;             // 4 compute warps + 1 producer warp
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk (key, 8-column group d8) in a TMA SWIZZLE_128B tile
// stored as [D/64 slabs][BN keys][64 columns].
template <int D>
__device__ __forceinline__ uint32_t sw_off(int key, int d8) {
  return (uint32_t)((d8 >> 3) * DecodeCfg<D>::SLAB + key * 128 + (((d8 & 7) ^ (key & 7)) << 4));
}

// Key range of sequence b: [lo, len) holds every key one of its nq queries may see (lo is the
// window start of the first new token); the chunks cover [base, len) with base = lo for a
// contiguous cache and lo rounded down to a multiple of 64 for a paged one (so that no 64-key
// tile straddles two pages; keys below a row's own window start are masked).
struct DecodeRange {
  int len, lo, base;
};
__device__ __forceinline__ DecodeRange decode_range(const DecodeParams& p, int b, bool paged) {
  DecodeRange r;
  const int cap = paged ? p.max_blocks * p.page_size : p.Ncap;
  r.len = min(max(p.seqlens_k[b], 0), cap);
  r.lo = p.window > 0 ? max(0, r.len - p.nq + 1 - p.window) : 0;
  r.base = paged ? (r.lo & ~63) : r.lo;
  return r;
}

// Physical row of the first key of a 64-key tile.  A block-table entry outside [0, num_pages)
// is recorded in the device status word and replaced by page 0, so a bad table cannot fault.
__device__ __forceinline__ int paged_row(const DecodeParams& p, int b, int key) {
  const int blk = key / p.page_size;
  int page = (blk < p.max_blocks) ? p.block_table[(size_t)b * p.max_blocks + blk] : -1;
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.err, kDevErrBounds);
    page = 0;
  }
  return page * p.page_size + (key - blk * p.page_size);
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int D, bool PAGED, bool ALIBI>
__global__ void __launch_bounds__(DecodeCfg<D>::THREADS)
    fa_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecodeParams p) {
  using C = DecodeCfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int n_rows = p.nq * p.group;                 // (token, head) rows of one KV head
  const int n_rb = (n_rows + 15) / 16;
  const int hkv = blockIdx.y / n_rb;
  const int rb = blockIdx.y % n_rb;
  const int b = blockIdx.z;
  const DecodeRange kr = decode_range(p, b, PAGED);
  const int len = kr.len;
  const int start = kr.base + split * p.chunk;
  const int end = min(start + p.chunk, len);
  if (start >= end) return;  // chunk past the end of this sequence's keys
  const int n_tiles = (end - start + C::BN - 1) / C::BN;
  const int row0 = rb * 16;                          // first row of this block: row r is token r / group,
  const int nrows = min(16, n_rows - row0);          // query head hkv * group + r % group

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* empty = full + C::ST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_BAR + 2 * C::ST * 8);

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int t = 0;
      // paged: the next tile's page is looked up one tile ahead, hiding the table load
      int row_next = PAGED ? paged_row(p, b, start) : 0;
      for (; t < n_tiles; ++t) {
        const int st = t % C::ST;
        const int row = PAGED ? row_next : b * p.Ncap + start + t * C::BN;
        if (PAGED && t + 1 < n_tiles) row_next = paged_row(p, b, start + (t + 1) * C::BN);
        if (t >= C::ST && !mbar_wait(&empty[st], ((t / C::ST) + 1) & 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&full[st], C::STAGE);
        uint8_t* dst = sm + st * C::STAGE;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(dst + c * C::SLAB, &tm_k, &full[st], c * 64, hkv, row);
          tma_load_3d(dst + C::TILE + c * C::SLAB, &tm_v, &full[st], c * 64, hkv, row);
        }
      }
      for (int st = 0; st < C::ST && st < t; ++st) {  // drain: all issued loads have landed
        const int last = st + ((t - 1 - st) / C::ST) * C::ST;
        mbar_wait_drain(&full[st], (last / C::ST) & 1);
      }
    }
    return;  // the producer takes no part in the merge below
  }

  // -------------------------------------------------------------- compute warps
  const int g = lane >> 2, tq = lane & 3;
  const bool v0 = g < nrows, v1 = g + 8 < nrows;  // this lane's two rows exist
  const int ra = row0 + (v0 ? g : 0), rb8 = row0 + (v1 ? g + 8 : 0);
  const int ta = ra / p.group, tb = rb8 / p.group;                 // their tokens
  const int hqa = hkv * p.group + ra % p.group, hqb = hkv * p.group + rb8 % p.group;
  const size_t qia = ((size_t)b * p.nq + ta) * p.Hq + hqa, qib = ((size_t)b * p.nq + tb) * p.Hq + hqb;
  // each row's visible keys [klo, khi) cut to this chunk: position pos = len - nq + token
  const int posa = len - p.nq + ta, posb = len - p.nq + tb;
  const int kloa = p.window > 0 ? max(0, posa - p.window + 1) : 0;
  const int klob = p.window > 0 ? max(0, posb - p.window + 1) : 0;
  const int khia = min(posa + 1, end), khib = min(posb + 1, end);
  // Q fragments (zero past nrows)
  uint32_t qa[D / 16][4];
  {
    const uint32_t* qrow_g =
        reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + qia * D);
    const uint32_t* qrow_g8 =
        reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + qib * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = v0 ? qrow_g[kk * 8 + tq] : 0u;
      qa[kk][1] = v1 ? qrow_g8[kk * 8 + tq] : 0u;
      qa[kk][2] = v0 ? qrow_g[kk * 8 + 4 + tq] : 0u;
      qa[kk][3] = v1 ? qrow_g8[kk * 8 + 4 + tq] : 0u;
    }
  }
  float oacc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  // With ALiBi the scale is applied together with the bias -m_h (pos - key), pos the row's token
  // position, and everything after works on scaled scores (xs = 1).
  const float xs = ALIBI ? 1.0f : p.scale_log2;
  const float slope_g = (ALIBI && v0) ? p.alibi[hqa] * 1.4426950408889634f : 0.f;
  const float slope_g8 = (ALIBI && v1) ? p.alibi[hqb] * 1.4426950408889634f : 0.f;
  float lr0 = 0.f, lr1 = 0.f;  // sums of the bf16-rounded weights P V actually uses (normalise O)
  const uint32_t sbase = smem_u32(sm);
  bool ok = true;

  for (int t = 0; t < n_tiles; ++t) {
    const int st = t % C::ST;
    ok = mbar_wait(&full[st], (t / C::ST) & 1, abort_flag, p.err);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const int kb = warp * 16;                              // this warp's keys within the tile
    const int kw0 = start + t * C::BN + kb;                // its first key
    const int nvalid = min(16, end - kw0);
    const uint32_t kaddr = sbase + st * C::STAGE;
    const uint32_t vaddr = kaddr + C::TILE;
    if (nvalid > 0) {
      if (nvalid < 16) {
        // cache slots past the end may hold anything; zero their V rows so 0 * V stays 0
        uint8_t* vt = sm + st * C::STAGE + C::TILE;
        for (int idx = lane; idx < (16 - nvalid) * (D / 8); idx += 32) {
          const int key = kb + nvalid + idx / (D / 8);
          *reinterpret_cast<uint4*>(vt + sw_off<D>(key, idx % (D / 8))) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();  // order these generic writes before the next TMA fill of this stage
        __syncwarp();
      }
      // S = Q K^T for 16 keys: two n8 tiles
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kaddr + sw_off<D>(kb + (mi >> 1) * 8 + r8, 2 * kk + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_bf16(sc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
      }
      // mask keys outside each row's [klo, khi) (this also drops keys past the chunk end)
      {
        const int la = kloa - kw0 - 2 * tq, ha = khia - kw0 - 2 * tq;
        const int lb = klob - kw0 - 2 * tq, hb = khib - kw0 - 2 * tq;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kr = n * 8 + (e & 1);
            if (e < 2 ? (kr < la || kr >= ha) : (kr < lb || kr >= hb)) sc[n][e] = -INFINITY;
          }
      }
      if (ALIBI) {
        const float da = (float)(posa - kw0 - 2 * tq), db = (float)(posb - kw0 - 2 * tq);  // pos - key, n=e=0
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sc[n][e] = fmaf(sc[n][e], p.scale_log2,
                            e < 2 ? -slope_g * (da - (float)(n * 8 + (e & 1)))
                                  : -slope_g8 * (db - (float)(n * 8 + (e & 1))));
      }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0 * xs), mn1 = fmaxf(m1, mx1 * xs);
      if (mn0 > m0 + 8.0f) {  // lazy rescale: the exponent base moves only on large jumps
        const float a = ex2_approx(m0 - mn0);
        l0 *= a;
        lr0 *= a;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) oacc[n][0] *= a, oacc[n][1] *= a;
        m0 = mn0;
      }
      if (mn1 > m1 + 8.0f) {
        const float a = ex2_approx(m1 - mn1);
        l1 *= a;
        lr1 *= a;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) oacc[n][2] *= a, oacc[n][3] *= a;
        m1 = mn1;
      }
      const float mu0 = (m0 == -INFINITY) ? 0.f : m0, mu1 = (m1 == -INFINITY) ? 0.f : m1;
      float pe[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        pe[n][0] = ex2_approx(fmaf(sc[n][0], xs, -mu0));
        pe[n][1] = ex2_approx(fmaf(sc[n][1], xs, -mu0));
        pe[n][2] = ex2_approx(fmaf(sc[n][2], xs, -mu1));
        pe[n][3] = ex2_approx(fmaf(sc[n][3], xs, -mu1));
        l0 += pe[n][0] + pe[n][1];
        l1 += pe[n][2] + pe[n][3];
      }
      const uint32_t pa0 = pack_bf16x2(pe[0][0], pe[0][1]);
      const uint32_t pa1 = pack_bf16x2(pe[0][2], pe[0][3]);
      const uint32_t pa2 = pack_bf16x2(pe[1][0], pe[1][1]);
      const uint32_t pa3 = pack_bf16x2(pe[1][2], pe[1][3]);
      lr0 += (__uint_as_float(pa0 << 16) + __uint_as_float(pa0 & 0xffff0000u)) +
             (__uint_as_float(pa2 << 16) + __uint_as_float(pa2 & 0xffff0000u));
      lr1 += (__uint_as_float(pa1 << 16) + __uint_as_float(pa1 & 0xffff0000u)) +
             (__uint_as_float(pa3 << 16) + __uint_as_float(pa3 & 0xffff0000u));
      // O += P V for 16 keys
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vaddr + sw_off<D>(kb + (mi & 1) * 8 + r8, 2 * j + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(oacc[2 * j], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16(oacc[2 * j + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---------------------------------------------------------------- merge the four warps
  named_bar_sync(1, 128);  // every compute warp is done with the ring
  float* mo = reinterpret_cast<float*>(sm);                  // [4][16][D]
  float* mm = mo + 4 * 16 * D;                               // [4][16]
  float* ml = mm + 4 * 16;                                   // [4][16]
  float* mr = ml + 4 * 16;                                   // [4][16]
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  lr0 += __shfl_xor_sync(0xffffffffu, lr0, 1);
  lr0 += __shfl_xor_sync(0xffffffffu, lr0, 2);
  lr1 += __shfl_xor_sync(0xffffffffu, lr1, 1);
  lr1 += __shfl_xor_sync(0xffffffffu, lr1, 2);
  if (ok) {
    if (tq == 0) {
      mm[warp * 16 + g] = m0;
      mm[warp * 16 + g + 8] = m1;
      ml[warp * 16 + g] = l0;
      ml[warp * 16 + g + 8] = l1;
      mr[warp * 16 + g] = lr0;
      mr[warp * 16 + g + 8] = lr1;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      float* r0p = mo + (warp * 16 + g) * D + n * 8 + 2 * tq;
      float* r1p = mo + (warp * 16 + g + 8) * D + n * 8 + 2 * tq;
      r0p[0] = oacc[n][0];
      r0p[1] = oacc[n][1];
      r1p[0] = oacc[n][2];
      r1p[1] = oacc[n][3];
    }
  }
  named_bar_sync(1, 128);
  if (*abort_flag) return;  // a wait timed out somewhere: leave the outputs unwritten
  for (int idx = tid; idx < nrows * D; idx += 128) {
    const int r = idx / D, d = idx % D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mstar = fmaxf(mstar, mm[w * 16 + r]);
    float lsum = 0.f, rsum = 0.f, osum = 0.f;
    if (mstar != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = ex2_approx(mm[w * 16 + r] - mstar);
        lsum += ml[w * 16 + r] * f;
        rsum += mr[w * 16 + r] * f;
        osum += mo[(w * 16 + r) * D + d] * f;
      }
    }
    const int row = row0 + r;
    const size_t qi = ((size_t)b * p.nq + row / p.group) * p.Hq + hkv * p.group + row % p.group;
    const size_t prow = qi * p.max_splits + split;
    p.o_part[prow * D + d] = rsum > 0.f ? osum / rsum : 0.f;
    if (d == 0) p.lse_part[prow] = lsum > 0.f ? (mstar + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

// One warp per (sequence, new token, query head): merge the chunk partials.  O is
// [B, nq, Hq, d]; LSE is [B, Hq, nq].
// Launched as a programmatic dependent of the split kernel: it may start while the split kernel
// drains and waits here until the split kernel's partials are complete and visible.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const DecodeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.B * p.nq * p.Hq) return;
  const int bt = warp_global / p.Hq, hq = warp_global % p.Hq;
  const int b = bt / p.nq, t = bt % p.nq;
  const DecodeRange kr = decode_range(p, b, p.page_size > 0);
  const int pos = kr.len - p.nq + t;  // this token's position; it sees keys (pos - window, pos]
  const int klo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
  const int nkeys = pos + 1 - klo;
  const int nspan = kr.len - kr.base;  // keys the chunks cover
  constexpr int PER = D / 32;  // output columns per lane
  __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((size_t)bt * p.Hq + hq) * D + lane * PER;
  float* lse_out = p.lse ? p.lse + ((size_t)b * p.Hq + hq) * p.nq + t : nullptr;
  if (nkeys <= 0) {
#pragma unroll
    for (int j = 0; j < PER; ++j) orow[j] = __float2bfloat16(0.f);
    if (lse_out && lane == 0) *lse_out = -INFINITY;
    return;
  }
  const int need = (nspan + p.chunk - 1) / p.chunk;  // chunks this sequence's keys fill
  // A host length that understated the device length planned too few splits: the keys past
  // max_splits chunks were not read.  Report it; never read past the workspace.
  if (need > p.max_splits && lane == 0) atomicOr(p.err, kDevErrBounds);
  const int ns = min(need, p.max_splits);
  const size_t prow0 = ((size_t)bt * p.Hq + hq) * p.max_splits;
  constexpr float LOG2E = 1.4426950408889634f;
  float mx = -INFINITY;
  for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, p.lse_part[prow0 + s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  float tot = 0.f;
#pragma unroll 4
  for (int s = 0; s < ns; ++s) {  // unrolled: several partials' loads in flight
    const float w = ex2_approx((p.lse_part[prow0 + s] - mx) * LOG2E);
    tot += w;
    const float* op = p.o_part + (prow0 + s) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(op);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(op);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
    }
  }
  const float inv = 1.0f / tot;
  if constexpr (PER == 4) {
    uint2 packed = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    *reinterpret_cast<uint2*>(orow) = packed;
  } else {
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lse_out && lane == 0) *lse_out = mx + __logf(tot);
}

template <int D, bool PAGED, bool ALIBI>
static cudaError_t launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                                   cudaStream_t stream) {
  using C = DecodeCfg<D>;
  // The shared-memory opt-in is a per-device function attribute: set it once per device.
  static int attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_decode_split_kernel<D, PAGED, ALIBI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = 1;
  }
  const int n_rb = (p.nq * p.group + 15) / 16;
  dim3 grid(p.max_splits, p.Hkv * n_rb, p.B);
  fa_decode_split_kernel<D, PAGED, ALIBI><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = p.B * p.nq * p.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the launch with the split's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_decode_combine_kernel<D>, p);
}

template <int D>
static cudaError_t launch_decode_dd(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                                    cudaStream_t stream) {
  const bool paged = p.page_size > 0, alibi = p.alibi != nullptr;
  if (paged) return alibi ? launch_decode_d<D, true, true>(tk, tv, p, stream)
                          : launch_decode_d<D, true, false>(tk, tv, p, stream);
  return alibi ? launch_decode_d<D, false, true>(tk, tv, p, stream) : launch_decode_d<D, false, false>(tk, tv, p, stream);
}

cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                          cudaStream_t stream) {
  return d == 64 ? launch_decode_dd<64>(tk, tv, p, stream) : launch_decode_dd<128>(tk, tv, p, stream);
}

int decode_block_n() { return DecodeCfg<128>::BN; }

}  // namespace fa
