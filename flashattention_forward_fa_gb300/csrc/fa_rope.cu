// Rotary position embedding applied in place to a bf16 tensor [rows, heads, d].
//
// What it computes: the rotation of the jsqmd page "CANN Transformer算子库ops-transformer
// 深度实践", §三 "RoPE的设计动机与计算特点": for every row at position p and every pair of
// adjacent dimensions (2i, 2i+1), i < rotary_dim / 2,
//     (x, y) -> (x cos(p, i) - y sin(p, i),  x sin(p, i) + y cos(p, i)),
// with cos / sin read from caller-given lookup tables [table_rows, rotary_dim / 2]
// (the table approach of the hwcomputing.csdn.net page, §1.2).  The math runs in fp32
// and the result is rounded to bf16 (round to nearest even).
//
// How: an elementwise, HBM-bound pass in one of two forms.  Rows of at least 512 16-byte
// chunks (e.g. 32 heads x d 128): a CTA takes one row at a time (grid-stride over rows); each
// thread takes one chunk position (four pairs) in four heads of the row and loads all four
// before storing any, so it keeps 64 bytes in flight and reads one float4 of each table per row
// (L2-resident), with 32-bit index arithmetic within the row.  Narrower rows, where that would
// leave threads idle or with one chunk each: two 16-byte chunks per thread over the flat chunk
// index of the whole tensor (grid-stride), each with its row's position and table entries.
// The prefill kernel rotates Q itself after loading it; this pass is for K (rotated once, as
// it is when written to a KV cache) or for any tensor a caller wants rotated.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Narrow rows: two 16-byte chunks of the flat chunk index per thread (idx and idx + stride), both
// loaded before either is stored; 32-bit index arithmetic when the tensor has fewer than 2^31
// chunks.
template <typename Idx>
__global__ void __launch_bounds__(256) fa_rope_flat_kernel(RopeParams p) {
  const int chunks = p.rotary_dim / 8;  // 16-byte chunks of the rotated part of a row and head
  const Idx per_row = (Idx)p.heads * (Idx)chunks;
  const Idx total = (Idx)p.rows * per_row;
  const int half = p.rotary_dim / 2;
  const Idx stride = (Idx)gridDim.x * blockDim.x;
  for (Idx i0 = (Idx)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    uint4 xv[2];
    float4 cv[2], sv[2];
    uint4* ptr[2];
    bool ok[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const Idx idx = i0 + (Idx)u * stride;
      ok[u] = false;
      if (idx < total) {
        const Idx r = idx / per_row;
        const int q = (int)(idx - r * per_row);
        const int h = q / chunks, c = q - h * chunks;
        const int pos = p.positions[r];
        ok[u] = pos >= 0 && pos < p.table_rows;
        if (!ok[u]) atomicOr(p.err, kDevErrBounds);  // no table row for this position: leave it, report it
        const size_t t0 = (size_t)(ok[u] ? pos : 0) * half + c * 4;
        ptr[u] = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.x) + ((size_t)r * p.heads + h) * p.d + c * 8);
        xv[u] = *ptr[u];
        cv[u] = __ldg(reinterpret_cast<const float4*>(p.cos_t + t0));
        sv[u] = __ldg(reinterpret_cast<const float4*>(p.sin_t + t0));
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (ok[u]) *ptr[u] = rope_rotate4(xv[u], cv[u], sv[u]);
  }
}

// Wide rows: one row per CTA at a time.
constexpr int kRopeThreads = 128;
constexpr int kRopeChunks = 4;  // 16-byte chunks a thread loads before it stores

__global__ void __launch_bounds__(kRopeThreads, 8) fa_rope_rows_kernel(RopeParams p) {
  // Thread t takes chunk c = t % chunks of heads t / chunks, t / chunks + hstep, ...: the same
  // four pairs of every head it visits, so it reads one float4 of each table per row.
  const int chunks = p.rotary_dim / 8;  // 16-byte chunks of the rotated part of one head
  const int hstep = kRopeThreads / chunks;
  const int c = threadIdx.x % chunks, h_first = threadIdx.x / chunks;
  if (h_first >= hstep) return;  // the threads past the last whole group of chunks
  const int half = p.rotary_dim / 2;
  for (long long r = blockIdx.x; r < p.rows; r += gridDim.x) {
    __nv_bfloat16* xr = reinterpret_cast<__nv_bfloat16*>(p.x) + r * p.heads * p.d + c * 8;
    const int pos = __ldg(p.positions + r);
    const bool okp = pos >= 0 && pos < p.table_rows;
    if (!okp && threadIdx.x == 0) atomicOr(p.err, kDevErrBounds);  // no table row: leave the row, report it
    const size_t t0 = (size_t)(okp ? pos : 0) * half + c * 4;
    const float4 cv = __ldg(reinterpret_cast<const float4*>(p.cos_t + t0));
    const float4 sv = __ldg(reinterpret_cast<const float4*>(p.sin_t + t0));
    for (int h0 = h_first; h0 < p.heads; h0 += hstep * kRopeChunks) {
      uint4 xv[kRopeChunks];
#pragma unroll
      for (int u = 0; u < kRopeChunks; ++u)
        if (h0 + u * hstep < p.heads) xv[u] = *reinterpret_cast<const uint4*>(xr + (h0 + u * hstep) * p.d);
      if (okp) {
#pragma unroll
        for (int u = 0; u < kRopeChunks; ++u)
          if (h0 + u * hstep < p.heads)
            *reinterpret_cast<uint4*>(xr + (h0 + u * hstep) * p.d) = rope_rotate4(xv[u], cv, sv);
      }
    }
  }
}

cudaError_t launch_rope(const RopeParams& p, int sm_count, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const int per_row = p.heads * (p.rotary_dim / 8);
  if (per_row >= kRopeThreads * kRopeChunks) {
    // measured on [32768, 32, 128], rotary_dim 128: 90 us against 101 us for the flat form
    long long blocks = p.rows;
    const long long cap = (long long)sm_count * 8;  // CTAs resident at once (registers), grid-stride beyond
    if (blocks > cap) blocks = cap;
    fa_rope_rows_kernel<<<(unsigned)blocks, kRopeThreads, 0, stream>>>(p);
  } else {
    const long long total = (long long)p.rows * per_row;
    long long blocks = (total + 511) / 512;
    const long long cap = (long long)sm_count * 6;  // CTAs resident at once (registers), grid-stride beyond
    if (blocks > cap) blocks = cap;
    // 32-bit indices while the index plus two grid strides stays below 2^32
    if (total < (1ll << 31)) fa_rope_flat_kernel<uint32_t><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else fa_rope_flat_kernel<long long><<<(unsigned)blocks, 256, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa
