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
// How: an elementwise, HBM-bound pass; one thread moves 16 bytes (four pairs) of one
// row and head with one 16-byte load and store, plus two 16-byte table loads.  The
// prefill kernel rotates Q itself after loading it; this pass is for K (rotated once,
// as it is when written to a KV cache) or for any tensor a caller wants rotated.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

__global__ void __launch_bounds__(256) fa_rope_kernel(RopeParams p) {
  const int chunks = p.rotary_dim / 8;  // 16-byte chunks of the rotated part of a row
  const long long total = (long long)p.rows * p.heads * chunks;
  const int half = p.rotary_dim / 2;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % chunks);
    const long long rh = idx / chunks;
    const int h = (int)(rh % p.heads);
    const long long r = rh / p.heads;
    const int pos = p.positions[r];
    if (pos < 0 || pos >= p.table_rows) {  // no table row for this position: leave it, report it
      atomicOr(p.err, kDevErrBounds);
      continue;
    }
    uint4* ptr = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.x) + (r * p.heads + h) * p.d + c * 8);
    const float4 cc = *reinterpret_cast<const float4*>(p.cos_t + (size_t)pos * half + c * 4);
    const float4 ss = *reinterpret_cast<const float4*>(p.sin_t + (size_t)pos * half + c * 4);
    *ptr = rope_rotate4(*ptr, cc, ss);
  }
}

cudaError_t launch_rope(const RopeParams& p, int sm_count, cudaStream_t stream) {
  const long long total = (long long)p.rows * p.heads * (p.rotary_dim / 8);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sm_count * 8;  // grid-stride beyond a few waves
  if (blocks > cap) blocks = cap;
  fa_rope_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
