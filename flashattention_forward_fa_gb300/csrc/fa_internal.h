// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

struct PrefillParams {
  void* o;                 // bf16 output
  float* lse;              // fp32 LSE or nullptr
  const int* cu_q;         // packed layout: int32 [B + 1] (nullptr otherwise)
  const int* cu_k;
  const int* seqlens_q;    // padded layout: int32 [B] valid lengths (nullptr = full)
  const int* seqlens_k;
  int B, Hq, Hkv, Nq, Nk;  // dense/padded: rows per sequence; packed: max lengths
  int total_q, total_k;     // packed: rows of q / k (the LSE is [Hq, total_q])
  int group;               // Hq / Hkv
  float scale_log2;        // scale * log2(e)
  int causal, window;
  uint32_t* err;           // device status word
  const float* alibi;      // per-query-head ALiBi slopes (fp32 [Hq]) or nullptr
  // RoPE of Q inside the kernel (rope_cos == nullptr: none): tables [rope_rows, rope_dim / 2]
  const float* rope_cos;
  const float* rope_sin;
  int rope_rows, rope_dim;
  int n_qblk;              // row blocks per sequence (set by the launcher)
  int pair_heads;          // items pair two query heads of one KV group (set by the launcher)
  int v_load_cap;          // > 0: each CTA's V producer issues only this many loads (the abort self-test)
};

struct RopeParams {
  void* x;                 // bf16 [rows, heads, d], rotated in place
  const int* positions;    // int32 [rows]
  const float* cos_t;      // fp32 [table_rows, rotary_dim / 2]
  const float* sin_t;
  long long rows;
  int heads, d, rotary_dim, table_rows;
  uint32_t* err;
};

cudaError_t launch_rope(const RopeParams& p, int sm_count, cudaStream_t stream);

struct DecodeParams {
  const void* q;           // bf16 [B, nq, Hq, d]
  void* o;                 // bf16 [B, nq, Hq, d]
  float* lse;              // fp32 [B, Hq, nq] or nullptr
  const int* seqlens_k;    // int32 [B]
  float* o_part;           // fp32 [B, nq, Hq, max_splits, d]
  float* lse_part;         // fp32 [B, nq, Hq, max_splits]
  int B, Hq, Hkv, Ncap, group;
  int nq;                  // new tokens per sequence (the last nq cache slots)
  int chunk;               // keys per split (multiple of 64)
  int max_splits;
  int window;
  float scale_log2;
  uint32_t* err;
  // paged cache (page_size > 0): k/v are [num_pages, page_size, Hkv, d] and key j of sequence b
  // lives in page block_table[b * max_blocks + j / page_size]; page_size is a multiple of 64.
  const int* block_table;
  int max_blocks, page_size, num_pages;
  const float* alibi;      // per-query-head ALiBi slopes (fp32 [Hq]) or nullptr
};

// max_rows: rows per sequence (padded layout) or the longest sequence (packed layout).
cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to,
                           const PrefillParams& p, int max_rows, int sm_count, cudaStream_t stream);
int prefill_box_rows();  // rows of one TMA box of Q / K / V / O

cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                          cudaStream_t stream);  // paged when p.page_size > 0
int decode_block_n();

}  // namespace fa
