/*
 * fa.h — C ABI of the GB300 (sm_103a) attention-forward library (libfa_gb300.so).
 *
 * The library computes the fused attention forward
 *     O = softmax(Q K^T * scale + mask) V,      LSE = log-sum-exp of each score row,
 * with a running-max / running-sum (online) softmax, so the score matrix never
 * reaches device memory.  The operation and its modes are those of the
 * ops-transformer pages:
 *   - the formula: jsqmd page "CANN Transformer算子库ops-transformer深度实践",
 *     §二 "SelfAttention的基础实现与瓶颈";
 *   - the fused, tiled evaluation (Q by row blocks, K/V by column blocks, all
 *     blocks reduced on chip): same page, §二 "FlashAttention的融合计算思想", and
 *     the hwcomputing.csdn.net page, §2.1 "分块计算策略与SRAM访存优化";
 *   - the max-subtracted softmax kept in fp32 with bf16/fp16 matmul inputs:
 *     hwcomputing.csdn.net page, §2.2 "数值稳定性优化";
 *   - causal, sliding-window and MQA/GQA modes: jsqmd page, §一 "核心能力矩阵"
 *     and §二 "因果掩码与解码优化" (implicit mask, no N x N mask tensor);
 *   - per-sequence valid lengths with no compute on padding: agent.csdn.net BERT
 *     walkthrough, 第三章 (actual_seq_q / actual_seq_kv) and 第六章;
 *   - incremental decode (one new token against the cached K/V): agent.csdn.net
 *     walkthrough, 结尾.
 *
 * Conventions shared by every entry point
 *   - All tensors live in device memory, are contiguous and row-major, and are
 *     owned by the caller; the library allocates no device memory.
 *   - q, k, v, o, caches: bf16.  lse and workspace: fp32.  Head dim d is 64 or 128.
 *   - Hq % Hkv == 0; query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *   - scale is the multiplier applied to Q K^T (e.g. 1/sqrt(d)); it must be > 0.
 *   - causal: bottom-right aligned — row i of a sequence with Lq queries and Lk
 *     keys may see key j iff j <= i + Lk - Lq.
 *   - window > 0: with causal, also j > i + Lk - Lq - window (the window holds the
 *     diagonal, so window = 1 keeps only it); without causal, |i + Lk - Lq - j| < window.
 *     window <= 0: no window.
 *   - A row that sees no key gets O = 0 and LSE = -inf.
 *   - LSE is the natural log of the row's normaliser in scaled-score units.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  Errors
 *     found on the host return before any launch; a failed launch returns
 *     FA_ERR_CUDA.  fa_last_error() describes the last failure of the calling
 *     thread.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same type as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = 1,     /* bad argument (null pointer, size, layout) */
  FA_ERR_UNSUPPORTED = 2, /* valid but not supported (d not 64/128, device not sm_103) */
  FA_ERR_CUDA = 3,        /* CUDA runtime/driver error */
  FA_ERR_TIMEOUT = 4      /* a kernel wait passed its time limit (see fa_device_status) */
} fa_status;

/*
 * Prefill / encoder attention forward on the padded-batch layout.
 *   q, o : [B, Nq, Hq, d] bf16          k, v : [B, Nk, Hkv, d] bf16
 *   lse  : [B, Hq, Nq] fp32 (may be NULL)
 *   seqlens_q, seqlens_k : NULL for full length, or device int32 [B] holding the
 *       valid length of each sequence (values clamped to [0, Nq] / [0, Nk]); rows
 *       and keys past a sequence's valid length take no part in the computation
 *       (the pages' actual_seq_q / actual_seq_kv), and output rows i with
 *       seqlens_q[b] <= i < Nq are written as O = 0, LSE = -inf.
 * Returns FA_ERR_INVALID for null q/k/v/o, non-positive sizes, Hq % Hkv != 0,
 * scale <= 0; FA_ERR_UNSUPPORTED for d not in {64, 128}.
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                 int causal, int window,
                 const int* seqlens_q, const int* seqlens_k,
                 fa_stream_t stream);

/*
 * Prefill on the packed variable-length layout (no padding rows at all).
 *   q, o : [total_q, Hq, d] bf16        k, v : [total_k, Hkv, d] bf16
 *   lse  : [Hq, total_q] fp32 (may be NULL)
 *   cu_seqlens_q, cu_seqlens_k : device int32 [B + 1], non-decreasing,
 *       cu[0] = 0, cu[B] = total; sequence b owns rows cu[b] .. cu[b+1]-1.
 *   max_seqlen_q / max_seqlen_k : upper bounds of the per-sequence lengths
 *       (the grid is sized from max_seqlen_q, so the caller must pass true bounds).
 *   cu_seqlens_q_host : optional host copy of cu_seqlens_q; when given it is
 *       checked (monotone, cu[0] = 0, cu[B] = total_q, lengths <= max_seqlen_q).
 * The kernel checks every sequence's device entries as well: a sequence whose
 * cu_seqlens_q/k entries are decreasing, run past total_q/total_k or exceed
 * max_seqlen_q/k is skipped (no row of it is written) and bit 1 of the device
 * status word is set (fa_device_status), so bad offsets cannot write outside o/lse.
 */
FA_API fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int total_q, int total_k,
                        int max_seqlen_q, int max_seqlen_k, int d, float scale,
                        int causal, int window,
                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                        const int* cu_seqlens_q_host,
                        fa_stream_t stream);

/*
 * All prefill options in one call (the entry points above are special cases).
 * Layout: packed when cu_seqlens_q and cu_seqlens_k are both set (as
 * fa_fwd_varlen: Nq/Nk are then the maximum lengths, total_q/total_k the row
 * counts, cu_seqlens_q_host optional), else padded (as fa_fwd, with optional
 * seqlens_q/seqlens_k).
 * alibi_slopes: NULL, or device fp32 [Hq]: ALiBi (jsqmd page, §三 "ALiBi位置编码的
 *   线性偏置") adds -alibi_slopes[h] * |p - j| to every scaled score, p the
 *   query's absolute position (i + Lk - Lq, the causal alignment).  The pages
 *   give no slope values; the caller chooses them.
 * rope_cos / rope_sin: NULL, or device fp32 tables [rope_rows, rope_dim / 2]: RoPE
 *   of Q fused into the kernel (jsqmd page, §三 "融合位置编码的Attention计算"): query
 *   row i is rotated at position p = i + Lk - Lq after it is loaded, pairs of
 *   adjacent dimensions (2j, 2j+1), j < rope_dim / 2, by (cos, sin)[p, j]; the
 *   result is rounded to bf16.  K must already be rotated (fa_rope), as it is in a
 *   KV cache.  rope_dim: multiple of 8, <= d; tables 16-byte aligned.  A query
 *   position outside [0, rope_rows) leaves that row unrotated and sets bit 1 of
 *   the device status word.  The rotation is the same arithmetic as fa_rope's, so
 *   rotating Q with fa_rope and calling without tables gives the same result; on
 *   GB300 the two cost about the same (within 1 %): the fused form saves a launch
 *   and a rotated copy of Q.
 */
typedef struct fa_fwd_args {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d;
  float scale;
  int causal, window;
  const int* seqlens_q;          /* padded layout (optional) */
  const int* seqlens_k;
  const int* cu_seqlens_q;       /* packed layout */
  const int* cu_seqlens_k;
  int total_q, total_k;
  const int* cu_seqlens_q_host;  /* packed layout, optional host copy for checking */
  const float* alibi_slopes;     /* optional */
  const float* rope_cos;         /* optional, with rope_sin, rope_rows, rope_dim */
  const float* rope_sin;
  int rope_rows, rope_dim;
} fa_fwd_args;

FA_API fa_status fa_fwd_ex(const fa_fwd_args* args, fa_stream_t stream);

/*
 * Rotary position embedding in place (the rotary_embedding op of the jsqmd page,
 * §三): x bf16 [rows, heads, d]; row r is rotated at position positions[r] (device
 * int32 [rows]) — pairs of adjacent dimensions (2j, 2j+1), j < rotary_dim / 2, by
 * cos_t / sin_t [table_rows, rotary_dim / 2] (device fp32), fp32 math, bf16
 * round-to-nearest-even result; dimensions >= rotary_dim are untouched.
 * rotary_dim: multiple of 8, <= d (FA_ERR_INVALID otherwise) and <= 1024
 * (FA_ERR_UNSUPPORTED above); heads x d below 2^31.  A position outside
 * [0, table_rows) leaves its row unchanged and sets bit 1 of the device status word.
 */
FA_API fa_status fa_rope(void* x, long long rows, int heads, int d, int rotary_dim, const int* positions,
                         const float* cos_t, const float* sin_t, int table_rows, fa_stream_t stream);

/*
 * Bytes of fp32 workspace fa_decode needs for a given split bound
 * (partial outputs [B, Hq, max_splits, d] and partial LSE [B, Hq, max_splits]).
 */
FA_API size_t fa_decode_workspace_size(int B, int Hq, int d, int max_splits);

/*
 * Single-query incremental decode over a KV cache, split over the key axis
 * and merged by a log-sum-exp combine kernel.
 *   q, o : [B, Hq, d] bf16 (the one new token of each sequence)
 *   k_cache, v_cache : [B, Ncap, Hkv, d] bf16; sequence b's keys are slots
 *       0 .. seqlens_k[b]-1 (the new token's K/V already appended)
 *   lse : [B, Hq] fp32 (may be NULL)
 *   seqlens_k : device int32 [B], values clamped to [0, Ncap]
 *   seqlens_k_host : optional host copy used only to plan the split size; it may
 *       overstate the device lengths but must not understate them: the plan covers
 *       max_splits chunks of keys, so keys of a longer device length past them would
 *       go unread — the combine kernel detects that case and sets bit 1 of the device
 *       status word (fa_device_status).  Without it the plan assumes Ncap keys.
 *   window : > 0 restricts the query to the last `window` keys
 *   num_splits : 0 = choose automatically; otherwise the maximum number of
 *       key chunks per sequence (each chunk a multiple of 64 keys)
 *   workspace : device memory of at least fa_decode_workspace_size(B, Hq, d, S)
 *       bytes, S the split bound actually used (fa_decode_max_splits tells it)
 * Returns FA_ERR_INVALID when workspace is NULL or too small.
 */
FA_API fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    int B, int Hq, int Hkv, int Ncap, int d, float scale, int window,
                    const int* seqlens_k, const int* seqlens_k_host,
                    int num_splits, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/*
 * Single-query decode over a paged KV cache (the plain gather of a block-table
 * KV cache: hwcomputing.csdn.net page, §4.1 "KV Cache内存优化", without its
 * importance-based selection).  As fa_decode, except for the cache layout:
 *   k_pages, v_pages : [num_pages, page_size, Hkv, d] bf16
 *   block_table : device int32 [B, max_blocks]; key j of sequence b lives in
 *       page block_table[b * max_blocks + j / page_size], row j % page_size
 *   page_size : a positive multiple of 64 (one 64-key tile never straddles pages)
 *   seqlens_k : device int32 [B], values clamped to [0, max_blocks * page_size]
 * A table entry outside [0, num_pages) sets bit 1 of the device status word
 * (fa_device_status) and reads page 0 instead; it cannot fault.
 * Workspace: fa_decode_workspace_size(B, Hq, d, S) with
 *   S = fa_decode_max_splits(B, Hq, Hkv, max_blocks * page_size,
 *                            window > 0 ? window + 63 : 0, seqlens_k_host, num_splits).
 */
FA_API fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o, float* lse,
                                 int B, int Hq, int Hkv, int num_pages, int page_size, int d, float scale,
                                 int window, const int* block_table, int max_blocks,
                                 const int* seqlens_k, const int* seqlens_k_host,
                                 int num_splits, void* workspace, size_t workspace_bytes,
                                 fa_stream_t stream);

/*
 * All decode options in one call (fa_decode and fa_decode_paged are special
 * cases).  The cache is paged when block_table is set (as fa_decode_paged: k/v
 * are the page pools, num_pages/page_size/max_blocks describe them), else
 * contiguous [B, Ncap, Hkv, d] (as fa_decode).  alibi_slopes as in fa_fwd_args:
 * the new token sits at position len - 1, so key j gets -m_h * (len - 1 - j).
 *
 * Nq (0 or 1: one token): new tokens per sequence, for speculative decoding or a
 * chunk of a prompt on top of a cache (the incremental mode of the agent.csdn.net
 * BERT walkthrough, 结尾, with several new tokens).  They are the last Nq cache
 * slots: token t of sequence b sits at position p = len_b - Nq + t and sees keys
 * j <= p (and j > p - window), the bottom-right alignment of fa_fwd.  Layouts:
 * q, o [B, Nq, Hq, d]; lse [B, Hq, Nq].  Tokens with p < 0 see no keys (O = 0,
 * LSE = -inf).  One CTA takes 16 (token, head) rows of a KV head, so K/V are read
 * ceil(Nq * Hq/Hkv / 16) times per KV head (from L2 when they are resident), while
 * fa_fwd with seqlens_k (128-row query tiles) reads them about once.  Measured on a
 * GB300 over a cache of 64 sequences x 8 KV heads x d=128, lengths U[512, 8192],
 * Hq/Hkv = 4: this entry point takes 0.18, 0.19, 0.26, 0.48, 0.94 ms for Nq = 1, 4,
 * 8, 16, 32 and fa_fwd 0.41-0.43 ms for every Nq up to 128 (0.81 at 256): use this
 * one up to Nq * Hq/Hkv = 32 rows per KV head and fa_fwd beyond.
 * Workspace: fa_decode_workspace_size(B * Nq, Hq, d, S) with S from
 * fa_decode_max_splits(B, Hq, Hkv, cap, window > 0 ? window + Nq - 1 : 0, ...)
 * (paged: window + Nq - 1 + 63), cap = Ncap or max_blocks * page_size.
 */
typedef struct fa_decode_args {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, d;
  float scale;
  int window;
  int Ncap;                      /* contiguous cache */
  const int* block_table;        /* paged cache (optional) */
  int max_blocks, page_size, num_pages;
  const int* seqlens_k;
  const int* seqlens_k_host;     /* optional */
  int num_splits;
  void* workspace;
  size_t workspace_bytes;
  const float* alibi_slopes;     /* optional */
  int Nq;                        /* new tokens per sequence; 0 or 1 = one */
} fa_decode_args;

FA_API fa_status fa_decode_ex(const fa_decode_args* args, fa_stream_t stream);

/*
 * The split bound S that fa_decode uses for the same arguments on the current
 * device (size the workspace with fa_decode_workspace_size(B, Hq, d, S)).
 * Returns 0 for invalid sizes.
 */
FA_API int fa_decode_max_splits(int B, int Hq, int Hkv, int Ncap, int window, const int* seqlens_k_host, int num_splits);

/*
 * fa_decode without any device allocation.  The attention pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc — for example a
 * plugin inside an inference engine that is handed only its input and output
 * buffers, or a serving loop that must not take the allocator's locks or the
 * device synchronisation an allocation can cause.
 *
 * Arguments and results are those of fa_decode, minus the workspace: the split
 * partials go to a fixed scratch array inside the library: 16 MiB (16777216
 * bytes) per device, held by every GPU that loads the library until the
 * process exits — enough for B = 64, Hq = 32, d = 128 with up to 15 splits.
 * A problem whose partials
 * (fa_decode_workspace_size for the split bound fa_decode_max_splits gives)
 * exceed it is rejected with FA_ERR_INVALID before any launch; a smaller
 * num_splits lowers the need.  The function calls no allocator: not cudaMalloc,
 * cudaFree, nor any allocating library routine.
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress with that device current) and caches it; make that
 * first call before any stream capture.  All calls on a device share the one
 * array, which keeps the last call's contents (nothing in it needs to start at
 * zero): calls that can overlap on the GPU — on different streams without
 * ordering between them — race on it and must not be issued that way.
 */
FA_API fa_status fa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                   int B, int Hq, int Hkv, int Ncap, int d, float scale, int window,
                                   const int* seqlens_k, const int* seqlens_k_host, int num_splits,
                                   fa_stream_t stream);

/* Description of the calling thread's last error ("" if none). */
FA_API const char* fa_last_error(void);

/*
 * Diagnostic: launch one warp that waits on a barrier nothing arrives at, through the same
 * bounded wait as every kernel, with a limit of limit_ms (1..1000) milliseconds.  The wait ends,
 * sets bit 0 of the device status word (fa_device_status) and the kernel returns: the check that
 * a wait which never completes ends with an error status, and leaves the context usable, instead
 * of hanging the GPU.  Asynchronous on `stream`; FA_ERR_INVALID for a limit out of range.
 */
FA_API fa_status fa_selftest_wait_timeout(int limit_ms, fa_stream_t stream);

/*
 * Diagnostic: fa_fwd_ex in which every CTA's V producer stops after v_loads (> 0) tile loads, so
 * the MMA issuer's wait for the next V tile gives up after the kernels' 2 s limit.  Every role then
 * unwinds: the waits of the others end on the abort flag, the P handoffs between the softmax warps
 * and the issuer (named barriers, which have no time limit) are completed without work by both
 * sides, copies and MMAs in flight are waited for, TMEM is freed and the kernel returns with bit 0
 * of the device status word set.  Outputs are then undefined.  The check that the abort path of the
 * prefill kernel ends instead of hanging; a problem whose CTAs need at most v_loads V tiles each
 * completes normally.  Asynchronous on `stream`; FA_ERR_INVALID for v_loads <= 0 and as fa_fwd_ex.
 */
FA_API fa_status fa_selftest_prefill_abort(const fa_fwd_args* args, int v_loads, fa_stream_t stream);

/*
 * Read (and optionally clear) the device status word of the current device:
 * bit 0 = some kernel wait passed its time limit, bit 1 = a device-side bounds
 * check fired.  Synchronises the device.  Returns FA_ERR_TIMEOUT when bits
 * are set, FA_OK otherwise.
 */
FA_API fa_status fa_device_status(uint32_t* bits, int clear);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
