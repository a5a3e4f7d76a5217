// C-ABI layer of libfa_gb300: argument checks, TMA descriptors, split planning,
// kernel launches.  Declarations and their contracts are in include/fa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace {

thread_local std::string g_last_error;

fa_status fail(fa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  cudaGetLastError();  // clear a sticky launch error
  return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

// Per-device status word the kernels OR error bits into.
__device__ uint32_t g_fa_status_word;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  uint32_t* status = nullptr;  // device address of g_fa_status_word
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The last supported device this thread used: repeated calls on one device skip the lock.
thread_local int t_last_dev = -1;
thread_local DeviceInfo* t_last_info = nullptr;

fa_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev == t_last_dev) {
    *out = t_last_info;
    return FA_OK;
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    di.supported = (major == 10 && minor == 3);
    void* addr = nullptr;
    if ((e = cudaGetSymbolAddress(&addr, g_fa_status_word)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    di.status = static_cast<uint32_t*>(addr);
    di.ready = true;
  }
  if (!di.supported) return fail(FA_ERR_UNSUPPORTED, "device %d is not sm_103 (GB300)", dev);
  t_last_dev = dev;
  t_last_info = &di;
  *out = &di;
  return FA_OK;
}

fa_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return FA_OK;
}

// 3-D view [rows, heads, d] of a row-major bf16 tensor; box = 64 columns x 1 head x box_rows rows,
// 128-byte swizzle (the layout the kernels' shared-memory descriptors assume).
fa_status encode_map(CUtensorMap* map, const void* base, int d, int heads, long long rows, int box_rows,
                     const char* name) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
  return FA_OK;
}

// Encoding a descriptor is a host call of a few microseconds; repeated calls on the same tensors
// (the usual case: one layer called step after step) reuse a small per-thread cache.  A descriptor
// depends only on the address, sizes and box, so a hit is always valid.
struct MapCacheEntry {
  const void* base = nullptr;
  int d = 0, heads = 0, box_rows = 0;
  long long rows = 0;
  CUtensorMap map;
};
constexpr int kMapCache = 16;
thread_local MapCacheEntry t_map_cache[kMapCache];
thread_local int t_map_next = 0;

fa_status make_map(CUtensorMap* map, const void* base, int d, int heads, long long rows, int box_rows,
                   const char* name) {
  for (int i = 0; i < kMapCache; ++i) {
    const MapCacheEntry& e = t_map_cache[i];
    if (e.base == base && e.d == d && e.heads == heads && e.rows == rows && e.box_rows == box_rows) {
      *map = e.map;
      return FA_OK;
    }
  }
  fa_status st = encode_map(map, base, d, heads, rows, box_rows, name);
  if (st != FA_OK) return st;
  MapCacheEntry& e = t_map_cache[t_map_next];
  t_map_next = (t_map_next + 1) % kMapCache;
  e.base = base;
  e.d = d;
  e.heads = heads;
  e.rows = rows;
  e.box_rows = box_rows;
  e.map = *map;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_common(const void* q, const void* k, const void* v, void* o, const float* lse, int B, int Hq,
                       int Hkv, int d, float scale) {
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID, "q, k, v and o must be non-null");
  if (B <= 0 || Hq <= 0 || Hkv <= 0) return fail(FA_ERR_INVALID, "B, Hq, Hkv must be positive");
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(FA_ERR_INVALID, "scale must be finite and > 0");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(FA_ERR_INVALID, "q, k, v, o must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(FA_ERR_INVALID, "lse must be 4-byte aligned");
  return FA_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// fa_fwd_ex with, for the abort self-test, a cap on each CTA's V loads (0: none).
fa_status fwd_impl(const fa_fwd_args* a, int v_load_cap, fa_stream_t stream);

}  // namespace

extern "C" {

const char* fa_last_error(void) { return g_last_error.c_str(); }

fa_status fa_fwd_ex(const fa_fwd_args* a, fa_stream_t stream) { return fwd_impl(a, 0, stream); }

fa_status fa_selftest_prefill_abort(const fa_fwd_args* a, int v_loads, fa_stream_t stream) {
  if (v_loads <= 0) return fail(FA_ERR_INVALID, "v_loads must be positive");
  return fwd_impl(a, v_loads, stream);
}

}  // extern "C"

namespace {

fa_status fwd_impl(const fa_fwd_args* a, int v_load_cap, fa_stream_t stream) {
  if (!a) return fail(FA_ERR_INVALID, "args must be non-null");
  const int B = a->B, Hq = a->Hq, Hkv = a->Hkv, d = a->d, window = a->window;
  fa_status st = check_common(a->q, a->k, a->v, a->o, a->lse, B, Hq, Hkv, d, a->scale);
  if (st != FA_OK) return st;
  if (a->alibi_slopes && (reinterpret_cast<uintptr_t>(a->alibi_slopes) & 3u))
    return fail(FA_ERR_INVALID, "alibi_slopes must be 4-byte aligned");
  if (a->rope_cos || a->rope_sin) {
    if (!a->rope_cos || !a->rope_sin) return fail(FA_ERR_INVALID, "rope_cos and rope_sin go together");
    if (a->rope_dim <= 0 || a->rope_dim % 8 != 0 || a->rope_dim > d)
      return fail(FA_ERR_INVALID, "rope_dim (%d) must be a positive multiple of 8, at most d", a->rope_dim);
    if (a->rope_rows <= 0) return fail(FA_ERR_INVALID, "rope_rows must be positive");
    if (!aligned16(a->rope_cos) || !aligned16(a->rope_sin))
      return fail(FA_ERR_INVALID, "rope tables must be 16-byte aligned");
  }
  const bool packed = a->cu_seqlens_q || a->cu_seqlens_k;
  long long q_rows, k_rows;
  int max_rows;
  if (packed) {
    if (!a->cu_seqlens_q || !a->cu_seqlens_k) return fail(FA_ERR_INVALID, "cu_seqlens_q/k must be non-null");
    if (a->total_q < 0 || a->total_k < 0 || a->Nq < 0 || a->Nk < 0)
      return fail(FA_ERR_INVALID, "totals and max lengths must be >= 0");
    if ((long long)a->Nq + a->Nk + (window > 0 ? window : 0) >= (1LL << 30))
      return fail(FA_ERR_INVALID, "sequence lengths too large");
    if (const int* cu = a->cu_seqlens_q_host) {
      if (cu[0] != 0) return fail(FA_ERR_INVALID, "cu_seqlens_q[0] must be 0");
      for (int b = 0; b < B; ++b) {
        const int len = cu[b + 1] - cu[b];
        if (len < 0) return fail(FA_ERR_INVALID, "cu_seqlens_q must be non-decreasing (at %d)", b);
        if (len > a->Nq) return fail(FA_ERR_INVALID, "sequence %d longer than max_seqlen_q", b);
      }
      if (cu[B] != a->total_q) return fail(FA_ERR_INVALID, "cu_seqlens_q[B] != total_q");
    }
    if (a->total_q == 0 || a->Nq == 0) return FA_OK;  // nothing to compute
    q_rows = a->total_q;
    k_rows = a->total_k > 0 ? a->total_k : 1;  // a map needs one row; no key row is read when total_k = 0
    max_rows = a->Nq;
  } else {
    if (a->Nq <= 0 || a->Nk <= 0) return fail(FA_ERR_INVALID, "Nq and Nk must be positive");
    if ((long long)B * a->Nq >= (1LL << 31) || (long long)B * a->Nk >= (1LL << 31))
      return fail(FA_ERR_INVALID, "B * N must be below 2^31 rows");
    if ((long long)a->Nq + a->Nk + (window > 0 ? window : 0) >= (1LL << 30))
      return fail(FA_ERR_INVALID, "sequence lengths too large");
    q_rows = (long long)B * a->Nq;
    k_rows = (long long)B * a->Nk;
    max_rows = a->Nq;
  }
  if (B > 65535) return fail(FA_ERR_INVALID, "grid too large");
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  if ((st = get_encoder()) != FA_OK) return st;
  const int bm = fa::prefill_box_rows();
  CUtensorMap tq, tk, tv, to;
  if ((st = make_map(&tq, a->q, d, Hq, q_rows, bm, "q")) != FA_OK) return st;
  if ((st = make_map(&to, a->o, d, Hq, q_rows, bm, "o")) != FA_OK) return st;
  if ((st = make_map(&tk, a->k, d, Hkv, k_rows, 128, "k")) != FA_OK) return st;
  if ((st = make_map(&tv, a->v, d, Hkv, k_rows, 128, "v")) != FA_OK) return st;
  fa::PrefillParams p{};
  p.o = a->o;
  p.lse = a->lse;
  p.cu_q = packed ? a->cu_seqlens_q : nullptr;
  p.cu_k = packed ? a->cu_seqlens_k : nullptr;
  p.seqlens_q = packed ? nullptr : a->seqlens_q;
  p.seqlens_k = packed ? nullptr : a->seqlens_k;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = a->Nq;
  p.Nk = a->Nk;
  p.total_q = packed ? a->total_q : 0;
  p.total_k = packed ? a->total_k : 0;
  p.group = Hq / Hkv;
  p.scale_log2 = a->scale * kLog2e;
  p.causal = a->causal ? 1 : 0;
  p.window = window > 0 ? window : 0;
  p.err = di->status;
  p.alibi = a->alibi_slopes;
  if (a->rope_cos) {
    p.rope_cos = a->rope_cos;
    p.rope_sin = a->rope_sin;
    p.rope_rows = a->rope_rows;
    p.rope_dim = a->rope_dim;
  }
  p.v_load_cap = v_load_cap;
  cudaError_t e = fa::launch_prefill(d, tq, tk, tv, to, p, max_rows, di->sm_count, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                 int Nk, int d, float scale, int causal, int window, const int* seqlens_q, const int* seqlens_k,
                 fa_stream_t stream) {
  fa_fwd_args a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.seqlens_q = seqlens_q;
  a.seqlens_k = seqlens_k;
  return fa_fwd_ex(&a, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, float scale,
                        int causal, int window, const int* cu_seqlens_q, const int* cu_seqlens_k,
                        const int* cu_seqlens_q_host, fa_stream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return fail(FA_ERR_INVALID, "cu_seqlens_q/k must be non-null");
  fa_fwd_args a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = max_seqlen_q;
  a.Nk = max_seqlen_k;
  a.d = d;
  a.scale = scale;
  a.causal = causal;
  a.window = window;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_q = total_q;
  a.total_k = total_k;
  a.cu_seqlens_q_host = cu_seqlens_q_host;
  return fa_fwd_ex(&a, stream);
}

size_t fa_decode_workspace_size(int B, int Hq, int d, int max_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || max_splits <= 0) return 0;
  return (size_t)B * Hq * max_splits * ((size_t)d + 1) * sizeof(float);
}

namespace {

struct DecodePlan {
  int chunk;
  int max_splits;
};

DecodePlan plan_decode(int B, int Hkv, int group, int Ncap, int window, const int* lens_host, int num_splits,
                       int sm_count) {
  const int bn = fa::decode_block_n();
  const int cap = window > 0 ? (window < Ncap ? window : Ncap) : Ncap;
  long long total = 0;
  int longest = 0;
  for (int b = 0; b < B; ++b) {
    int len = lens_host ? lens_host[b] : Ncap;
    len = len < 0 ? 0 : (len > Ncap ? Ncap : len);
    const int eff = window > 0 && len > window ? window : len;
    total += eff;
    longest = eff > longest ? eff : longest;
  }
  if (!lens_host) longest = cap;
  if (longest <= 0) longest = 1;
  int chunk;
  if (num_splits > 0) {
    chunk = (longest + num_splits - 1) / num_splits;
  } else {
    // Aim for ~4 resident-CTA waves of equal-sized chunks: enough that the tail wave is short,
    // few enough that the split partials (written here, read back by the combine; nq times more
    // with several new tokens) stay a small share of the bytes.  Measured on decode_cache:
    // 2, 3, 4, 6 and 8 waves took 181.8, 179.6, 178.5, 179.6 and 180.6 us.
    const long long units = (long long)sm_count * 2 * 4;
    const long long row_blocks = (long long)Hkv * ((group + 15) / 16);
    const long long keys = total * row_blocks;
    chunk = (int)((keys + units - 1) / units);
    if (chunk < 256) chunk = 256;
  }
  chunk = ((chunk + bn - 1) / bn) * bn;
  if (chunk < bn) chunk = bn;
  DecodePlan pl;
  pl.chunk = chunk;
  pl.max_splits = (longest + chunk - 1) / chunk;
  if (pl.max_splits < 1) pl.max_splits = 1;
  return pl;
}

}  // namespace

int fa_decode_max_splits(int B, int Hq, int Hkv, int Ncap, int window, const int* seqlens_k_host,
                         int num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Ncap <= 0 || Hq % Hkv != 0 || num_splits < 0) return 0;
  int sm = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sm <= 0) {
    cudaGetLastError();
    sm = 152;
  }
  return plan_decode(B, Hkv, Hq / Hkv, Ncap, window, seqlens_k_host, num_splits, sm).max_splits;
}

fa_status fa_decode_ex(const fa_decode_args* a, fa_stream_t stream) {
  if (!a) return fail(FA_ERR_INVALID, "args must be non-null");
  const int B = a->B, Hq = a->Hq, Hkv = a->Hkv, d = a->d, window = a->window;
  fa_status st = check_common(a->q, a->k, a->v, a->o, a->lse, B, Hq, Hkv, d, a->scale);
  if (st != FA_OK) return st;
  if (!a->seqlens_k) return fail(FA_ERR_INVALID, "seqlens_k must be non-null");
  if (a->num_splits < 0) return fail(FA_ERR_INVALID, "num_splits must be >= 0");
  if (a->alibi_slopes && (reinterpret_cast<uintptr_t>(a->alibi_slopes) & 3u))
    return fail(FA_ERR_INVALID, "alibi_slopes must be 4-byte aligned");
  if (B > 65535) return fail(FA_ERR_INVALID, "B too large");
  if (a->Nq < 0) return fail(FA_ERR_INVALID, "Nq must be >= 0");
  const int nq = a->Nq > 1 ? a->Nq : 1;
  if ((long long)Hkv * (((long long)nq * (Hq / Hkv) + 15) / 16) > 65535 || (long long)B * nq * Hq >= (1LL << 31))
    return fail(FA_ERR_INVALID, "Nq (%d) too large for one launch", nq);
  const bool paged = a->block_table != nullptr;
  long long rows;  // rows of the K/V tensors as TMA sees them
  int cap;         // keys a sequence can hold
  if (paged) {
    if (a->page_size <= 0 || a->page_size % 64 != 0)
      return fail(FA_ERR_INVALID, "page_size (%d) must be a positive multiple of 64", a->page_size);
    if (a->num_pages <= 0 || a->max_blocks <= 0)
      return fail(FA_ERR_INVALID, "num_pages and max_blocks must be positive");
    if ((long long)a->num_pages * a->page_size >= (1LL << 31) || (long long)a->max_blocks * a->page_size >= (1LL << 30))
      return fail(FA_ERR_INVALID, "paged cache too large");
    rows = (long long)a->num_pages * a->page_size;
    cap = a->max_blocks * a->page_size;
  } else {
    if (a->Ncap <= 0) return fail(FA_ERR_INVALID, "Ncap must be positive");
    if ((long long)B * a->Ncap >= (1LL << 31)) return fail(FA_ERR_INVALID, "B * Ncap must be below 2^31 rows");
    rows = (long long)B * a->Ncap;
    cap = a->Ncap;
  }
  DeviceInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  // the keys of a sequence's Nq tokens span window + Nq - 1 slots; paged chunks start on a 64-key
  // boundary at or below the window start: plan with 63 more
  const int plan_window = window > 0 ? window + (nq - 1) + (paged ? 63 : 0) : window;
  const DecodePlan pl =
      plan_decode(B, Hkv, Hq / Hkv, cap, plan_window, a->seqlens_k_host, a->num_splits, di->sm_count);
  const size_t need = fa_decode_workspace_size(B * nq, Hq, d, pl.max_splits);
  if (!a->workspace) return fail(FA_ERR_INVALID, "workspace must be non-null (%zu bytes needed)", need);
  if (!aligned16(a->workspace)) return fail(FA_ERR_INVALID, "workspace must be 16-byte aligned");
  if (a->workspace_bytes < need)
    return fail(FA_ERR_INVALID, "workspace too small: %zu bytes given, %zu needed", a->workspace_bytes, need);
  if (pl.max_splits > 65535) return fail(FA_ERR_INVALID, "too many splits");
  if ((st = get_encoder()) != FA_OK) return st;
  CUtensorMap tk, tv;
  const int bn = fa::decode_block_n();
  if ((st = make_map(&tk, a->k, d, Hkv, rows, bn, "k cache")) != FA_OK) return st;
  if ((st = make_map(&tv, a->v, d, Hkv, rows, bn, "v cache")) != FA_OK) return st;
  fa::DecodeParams p{};
  p.q = a->q;
  p.o = a->o;
  p.lse = a->lse;
  p.seqlens_k = a->seqlens_k;
  p.o_part = static_cast<float*>(a->workspace);
  p.lse_part = p.o_part + (size_t)B * nq * Hq * pl.max_splits * d;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Ncap = cap;
  p.group = Hq / Hkv;
  p.nq = nq;
  p.chunk = pl.chunk;
  p.max_splits = pl.max_splits;
  p.window = window > 0 ? window : 0;
  p.scale_log2 = a->scale * kLog2e;
  p.err = di->status;
  if (paged) {
    p.block_table = a->block_table;
    p.max_blocks = a->max_blocks;
    p.page_size = a->page_size;
    p.num_pages = a->num_pages;
  }
  p.alibi = a->alibi_slopes;
  cudaError_t e = fa::launch_decode(d, tk, tv, p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return FA_OK;
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Hq,
                    int Hkv, int Ncap, int d, float scale, int window, const int* seqlens_k,
                    const int* seqlens_k_host, int num_splits, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
  fa_decode_args a{};
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.scale = scale;
  a.window = window;
  a.Ncap = Ncap;
  a.seqlens_k = seqlens_k;
  a.seqlens_k_host = seqlens_k_host;
  a.num_splits = num_splits;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return fa_decode_ex(&a, stream);
}

fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o, float* lse, int B,
                          int Hq, int Hkv, int num_pages, int page_size, int d, float scale, int window,
                          const int* block_table, int max_blocks, const int* seqlens_k, const int* seqlens_k_host,
                          int num_splits, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!block_table) return fail(FA_ERR_INVALID, "seqlens_k and block_table must be non-null");
  fa_decode_args a{};
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.scale = scale;
  a.window = window;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.seqlens_k = seqlens_k;
  a.seqlens_k_host = seqlens_k_host;
  a.num_splits = num_splits;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return fa_decode_ex(&a, stream);
}

fa_status fa_rope(void* x, long long rows, int heads, int d, int rotary_dim, const int* positions,
                  const float* cos_t, const float* sin_t, int table_rows, fa_stream_t stream) {
  if (!x || !positions || !cos_t || !sin_t) return fail(FA_ERR_INVALID, "x, positions and tables must be non-null");
  if (rows < 0 || heads <= 0 || d <= 0 || table_rows <= 0) return fail(FA_ERR_INVALID, "bad sizes");
  if (rotary_dim <= 0 || rotary_dim % 8 != 0 || rotary_dim > d)
    return fail(FA_ERR_INVALID, "rotary_dim (%d) must be a positive multiple of 8, at most d", rotary_dim);
  if (d % 8 != 0) return fail(FA_ERR_INVALID, "d must be a multiple of 8");
  if (rotary_dim > 1024) return fail(FA_ERR_UNSUPPORTED, "rotary_dim (%d) above 1024", rotary_dim);
  if ((long long)heads * d > 0x7fffffffLL) return fail(FA_ERR_INVALID, "heads x d must fit in 31 bits");
  if (!aligned16(x) || !aligned16(cos_t) || !aligned16(sin_t))
    return fail(FA_ERR_INVALID, "x and the tables must be 16-byte aligned");
  if (rows == 0) return FA_OK;
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  fa::RopeParams p{};
  p.x = x;
  p.positions = positions;
  p.cos_t = cos_t;
  p.sin_t = sin_t;
  p.rows = rows;
  p.heads = heads;
  p.d = d;
  p.rotary_dim = rotary_dim;
  p.table_rows = table_rows;
  p.err = di->status;
  cudaError_t e = fa::launch_rope(p, di->sm_count, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rope launch");
  return FA_OK;
}

namespace fa {
// One warp waits on an mbarrier that nothing arrives at, through the same bounded wait every
// kernel uses, with a short limit: the wait must end with the timeout bit in the status word.
__global__ void fa_selftest_wait_kernel(uint32_t* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}
}  // namespace fa

fa_status fa_selftest_wait_timeout(int limit_ms, fa_stream_t stream) {
  if (limit_ms <= 0 || limit_ms > 1000) return fail(FA_ERR_INVALID, "limit_ms must be in 1..1000");
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  fa::fa_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      di->status, (unsigned long long)limit_ms * 1000000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return FA_OK;
}

fa_status fa_device_status(uint32_t* bits, int clear) {
  DeviceInfo* di = nullptr;
  fa_status st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t v = 0;
  if ((e = cudaMemcpy(&v, di->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status word");
  if (clear && v) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(di->status, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear status word");
  }
  if (bits) *bits = v;
  if (v) return fail(FA_ERR_TIMEOUT, "device status word 0x%x (bit0 wait timeout, bit1 bounds)", v);
  return FA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Decode without any device allocation (fa_decode_noalloc, declared in include/fa.h).
//
// Some callers cannot call cudaMalloc: a plugin inside an inference engine that is handed only
// its input and output buffers, or a serving loop that must never take the allocator's locks or
// the device synchronisation an allocation can cause.  For them the split-KV partials live in
// this fixed, file-scope device array instead of a caller workspace.  Every GPU that loads the
// library holds the array until the process exits, so it is kept modest: 16 MiB, enough for the
// partials of B x Hq x splits x (d + 1) fp32 values up to that size (for example B = 64, Hq = 32,
// d = 128 with up to 15 splits).
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch, looked up once per device with that device current.
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

fa_status decode_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    if (!p) return fail(FA_ERR_CUDA, "cudaGetSymbolAddress(decode scratch) returned null");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                       int B, int Hq, int Hkv, int Ncap, int d, float scale, int window,
                                       const int* seqlens_k, const int* seqlens_k_host, int num_splits,
                                       fa_stream_t stream) {
  // Reject problems whose partials do not fit before touching the device.
  const int S = fa_decode_max_splits(B, Hq, Hkv, Ncap, window, seqlens_k_host, num_splits);
  if (S > 0) {
    const size_t need = fa_decode_workspace_size(B, Hq, d, S);
    if (need > kNoAllocScratchBytes)
      return fail(FA_ERR_INVALID,
                  "fa_decode_noalloc: these sizes need %zu bytes of split scratch (B=%d, Hq=%d, d=%d, %d splits) "
                  "but the built-in scratch holds %zu bytes; pass a smaller num_splits or call fa_decode "
                  "with a caller-owned workspace",
                  need, B, Hq, d, S, kNoAllocScratchBytes);
  }
  void* scratch = nullptr;
  fa_status st = decode_scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Ncap, d, scale, window, seqlens_k, seqlens_k_host,
                   num_splits, scratch, kNoAllocScratchBytes, stream);
}

