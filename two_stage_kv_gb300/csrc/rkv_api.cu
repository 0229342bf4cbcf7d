// C ABI of the library (declared in include/rkv.h): host-side argument checks,
// TMA descriptor encoding and kernel launches.  Every entry point validates its
// arguments before any launch and returns a status; no exception escapes.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "rkv.h"
#include "rkv_internal.h"

namespace {

thread_local std::string g_last_error;

// Bounded-wait test setting (rkv_debug_set_wait): 0 = normal operation.
std::atomic<uint64_t> g_test_wait_ns{0};
std::atomic<uint32_t> g_test_extra_tx{0};

rkv_status fail(rkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

rkv_status cuda_fail(cudaError_t e, const char* where) {
  return fail(RKV_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

// One NVTX range per entry point call (its name), so a profiler timeline shows
// each library call around the kernels it launched; without a profiler
// attached a push / pop costs a few nanoseconds.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The address kernels use for a source that may live in device memory or in
// page-locked host memory (read over the host link; only the rows a kernel
// touches cross it).  Anything else is refused rather than dereferenced.
rkv_status device_view(const void* p, const void** out, const char* what) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return fail(RKV_ERR_INVALID_ARG, "%s: not an address the device can reach", what);
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *out = p;
    return RKV_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    *out = at.devicePointer;
    return RKV_OK;
  }
  return fail(RKV_ERR_INVALID_ARG, "%s must be device memory or page-locked host memory", what);
}

// Refuses a pointer that is not device (or managed) memory of the current
// context: a made-up or host address must never reach a kernel.
rkv_status require_device(const void* p, const char* what) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return fail(RKV_ERR_INVALID_ARG, "%s: not an address the device can reach", what);
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return RKV_OK;
  return fail(RKV_ERR_INVALID_ARG, "%s must be device memory", what);
}

rkv_status check_dims(const rkv_dims& d) {
  if (d.batch < 0 || d.n_q_heads < 1 || d.n_kv_heads < 1 || d.head_dim < 1)
    return fail(RKV_ERR_INVALID_ARG, "dims: batch=%d Hq=%d Hkv=%d D=%d", d.batch, d.n_q_heads, d.n_kv_heads,
                d.head_dim);
  if (d.n_q_heads % d.n_kv_heads != 0)
    return fail(RKV_ERR_INVALID_ARG, "dims: Hq=%d is not a multiple of Hkv=%d", d.n_q_heads, d.n_kv_heads);
  if (d.head_dim != rkv::HD_HOST)
    return fail(RKV_ERR_UNSUPPORTED, "dims: head_dim=%d (only 128 is implemented)", d.head_dim);
  if (d.n_q_heads / d.n_kv_heads > 16)
    return fail(RKV_ERR_UNSUPPORTED, "dims: group size %d > 16", d.n_q_heads / d.n_kv_heads);
  return RKV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a [pairs, cap, 128] bf16 cache: rows >= `rows` read as zero.
// Box = 64 channels (128 bytes, 128-byte swizzle) x box_rows rows x 1 pair.
rkv_status make_kv_map(CUtensorMap* m, const void* base, int64_t pairs, int64_t cap, int64_t rows, int box_rows,
                       const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)rkv::HD_HOST, (cuuint64_t)rows, (cuuint64_t)pairs};
  cuuint64_t strides[2] = {(cuuint64_t)rkv::HD_HOST * 2, (cuuint64_t)cap * rkv::HD_HOST * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return RKV_OK;
}

// 3-D map over a [pairs, cap, 128] e4m3 code cache (128-byte rows): rows >= `rows`
// read as zero.  Box = 128 codes x box_rows rows x 1 pair, unswizzled.
rkv_status make_kv_map_u8(CUtensorMap* m, const void* base, int64_t pairs, int64_t cap, int64_t rows, int box_rows,
                          const char* what) {
  auto fn = encode_fn();
  if (!fn) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)rkv::HD_HOST, (cuuint64_t)rows, (cuuint64_t)pairs};
  cuuint64_t strides[2] = {(cuuint64_t)rkv::HD_HOST, (cuuint64_t)cap * rkv::HD_HOST};
  cuuint32_t box[3] = {(cuuint32_t)rkv::HD_HOST, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return RKV_OK;
}

// 2-D map over the KT cache viewed as [pairs * 2 * 128 rows, nblk_cap] bf16, box
// box_cols blocks x 256 rows (all Kmax and Kmin rows of one pair), no swizzle.
// (e4m3 codes: one byte per entry, box_cols a multiple of 16)
rkv_status make_kt_map(CUtensorMap* m, const void* base, int64_t pairs, int64_t nblk_cap, int box_cols,
                       bool f8 = false) {
  auto fn = encode_fn();
  if (!fn) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)nblk_cap, (cuuint64_t)pairs * 2 * rkv::HD_HOST};
  cuuint64_t strides[1] = {(cuuint64_t)nblk_cap * (f8 ? 1 : 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, 2 * rkv::HD_HOST};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                  dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled(kt) failed with %d", (int)r);
  return RKV_OK;
}

// 2-D map over window queries [rows, 128] bf16, box 64 channels x box_rows rows (128-byte swizzle).
rkv_status make_q_map(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)rkv::HD_HOST, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)rkv::HD_HOST * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RKV_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed with %d", (int)r);
  return RKV_OK;
}

rkv_status hsa_common(const rkv_dims& d, const void* q, void* k, void* v, int64_t cap, int32_t* idx,
                      int64_t idx_cap, int64_t n, void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2,
                      float scale, float* out, int32_t* sel_blocks, int32_t* sel_channels, const void* k_new,
                      const void* v_new, int64_t row, void* stream, bool mt, const int32_t* n_rows = nullptr,
                      const int32_t* block_table = nullptr, int64_t bt_stride = 0, int64_t num_pages = 0,
                      const uint32_t* mask = nullptr, int64_t mask_ld = 0, int64_t n_prompt = 0,
                      const float* k_scale = nullptr, const float* v_scale = nullptr) {
  const bool f8 = k_scale != nullptr;
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0) return RKV_OK;
  const bool app = k_new != nullptr;
  if (!q || !k || !v || !kt || !out) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: NULL tensor pointer");
  if ((k_new == nullptr) != (v_new == nullptr))
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode: k_new and v_new must both be set or both be NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(kt) || (app && (!aligned16(k_new) ||
                                                                                    !aligned16(v_new))))
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode: q/k/v/kt/k_new/v_new must be 16-byte aligned");
  if (mt && !idx) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt: idx is NULL");
  const int64_t n_tot = n + (app ? 1 : 0);
  if (n < 0 || n_tot < 1) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: no tokens to attend (n=%lld)", (long long)n);
  if (!mt && n_tot > cap)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode: %lld tokens > cap=%lld", (long long)n_tot, (long long)cap);
  if (mt && n_tot > idx_cap)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt: %lld candidates > idx_cap=%lld", (long long)n_tot,
                (long long)idx_cap);
  if (mt && app && (row < 0 || row >= cap))
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt: append row %lld outside [0, cap)", (long long)row);
  if (blk < 1 || blk > 128) return fail(RKV_ERR_UNSUPPORTED, "hsa_decode: block size %d outside [1,128]", blk);
  if (nblk_cap % 8 != 0) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: nblk_cap=%lld is not a multiple of 8",
                                     (long long)nblk_cap);
  const int64_t nblk = (n_tot + blk - 1) / blk;
  if (nblk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: ceil(n/blk)=%lld > nblk_cap=%lld",
                                   (long long)nblk, (long long)nblk_cap);
  if (nblk > 8192) return fail(RKV_ERR_UNSUPPORTED, "hsa_decode: %lld blocks > 8192", (long long)nblk);
  if (k1 < 1 || k1 > rkv::HD_HOST) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: k1=%d outside [1,128]", k1);
  if (k2 < 1) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: k2=%d < 1", k2);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "hsa_decode: bad scale");
  if (cap >= (int64_t)1 << 31) return fail(RKV_ERR_UNSUPPORTED, "hsa_decode: cap >= 2^31");

  rkv::HsaArgs a = {};
  a.q = q; a.k = k; a.v = v; a.kt = kt; a.idx = idx; a.idx_w = idx; a.out = out;
  a.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
  a.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
  a.row = mt ? row : n;
  a.sel_blocks = sel_blocks; a.sel_channels = sel_channels;
  a.cap = cap; a.nblk_cap = nblk_cap; a.idx_cap = idx_cap;
  a.n = (int32_t)n; a.n_rows = n_rows; a.B = d.batch;
  a.block_table = block_table; a.bt_stride = bt_stride; a.num_pages = num_pages; a.Hq = d.n_q_heads; a.Hkv = d.n_kv_heads; a.G = d.n_q_heads / d.n_kv_heads;
  a.mask = mask; a.mask_ld = mask_ld; a.n_prompt = n_prompt;
  a.k_scale = k_scale; a.v_scale = v_scale; a.f8 = f8 ? 1 : 0;
  a.blk = blk; a.k1 = k1; a.k2 = k2;
  a.scale_log2 = scale * 1.4426950408889634f;
  {
    const uint64_t w = g_test_wait_ns.load(std::memory_order_relaxed);
    a.wait_ns = w ? w : rkv::WAIT_LIMIT_NS_HOST;
    a.sbar_extra_tx = g_test_extra_tx.load(std::memory_order_relaxed);
  }
  a.tma_kv = (!mt && blk % 8 == 0) ? 1 : 0;
  if (!rkv::hsa_plan(a)) return fail(RKV_ERR_UNSUPPORTED, "hsa_decode: shared memory plan does not fit");

  CUtensorMap tmK, tmV, tmKT;
  std::memset(&tmK, 0, sizeof(tmK));
  std::memset(&tmV, 0, sizeof(tmV));
  std::memset(&tmKT, 0, sizeof(tmKT));
  const int64_t pairs = (int64_t)d.batch * d.n_kv_heads;
  if (f8) {
    if ((s = make_kv_map_u8(&tmK, k, pairs, cap, std::max<int64_t>(n, 1), blk, "k codes")) != RKV_OK) return s;
    if ((s = make_kv_map_u8(&tmV, v, pairs, cap, std::max<int64_t>(n, 1), blk, "v codes")) != RKV_OK) return s;
  } else if (a.tma_kv && block_table) {
    // one (page, KV head) slab of blk rows per box; the kernel masks rows past n
    const int64_t slabs = num_pages * d.n_kv_heads;
    if ((s = make_kv_map(&tmK, k, slabs, blk, blk, blk, "k pages")) != RKV_OK) return s;
    if ((s = make_kv_map(&tmV, v, slabs, blk, blk, blk, "v pages")) != RKV_OK) return s;
  } else if (a.tma_kv) {
    // rows at or past n (the appended token included) read as zero; with
    // per-row lengths every row up to cap is readable and the kernel masks
    const int64_t extent = n_rows ? cap : std::max<int64_t>(n, 1);
    if ((s = make_kv_map(&tmK, k, pairs, cap, extent, blk, "k")) != RKV_OK) return s;
    if ((s = make_kv_map(&tmV, v, pairs, cap, extent, blk, "v")) != RKV_OK) return s;
  }
  if (a.kt_spec) {
    if ((s = make_kt_map(&tmKT, kt, pairs, nblk_cap, a.cpr, f8)) != RKV_OK) return s;
  }
  cudaError_t e = rkv::hsa_launch(a, &tmK, &tmV, &tmKT, mt, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "hsa_decode launch");
  return RKV_OK;
}

}  // namespace

void rkv::set_last_error(const char* msg) { g_last_error = msg; }

extern "C" {

const char* rkv_last_error(void) { return g_last_error.c_str(); }

int32_t rkv_abi_version(void) { return 1; }

rkv_status rkv_budget_split(int64_t S, int64_t t, int32_t blk, int32_t W, double r_override, double* r,
                            int64_t* B1, int32_t* k2) {
  if (!r || !B1 || !k2) return fail(RKV_ERR_INVALID_ARG, "budget_split: NULL output");
  if (S < 1 || t < 1 || blk < 1 || W < 0) return fail(RKV_ERR_INVALID_ARG, "budget_split: S, t, blk >= 1 and W >= 0");
  const double c = (double)S / (double)t;
  double rr;
  if (r_override >= 0.0) {
    rr = r_override;
  } else {
    rr = std::fmin(0.2 + 0.06 * std::log2(c), 0.8);
    rr = std::fmax(rr, 0.2);
  }
  int64_t b1 = (int64_t)std::floor((double)S * std::pow(c, -rr));
  const int64_t lo = std::min<int64_t>((int64_t)W + 1, S);
  b1 = std::max(lo, std::min(b1, S));
  *r = rr;
  *B1 = b1;
  *k2 = (int32_t)std::max<int64_t>(1, (t / 2) / blk);
  return RKV_OK;
}

size_t rkv_snap_evict_workspace(rkv_dims d, int64_t S, int32_t W) {
  if (check_dims(d) != RKV_OK || S < 1 || W < 1) return 0;
  const int64_t w = std::min<int64_t>(W, S);
  return rkv::snap_workspace_bytes(d.batch, d.n_q_heads, d.n_kv_heads, S, (int32_t)w);
}

}  // extern "C"

namespace {

// Stage 1 for both entry points: S / B1 are the call's lengths, or with
// per-row arrays their maxima.
rkv_status snap_common(const char* who, rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v,
                       int64_t cap, int64_t S, int32_t pool_kernel, int32_t n_sink, int64_t B1, float scale,
                       int32_t* keep_idx, int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap, float* pooled_out,
                       void* ws, size_t ws_bytes, void* stream, const int32_t* S_rows, const int32_t* B1_rows,
                       bool per_row, const int32_t* bt = nullptr, int64_t bt_stride = 0, int64_t num_pages = 0,
                       int32_t page = 0) {
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0) return RKV_OK;
  const bool ragged = per_row;
  if (!q_obs || !k || !keep_idx) return fail(RKV_ERR_INVALID_ARG, "%s: NULL q_obs, k or keep_idx", who);
  if ((k_out == nullptr) != (v_out == nullptr))
    return fail(RKV_ERR_INVALID_ARG, "%s: k_out and v_out must both be set or both be NULL", who);
  if (k_out && !v) return fail(RKV_ERR_INVALID_ARG, "%s: v is NULL but compaction was requested", who);
  if (!aligned16(q_obs) || !aligned16(k) || (v && !aligned16(v)) || (k_out && (!aligned16(k_out) || !aligned16(v_out))))
    return fail(RKV_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", who);
  if ((reinterpret_cast<uintptr_t>(S_rows) & 3u) || (reinterpret_cast<uintptr_t>(B1_rows) & 3u) ||
      (reinterpret_cast<uintptr_t>(bt) & 3u))
    return fail(RKV_ERR_INVALID_ARG, "%s: S_rows, B1_rows and block_table must be 4-byte aligned", who);
  int32_t page_shift = 0;
  if (bt) {
    if (page < 8 || page > 128 || (page & (page - 1)) != 0)
      return fail(RKV_ERR_UNSUPPORTED, "%s: page of %d rows (a power of two in [8, 128] is required)", who, page);
    page_shift = __builtin_ctz((unsigned)page);
    if (num_pages < 1 || num_pages * d.n_kv_heads >= ((int64_t)1 << 31))
      return fail(RKV_ERR_INVALID_ARG, "%s: num_pages=%lld out of range", who, (long long)num_pages);
    if (bt_stride * page < S)
      return fail(RKV_ERR_INVALID_ARG, "%s: bt_stride=%lld pages cover fewer than S_max=%lld rows", who,
                  (long long)bt_stride, (long long)S);
    cap = bt_stride * page;       // rows a batch row's pages cover
  }
  if (W < 1) return fail(RKV_ERR_INVALID_ARG, "%s: W=%d < 1", who, W);
  if (S < 1 || S > cap) return fail(RKV_ERR_INVALID_ARG, "%s: S=%lld outside [1, cap=%lld]", who, (long long)S,
                                    (long long)cap);
  if (ragged && B1 > S) B1 = S;       // (a keep count past the longest prompt keeps it whole)
  if (cap >= (int64_t)1 << 31) return fail(RKV_ERR_UNSUPPORTED, "%s: cap >= 2^31", who);
  if (pool_kernel < 1 || pool_kernel % 2 == 0 || pool_kernel > 1025)
    return fail(RKV_ERR_INVALID_ARG, "%s: pool kernel %d must be odd in [1, 1025]", who, pool_kernel);
  if (n_sink < 0) return fail(RKV_ERR_INVALID_ARG, "%s: n_sink < 0", who);
  const int64_t w = ragged ? W : std::min<int64_t>(W, S);
  const int64_t L = std::max<int64_t>(S - w, 0);
  const int64_t sinks = std::min<int64_t>(n_sink, L);
  const bool keep_all = !ragged && (B1 >= S || L <= 0);
  if (ragged) {
    // every row's window and sinks must fit the longest keep list
    if (B1 < 1 || B1 < std::min<int64_t>(S, (int64_t)W + n_sink + 1))
      return fail(RKV_ERR_INVALID_ARG, "%s: B1_max=%lld < min(S_max, W + n_sink + 1)", who, (long long)B1);
  } else {
    if (keep_all && B1 != S)
      return fail(RKV_ERR_INVALID_ARG, "%s: B1=%lld must equal S=%lld when nothing is evicted", who, (long long)B1,
                  (long long)S);
    if (!keep_all && B1 < w + sinks)
      return fail(RKV_ERR_INVALID_ARG, "%s: B1=%lld < window %lld + sinks %lld", who, (long long)B1, (long long)w,
                  (long long)sinks);
  }
  if (keep_ld < B1) return fail(RKV_ERR_INVALID_ARG, "%s: keep_ld=%lld < B1", who, (long long)keep_ld);
  if (k_out && out_cap < B1) return fail(RKV_ERR_INVALID_ARG, "%s: out_cap=%lld < B1", who, (long long)out_cap);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(RKV_ERR_INVALID_ARG, "%s: bad scale", who);
  const bool scored = !keep_all && L > 0;
  const size_t need = rkv::snap_workspace_bytes(d.batch, d.n_q_heads, d.n_kv_heads, S, (int32_t)w);
  if (scored && (ws == nullptr || ws_bytes < need))
    return fail(RKV_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu required", who, ws_bytes, need);
  if (scored && (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(RKV_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  {
    // (v is read only when the call compacts)
    const void* ptrs[11] = {q_obs, k, k_out ? v : nullptr, keep_idx, k_out, v_out, pooled_out,
                            scored ? ws : nullptr, S_rows, B1_rows, bt};
    const char* names[11] = {"q_obs", "k", "v", "keep_idx", "k_out", "v_out", "pooled_out", "ws", "S_rows",
                             "B1_rows", "block_table"};
    for (int i = 0; i < 11; ++i)
      if (ptrs[i] && (s = require_device(ptrs[i], names[i])) != RKV_OK) return s;
  }

  rkv::SnapArgs a = {};
  a.q_obs = q_obs; a.k = k; a.v = v; a.cap = cap; a.S = S; a.out_cap = out_cap; a.B1 = B1;
  a.B = d.batch; a.Hq = d.n_q_heads; a.Hkv = d.n_kv_heads; a.G = d.n_q_heads / d.n_kv_heads;
  a.W = ragged ? W : (int32_t)w; a.pool = pool_kernel; a.n_sink = ragged ? n_sink : (int32_t)sinks;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.keep = keep_idx; a.keep_ld = keep_ld; a.k_out = k_out; a.v_out = v_out; a.pooled_out = pooled_out;
  a.S_rows = S_rows; a.B1_rows = B1_rows;
  a.bt = bt; a.bt_stride = bt_stride; a.num_pages = num_pages; a.page_shift = page_shift;
  a.ws = ws; a.ws_bytes = ws_bytes;
  CUtensorMap tmK, tmQ1, tmQ2;
  std::memset(&tmK, 0, sizeof(tmK));
  std::memset(&tmQ1, 0, sizeof(tmQ1));
  std::memset(&tmQ2, 0, sizeof(tmQ2));
  if (scored) {
    const int64_t qrows = (int64_t)d.batch * d.n_q_heads * W;
    if (bt) {
      // one (page, KV head) slab of `page` rows per box
      if ((s = make_kv_map(&tmK, k, num_pages * d.n_kv_heads, page, page, page, "k pages")) != RKV_OK) return s;
    } else if ((s = make_kv_map(&tmK, k, (int64_t)d.batch * d.n_kv_heads, cap, S, 128, "k")) != RKV_OK) {
      return s;
    }
    if ((s = make_q_map(&tmQ1, q_obs, qrows, rkv::snap_pass1_rows(d.n_q_heads / d.n_kv_heads, (int32_t)w))) !=
        RKV_OK)
      return s;
    if ((s = make_q_map(&tmQ2, q_obs, qrows, rkv::snap_pass2_rows(d.n_q_heads / d.n_kv_heads, (int32_t)w))) !=
        RKV_OK)
      return s;
  }
  cudaError_t e = rkv::snap_launch(a, &tmK, &tmQ1, &tmQ2, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "snap_evict launch");
  return RKV_OK;
}

}  // namespace

extern "C" {

rkv_status rkv_snap_evict(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v, int64_t cap,
                          int64_t S, int32_t pool_kernel, int32_t n_sink, int64_t B1, float scale, int32_t* keep_idx,
                          int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap, float* pooled_out, void* ws,
                          size_t ws_bytes, void* stream) {
  TraceRange trace("rkv_snap_evict");
  return snap_common("snap_evict", d, q_obs, W, k, v, cap, S, pool_kernel, n_sink, B1, scale, keep_idx, keep_ld, k_out,
                     v_out, out_cap, pooled_out, ws, ws_bytes, stream, nullptr, nullptr, false);
}

rkv_status rkv_snap_evict_ragged(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v, int64_t cap,
                                 const int32_t* S_rows, int64_t S_max, int32_t pool_kernel, int32_t n_sink,
                                 const int32_t* B1_rows, int64_t B1_max, float scale, int32_t* keep_idx,
                                 int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap, float* pooled_out,
                                 void* ws, size_t ws_bytes, void* stream) {
  TraceRange trace("rkv_snap_evict_ragged");
  if (d.batch > 0 && (!S_rows || !B1_rows))
    return fail(RKV_ERR_INVALID_ARG, "snap_evict_ragged: S_rows and B1_rows are required");
  return snap_common("snap_evict_ragged", d, q_obs, W, k, v, cap, S_max, pool_kernel, n_sink, B1_max, scale, keep_idx,
                     keep_ld, k_out, v_out, out_cap, pooled_out, ws, ws_bytes, stream, S_rows, B1_rows, true);
}

rkv_status rkv_snap_evict_paged(rkv_dims d, const void* q_obs, int32_t W, const void* k_pages, const void* v_pages,
                                int64_t num_pages, int32_t page, const int32_t* block_table, int64_t bt_stride,
                                const int32_t* S_rows, int64_t S_max, int32_t pool_kernel, int32_t n_sink,
                                const int32_t* B1_rows, int64_t B1_max, float scale, int32_t* keep_idx,
                                int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap, float* pooled_out,
                                void* ws, size_t ws_bytes, void* stream) {
  TraceRange trace("rkv_snap_evict_paged");
  if (d.batch > 0 && !block_table) return fail(RKV_ERR_INVALID_ARG, "snap_evict_paged: block_table is NULL");
  return snap_common("snap_evict_paged", d, q_obs, W, k_pages, v_pages, 0, S_max, pool_kernel, n_sink, B1_max, scale,
                     keep_idx, keep_ld, k_out, v_out, out_cap, pooled_out, ws, ws_bytes, stream, S_rows, B1_rows,
                     true, block_table, bt_stride, num_pages, page);
}

rkv_status rkv_build_kt(rkv_dims d, const void* k, int64_t cap, int64_t n, const int32_t* idx, int64_t idx_cap,
                        int32_t blk, void* kt, int64_t nblk_cap, void* stream) {
  TraceRange trace("rkv_build_kt");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || n == 0) return RKV_OK;
  if (!k || !kt) return fail(RKV_ERR_INVALID_ARG, "build_kt: NULL k or kt");
  if (!aligned16(k)) return fail(RKV_ERR_INVALID_ARG, "build_kt: k must be 16-byte aligned");
  if (blk < 1) return fail(RKV_ERR_INVALID_ARG, "build_kt: blk < 1");
  if (n < 0 || (!idx && n > cap) || (idx && n > idx_cap))
    return fail(RKV_ERR_INVALID_ARG, "build_kt: n=%lld out of range", (long long)n);
  if ((n + blk - 1) / blk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "build_kt: nblk_cap too small");
  cudaError_t e = rkv::kt_build_launch(k, cap, n, idx, idx_cap, blk, kt, nblk_cap, d.batch * d.n_kv_heads,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "build_kt launch");
  return RKV_OK;
}

rkv_status rkv_keep_mask(rkv_dims d, const int32_t* keep_idx, int64_t keep_ld, int64_t B1, int64_t n_prompt,
                         uint32_t* mask, int64_t mask_ld, void* stream) {
  TraceRange trace("rkv_keep_mask");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || n_prompt == 0) return RKV_OK;
  if (!keep_idx || !mask) return fail(RKV_ERR_INVALID_ARG, "keep_mask: NULL keep_idx or mask");
  if (reinterpret_cast<uintptr_t>(mask) % 4 != 0 || reinterpret_cast<uintptr_t>(keep_idx) % 4 != 0)
    return fail(RKV_ERR_INVALID_ARG, "keep_mask: keep_idx and mask must be 4-byte aligned");
  if (n_prompt < 0 || B1 < 0 || keep_ld < B1)
    return fail(RKV_ERR_INVALID_ARG, "keep_mask: need n_prompt >= 0 and 0 <= B1 <= keep_ld");
  if (mask_ld < (n_prompt + 31) / 32)
    return fail(RKV_ERR_INVALID_ARG, "keep_mask: mask_ld=%lld < ceil(n_prompt/32)", (long long)mask_ld);
  cudaError_t e = rkv::keep_mask_launch(keep_idx, keep_ld, B1, n_prompt, mask, mask_ld, d.batch * d.n_kv_heads,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "keep_mask launch");
  return RKV_OK;
}

rkv_status rkv_build_kt_masked(rkv_dims d, const void* k, int64_t cap, int64_t n, const uint32_t* mask,
                               int64_t mask_ld, int64_t n_prompt, int32_t blk, void* kt, int64_t nblk_cap,
                               void* stream) {
  TraceRange trace("rkv_build_kt_masked");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || n == 0) return RKV_OK;
  if (!k || !kt || !mask) return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: NULL k, kt or mask");
  if (!aligned16(k)) return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: k must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(mask) % 4 != 0)
    return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: mask must be 4-byte aligned");
  if (blk < 1) return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: blk < 1");
  if (n < 0 || n > cap) return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: n=%lld out of range", (long long)n);
  if (n_prompt < 0 || n_prompt > n)
    return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: n_prompt=%lld outside [0, n]", (long long)n_prompt);
  if (mask_ld < (n_prompt + 31) / 32)
    return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: mask_ld=%lld < ceil(n_prompt/32)", (long long)mask_ld);
  if ((n + blk - 1) / blk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "build_kt_masked: nblk_cap too small");
  cudaError_t e = rkv::kt_build_launch(k, cap, n, nullptr, 0, blk, kt, nblk_cap, d.batch * d.n_kv_heads,
                                       reinterpret_cast<cudaStream_t>(stream), mask, mask_ld, n_prompt);
  if (e != cudaSuccess) return cuda_fail(e, "build_kt_masked launch");
  return RKV_OK;
}

rkv_status rkv_compact_kt(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                          int64_t keep_ld, int64_t B1, void* k_out, void* v_out, int64_t out_cap, int32_t blk, void* kt,
                          int64_t nblk_cap, void* stream) {
  TraceRange trace("rkv_compact_kt");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || B1 == 0) return RKV_OK;
  if (!k || !v || !keep_idx || !k_out || !v_out || !kt) return fail(RKV_ERR_INVALID_ARG, "compact_kt: NULL pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out) || !aligned16(kt))
    return fail(RKV_ERR_INVALID_ARG, "compact_kt: k, v, k_out, v_out and kt must be 16-byte aligned");
  if (cap < 1 || B1 < 0 || B1 > out_cap || keep_ld < B1)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt: need cap >= 1, 0 <= B1 <= out_cap and keep_ld >= B1");
  if (blk < 1) return fail(RKV_ERR_INVALID_ARG, "compact_kt: blk < 1");
  if (nblk_cap % 8 != 0) return fail(RKV_ERR_INVALID_ARG, "compact_kt: nblk_cap=%lld is not a multiple of 8",
                                     (long long)nblk_cap);
  if ((B1 + blk - 1) / blk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "compact_kt: nblk_cap too small");
  if ((s = device_view(k, &k, "compact_kt: k")) != RKV_OK || (s = device_view(v, &v, "compact_kt: v")) != RKV_OK)
    return s;
  cudaError_t e = rkv::compact_kt_launch(k, v, cap, keep_idx, keep_ld, B1, blk, k_out, v_out, out_cap, kt, nblk_cap,
                                         d.batch * d.n_kv_heads, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "compact_kt launch");
  return RKV_OK;
}

rkv_status rkv_compact_kt_fp8(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                              int64_t keep_ld, int64_t B1, const float* k_scale, const float* v_scale, void* k_out,
                              void* v_out, int64_t out_cap, int32_t blk, void* kt, int64_t nblk_cap, void* stream) {
  TraceRange trace("rkv_compact_kt_fp8");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || B1 == 0) return RKV_OK;
  if (!k || !v || !keep_idx || !k_out || !v_out || !kt || !k_scale || !v_scale)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: NULL pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out) || !aligned16(kt))
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: k, v, k_out, v_out and kt must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(k_scale) % 4 != 0 || reinterpret_cast<uintptr_t>(v_scale) % 4 != 0)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: scales must be 4-byte aligned");
  if (cap < 1 || B1 < 0 || B1 > out_cap || keep_ld < B1)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: need cap >= 1, 0 <= B1 <= out_cap and keep_ld >= B1");
  if (blk < 1) return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: blk < 1");
  if (nblk_cap % 16 != 0)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: nblk_cap=%lld is not a multiple of 16", (long long)nblk_cap);
  if ((B1 + blk - 1) / blk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "compact_kt_fp8: nblk_cap too small");
  if ((s = device_view(k, &k, "compact_kt_fp8: k")) != RKV_OK || (s = device_view(v, &v, "compact_kt_fp8: v")) != RKV_OK)
    return s;
  cudaError_t e = rkv::compact_kt_fp8_launch(k, v, cap, keep_idx, keep_ld, B1, blk, k_scale, v_scale, k_out, v_out,
                                             out_cap, kt, nblk_cap, d.batch * d.n_kv_heads,
                                             reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "compact_kt_fp8 launch");
  return RKV_OK;
}

rkv_status rkv_compact_kt_paged(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                                int64_t keep_ld, int64_t B1, void* k_pages, void* v_pages, int64_t num_pages,
                                const int32_t* block_table, int64_t bt_stride, int32_t blk, void* kt,
                                int64_t nblk_cap, void* stream) {
  TraceRange trace("rkv_compact_kt_paged");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0 || B1 == 0) return RKV_OK;
  if (!k || !v || !keep_idx || !k_pages || !v_pages || !block_table || !kt)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: NULL pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(kt))
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: k, v, k_pages, v_pages and kt must be 16-byte aligned");
  if (cap < 1 || B1 < 0 || keep_ld < B1)
    return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: need cap >= 1, B1 >= 0 and keep_ld >= B1");
  if (blk < 1) return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: blk < 1");
  const int64_t nblk = (B1 + blk - 1) / blk;
  if (bt_stride < nblk) return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: bt_stride < ceil(B1/blk)");
  if (num_pages < 1) return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: num_pages < 1");
  if (nblk_cap % 8 != 0) return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: nblk_cap=%lld is not a multiple of 8",
                                     (long long)nblk_cap);
  if (nblk > nblk_cap) return fail(RKV_ERR_INVALID_ARG, "compact_kt_paged: nblk_cap too small");
  if ((s = device_view(k, &k, "compact_kt_paged: k")) != RKV_OK ||
      (s = device_view(v, &v, "compact_kt_paged: v")) != RKV_OK)
    return s;
  cudaError_t e = rkv::compact_kt_launch(k, v, cap, keep_idx, keep_ld, B1, blk, k_pages, v_pages, 0, kt, nblk_cap,
                                         d.batch * d.n_kv_heads, reinterpret_cast<cudaStream_t>(stream), block_table,
                                         bt_stride, num_pages, d.n_kv_heads);
  if (e != cudaSuccess) return cuda_fail(e, "compact_kt_paged launch");
  return RKV_OK;
}

rkv_status rkv_append_kv(rkv_dims d, const void* k_new, const void* v_new, void* k, void* v, int64_t cap, int64_t n,
                         int64_t row, int32_t* idx, int64_t idx_cap, void* kt, int64_t nblk_cap, int32_t blk,
                         void* stream) {
  TraceRange trace("rkv_append_kv");
  rkv_status s = check_dims(d);
  if (s != RKV_OK) return s;
  if (d.batch == 0) return RKV_OK;
  if (!k_new || !v_new || !k || !v || !kt) return fail(RKV_ERR_INVALID_ARG, "append_kv: NULL pointer");
  if (blk < 1 || n < 0 || row < 0 || row >= cap) return fail(RKV_ERR_INVALID_ARG, "append_kv: bad n/row/blk");
  if (!idx && row != n) return fail(RKV_ERR_INVALID_ARG, "append_kv: without idx the row must equal n");
  if (idx && n >= idx_cap) return fail(RKV_ERR_INVALID_ARG, "append_kv: n >= idx_cap");
  if (n / blk >= nblk_cap) return fail(RKV_ERR_INVALID_ARG, "append_kv: block %lld >= nblk_cap", (long long)(n / blk));
  cudaError_t e = rkv::append_launch(k_new, v_new, k, v, cap, n, row, idx, idx_cap, kt, nblk_cap, blk,
                                     d.batch * d.n_kv_heads, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append_kv launch");
  return RKV_OK;
}

rkv_status rkv_hsa_decode(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n, void* kt,
                          int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale, float* out,
                          int32_t* sel_blocks, int32_t* sel_channels, const void* k_new, const void* v_new,
                          void* stream) {
  TraceRange trace("rkv_hsa_decode");
  return hsa_common(d, q, k, v, cap, nullptr, 0, n, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks, sel_channels,
                    k_new, v_new, n, stream, false);
}

rkv_status rkv_hsa_decode_mt(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int32_t* idx, int64_t idx_cap,
                             int64_t n, void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale,
                             float* out, int32_t* sel_blocks, int32_t* sel_channels, const void* k_new,
                             const void* v_new, int64_t row, void* stream) {
  TraceRange trace("rkv_hsa_decode_mt");
  return hsa_common(d, q, k, v, cap, idx, idx_cap, n, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks,
                    sel_channels, k_new, v_new, row, stream, true);
}

rkv_status rkv_hsa_decode_mt_masked(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n,
                                    const uint32_t* mask, int64_t mask_ld, int64_t n_prompt, void* kt,
                                    int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale, float* out,
                                    int32_t* sel_blocks, int32_t* sel_channels, const void* k_new, const void* v_new,
                                    void* stream) {
  TraceRange trace("rkv_hsa_decode_mt_masked");
  if (!mask) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt_masked: mask is NULL");
  if (reinterpret_cast<uintptr_t>(mask) % 4 != 0)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt_masked: mask must be 4-byte aligned");
  if (n_prompt < 0 || n_prompt > n || n_prompt > cap)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt_masked: n_prompt=%lld outside [0, min(n, cap)]",
                (long long)n_prompt);
  if (mask_ld < (n_prompt + 31) / 32)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_mt_masked: mask_ld=%lld < ceil(n_prompt/32)", (long long)mask_ld);
  return hsa_common(d, q, k, v, cap, nullptr, 0, n, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks, sel_channels,
                    k_new, v_new, n, stream, false, nullptr, nullptr, 0, 0, mask, mask_ld, n_prompt);
}

rkv_status rkv_hsa_decode_fp8(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n,
                              const float* k_scale, const float* v_scale, void* kt, int64_t nblk_cap, int32_t blk,
                              int32_t k1, int32_t k2, float scale, float* out, int32_t* sel_blocks,
                              int32_t* sel_channels, const void* k_new, const void* v_new, void* stream) {
  TraceRange trace("rkv_hsa_decode_fp8");
  if (!k_scale || !v_scale) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_fp8: NULL k_scale or v_scale");
  if (reinterpret_cast<uintptr_t>(k_scale) % 4 != 0 || reinterpret_cast<uintptr_t>(v_scale) % 4 != 0)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_fp8: scales must be 4-byte aligned");
  if (blk % 8 != 0) return fail(RKV_ERR_UNSUPPORTED, "hsa_decode_fp8: block size %d is not a multiple of 8", blk);
  if (nblk_cap % 16 != 0)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_fp8: nblk_cap=%lld is not a multiple of 16", (long long)nblk_cap);
  return hsa_common(d, q, k, v, cap, nullptr, 0, n, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks, sel_channels,
                    k_new, v_new, n, stream, false, nullptr, nullptr, 0, 0, nullptr, 0, 0, k_scale, v_scale);
}

rkv_status rkv_hsa_decode_ragged(rkv_dims d, const void* q, void* k, void* v, int64_t cap, const int32_t* n_rows,
                                 int64_t n_max, void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2,
                                 float scale, float* out, int32_t* sel_blocks, int32_t* sel_channels,
                                 const void* k_new, const void* v_new, void* stream) {
  TraceRange trace("rkv_hsa_decode_ragged");
  if (d.batch > 0 && !n_rows) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_ragged: n_rows is NULL");
  if (n_max < 1) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_ragged: n_max=%lld < 1", (long long)n_max);
  return hsa_common(d, q, k, v, cap, nullptr, 0, n_max, kt, nblk_cap, blk, k1, k2, scale, out, sel_blocks,
                    sel_channels, k_new, v_new, 0, stream, false, n_rows);
}

rkv_status rkv_hsa_decode_paged(rkv_dims d, const void* q, void* k_pages, void* v_pages, int64_t num_pages,
                                const int32_t* block_table, int64_t bt_stride, const int32_t* n_rows, int64_t n_max,
                                void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale,
                                float* out, int32_t* sel_blocks, int32_t* sel_channels, const void* k_new,
                                const void* v_new, void* stream) {
  TraceRange trace("rkv_hsa_decode_paged");
  if (d.batch > 0 && !block_table) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_paged: block_table is NULL");
  if (n_max < 1) return fail(RKV_ERR_INVALID_ARG, "hsa_decode_paged: n_max=%lld < 1", (long long)n_max);
  if (num_pages < 1 || num_pages * (int64_t)d.n_kv_heads * blk >= ((int64_t)1 << 31))
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_paged: num_pages=%lld outside [1, 2^31 / (Hkv * blk))",
                (long long)num_pages);
  if (blk < 1 || bt_stride < 1 || bt_stride > ((int64_t)1 << 31) / blk)
    return fail(RKV_ERR_INVALID_ARG, "hsa_decode_paged: bt_stride=%lld, blk=%d", (long long)bt_stride, blk);
  // a row's logical capacity is bt_stride pages of blk rows
  return hsa_common(d, q, k_pages, v_pages, bt_stride * blk, nullptr, 0, n_max, kt, nblk_cap, blk, k1, k2, scale,
                    out, sel_blocks, sel_channels, k_new, v_new, 0, stream, false, n_rows, block_table, bt_stride,
                    num_pages);
}

rkv_status rkv_debug_set_wait(uint64_t limit_ns, uint32_t extra_bytes) {
  if (extra_bytes > 4096) return fail(RKV_ERR_INVALID_ARG, "debug_set_wait: extra_bytes above 4096");
  if (limit_ns != 0 && limit_ns < 1000)
    return fail(RKV_ERR_INVALID_ARG, "debug_set_wait: limit below 1 us");
  g_test_wait_ns.store(limit_ns, std::memory_order_relaxed);
  g_test_extra_tx.store(extra_bytes, std::memory_order_relaxed);
  return RKV_OK;
}

rkv_status rkv_read_device_flags(uint32_t* flags) {
  TraceRange trace("rkv_read_device_flags");
  if (!flags) return fail(RKV_ERR_INVALID_ARG, "read_device_flags: NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "read_device_flags");
  *flags = rkv::hsa_take_device_error() | rkv::snap_take_device_error();
  if (*flags)
    return fail(RKV_ERR_TIMEOUT, "device flags 0x%x (bit 0: a bounded wait gave up, bit 1: a per-row length was "
                "out of range)", *flags);
  return RKV_OK;
}

}  // extern "C"
