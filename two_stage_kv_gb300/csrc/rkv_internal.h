// Internal launch interfaces between the C-ABI layer (rkv_api.cu) and the
// kernel translation units.  Host-side only; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rkv {

constexpr int HD_HOST = 128;   // head dimension of the implemented path
constexpr uint64_t WAIT_LIMIT_NS_HOST = 1000000000ull;   // limit of a bounded device wait (1 s)

// ------------------------------------------------------------ HSA decode ---
struct HsaArgs {
  const void* q;        // [B, Hq, D] bf16
  void* k;              // [B, Hkv, cap, D] bf16 (written only by a fused append)
  void* v;
  void* kt;             // [B, Hkv, 2, D, nblk_cap] bf16 (written only by a fused append)
  const int32_t* idx;   // MT candidate rows [B, Hkv, idx_cap] or nullptr
  int32_t* idx_w;       // same rows, written by a fused MT append
  const __nv_bfloat16* k_new;   // [B, Hkv, D] token appended by this step, or nullptr
  const __nv_bfloat16* v_new;
  int64_t row;          // cache row of the appended token (n without idx)
  float* out;           // [B, Hq, D] fp32
  int32_t* sel_blocks;  // [B, Hkv, k2] or nullptr
  int32_t* sel_channels;  // [B, Hkv, k1] or nullptr
  int64_t cap, nblk_cap, idx_cap;
  int32_t n, B, Hq, Hkv, G, blk, k1, k2;   // n = candidates before the append (ragged: the rows' maximum)
  const int32_t* n_rows; // ragged: [B] candidates before the append per batch row (device), else nullptr
  const int32_t* block_table;  // paged: [B, bt_stride] page of each logical block (device), else nullptr
  int64_t bt_stride, num_pages;  // paged: K/V pools are [num_pages, Hkv, blk, D]
  const uint32_t* mask;  // masked MT: [B, Hkv, mask_ld] bit r = prompt row r kept by stage 1, else nullptr
  int64_t mask_ld, n_prompt;     // rows >= n_prompt (decoded after the prompt) are always candidates
  const float* k_scale;  // e4m3 storage: [B, Hkv] value = code * scale for K and V (k, v, kt hold codes)
  const float* v_scale;
  int32_t f8;           // 1: k, v and kt hold e4m3 codes
  int32_t nblk;         // blocks over the attended candidates
  int32_t k2e;          // min(k2, nblk)
  int32_t ns;           // CTAs per cluster (one cluster per (b, kv head))
  int32_t chunk;        // selected blocks per CTA: ceil(k2e / ns)
  int32_t slots_round;  // blocks staged in shared memory per round
  int32_t kt_chunk;     // blocks per shared-memory KT gather (multiple of 8)
  int32_t cpr;          // blocks scored per CTA of the cluster (multiple of 8); CTA r scores [r*cpr, r*cpr + cpr)
  int32_t kt_spec;      // 1: each CTA prefetches all 2*D KT rows of its blocks with one TMA box at launch
  int32_t blk_shift;    // log2(blk) when blk is a power of two, else -1
  int32_t ns_shift;     // log2(ns) when ns is a power of two, else -1
  int32_t wflash;       // 1: per-warp online softmax (several staging rounds per CTA, narrow groups)
  int32_t tma_kv;       // 1: K/V block rows by TMA (blk a multiple of 8, no idx); 0: gathered rows
  float scale_log2;     // softmax scale * log2(e)
  uint64_t wait_ns;     // limit of each bounded wait (WAIT_LIMIT_NS unless shortened for a test)
  uint32_t sbar_extra_tx;   // test only: bytes the block-score barrier expects that no copy delivers
  // dynamic shared-memory layout (bytes)
  uint32_t off_x, off_scores, off_flags, off_sel, off_bt, off_recv, off_tiles, tile_half_bytes, smem_bytes;
};

// Computes ns/chunk/slots_round and the shared-memory layout.  Returns false if
// the configuration does not fit on the device.
bool hsa_plan(HsaArgs& a);
cudaError_t hsa_launch(const HsaArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmKT,
                       bool mt, cudaStream_t st);
constexpr int HSA_SPEC_MAX_COLS = 128;   // KT columns per CTA for the launch-time prefetch (256 rows x 128 x 2 B)

// ------------------------------------------------------------ stage 1 -------
struct SnapArgs {
  const void* q_obs;    // [B, Hq, W, D]
  const void* k;        // [B, Hkv, cap, D]
  const void* v;
  int64_t cap, S, out_cap, B1;
  int32_t B, Hq, Hkv, G, W, pool, n_sink;
  float scale_log2;
  int32_t* keep;        // [B, Hkv, keep_ld]
  int64_t keep_ld;
  void* k_out;          // [B, Hkv, out_cap, D] or nullptr (mask mode)
  void* v_out;
  float* pooled_out;    // [B, Hkv, S-W] or nullptr
  const int32_t* S_rows;    // [B] per-row prompt lengths (S is their maximum), or nullptr
  const int32_t* B1_rows;   // [B] per-row keep counts (B1 is their maximum), or nullptr
  const int32_t* bt;        // paged prompt cache: k, v are [num_pages, Hkv, page, D] pools and bt [B, bt_stride]
  int64_t bt_stride, num_pages;   // the page of each logical page of a row; nullptr = dense [B, Hkv, cap, D]
  int32_t page_shift;       // log2 of the rows per page
  // workspace carve-up
  void* ws;
  size_t ws_bytes;
};
size_t snap_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t S, int32_t W);
// Query rows per pass-2 CTA (the MMA N of the key-major pass) for a group of G*W rows.
int snap_pass2_rows(int32_t G, int32_t W);
int snap_pass1_rows(int32_t G, int32_t W);
cudaError_t snap_launch(const SnapArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmQ1, const CUtensorMap* tmQ2,
                        cudaStream_t st);

// ------------------------------------------------------------ KT / append ---
cudaError_t kt_build_launch(const void* k, int64_t cap, int64_t n, const int32_t* idx, int64_t idx_cap,
                            int32_t blk, void* kt, int64_t nblk_cap, int32_t pairs, cudaStream_t st,
                            const uint32_t* mask = nullptr, int64_t mask_ld = 0, int64_t n_prompt = 0);
cudaError_t compact_kt_fp8_launch(const void* k, const void* v, int64_t cap, const int32_t* keep, int64_t keep_ld,
                                  int64_t B1, int blk, const float* k_scale, const float* v_scale, void* ko, void* vo,
                                  int64_t out_cap, void* kt, int64_t nblk_cap, int pairs, cudaStream_t st);
cudaError_t keep_mask_launch(const int32_t* keep, int64_t keep_ld, int64_t B1, int64_t n_prompt, uint32_t* mask,
                             int64_t mask_ld, int32_t pairs, cudaStream_t st);
cudaError_t compact_kt_launch(const void* k, const void* v, int64_t cap, const int32_t* keep, int64_t keep_ld,
                              int64_t B1, int blk, void* ko, void* vo, int64_t out_cap, void* kt, int64_t nblk_cap,
                              int pairs, cudaStream_t st, const int32_t* bt = nullptr, int64_t bt_stride = 0,
                              int64_t num_pages = 0, int Hkv = 1);
cudaError_t append_launch(const void* k_new, const void* v_new, void* k, void* v, int64_t cap, int64_t n,
                          int64_t row, int32_t* idx, int64_t idx_cap, void* kt, int64_t nblk_cap, int32_t blk,
                          int32_t pairs, cudaStream_t st);

// Device error words of each translation unit (read and cleared).
unsigned int hsa_take_device_error();
unsigned int snap_take_device_error();

// Records the message returned by rkv_last_error() on this host thread.
void set_last_error(const char* msg);

}  // namespace rkv
