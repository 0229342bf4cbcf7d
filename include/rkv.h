/*
 * rkv.h -- C ABI of the GB300 (sm_103a) two-stage compressed decode library.
 *
 * The library implements the decode hot path of RocketKV ("RocketKV:
 * Accelerating Long-Context LLM Inference via Two-Stage KV Cache
 * Compression", papercache digest of arXiv:2502.14051, section 方法细节):
 *   stage 1  SnapKV eviction at the end of prefill (observation-window scores
 *            summed over the GQA group, 1-D max-pool, top-k, compaction);
 *   KT cache per-block elementwise Kmax / Kmin of the keys (HSA step 1);
 *   stage 2  Hybrid Sparse Attention per decode step (Algorithm 1: top-k1
 *            channels of sum|q|, sign-selected Kmax/Kmin block scores, top-k2
 *            blocks, exact attention over the selected blocks);
 *   MT       RocketKV-MT: the full cache is kept and stage 2 is restricted to
 *            the stage-1 survivors plus decoded tokens.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller.  The
 *     library never allocates or frees device memory and keeps no state
 *     between calls (apart from a per-library device error word, see
 *     rkv_read_device_flags).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Argument checks run on the host before any launch and
 *     their status is returned synchronously; a failed launch returns
 *     RKV_ERR_CUDA.  No C++ exception crosses the ABI.
 *   - bf16 tensors hold IEEE bfloat16; fp32 outputs are IEEE float.
 *   - Layouts are row-major with the last index fastest:
 *       K, V (caches)   [B, Hkv, cap, D]         bf16
 *       q (decode)      [B, Hq, D]               bf16
 *       q_obs (window)  [B, Hq, W, D]            bf16
 *       KT              [B, Hkv, 2, D, nblk_cap] bf16, index 0 = Kmax, 1 = Kmin
 *       idx (MT)        [B, Hkv, idx_cap]        int32 physical cache rows
 *     Query head h belongs to KV head h / (Hq / Hkv).
 *   - Supported on the GPU: head_dim == 128, 1 <= Hq/Hkv <= 16, block size a
 *     multiple of 8 in [8, 128].  Other shapes return RKV_ERR_UNSUPPORTED.
 *   - Thread safety: entry points may be called from several host threads;
 *     rkv_last_error() is per thread.
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RKV_OK = 0,
  RKV_ERR_INVALID_ARG = 1,   /* a pointer, size or stride is invalid */
  RKV_ERR_UNSUPPORTED = 2,   /* valid, but outside the shapes this library runs */
  RKV_ERR_WORKSPACE = 3,     /* workspace pointer NULL or smaller than required */
  RKV_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  RKV_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (device flag) */
} rkv_status;

typedef struct {
  int32_t batch;        /* B   */
  int32_t n_q_heads;    /* Hq  */
  int32_t n_kv_heads;   /* Hkv */
  int32_t head_dim;     /* D   */
} rkv_dims;

/* Message describing the last non-OK status returned on this host thread. */
const char* rkv_last_error(void);

/* Library ABI version (incremented when a signature changes). */
int32_t rkv_abi_version(void);

/*
 * Budget split.  [RocketKV digest, 方法细节: token budget definition; adaptive
 * split factor r = min(0.2 + 0.06*log2(c), 0.8) with r kept in [0.2, 0.8]]
 * c = S / t.  Stage 1 keeps B1 = floor(S / c^r) tokens, clamped to
 * [min(W+1, S), S].  The token budget t is split evenly between HSA steps 2
 * and 3, so step 3 reads k2 = max(1, floor((t/2)/blk)) blocks.
 * r_override >= 0 replaces the adaptive r (the static-split ablation).
 * Host only; no GPU work.  Output pointers must be non-NULL.
 */
rkv_status rkv_budget_split(int64_t S, int64_t t, int32_t blk, int32_t W, double r_override,
                            double* r, int64_t* B1, int32_t* k2);

/*
 * Workspace bytes needed by rkv_snap_evict for these dims, prompt length S and
 * window W (device memory, caller-allocated, 256-byte aligned).
 */
size_t rkv_snap_evict_workspace(rkv_dims d, int64_t S, int32_t W);

/*
 * Stage 1: SnapKV eviction.  [RocketKV digest, 方法细节: SnapKV in stage 1,
 * GQA group-level token selection, pooling kernel size 63]
 * For every (batch b, KV head h):
 *   score[j] = sum over the group's query heads g and window rows w of
 *              softmax_j(q_obs[b,g,w] . k[b,h,j] * scale), the softmax over
 *              keys 0 .. S-W+w (causal), for prefix keys j < S-W;
 *   pooled   = max-pool(score, kernel pool_kernel, stride 1, clipped ends);
 *   keep     = [0, n_sink) + top-(B1-W-n_sink) of pooled over [n_sink, S-W)
 *              (larger first, equal values: lower index first) + [S-W, S),
 *              sorted ascending, B1 entries.
 * If B1 >= S every token is kept.
 * Arguments
 *   q_obs      [B, Hq, W, D] bf16, window queries (the last W prompt tokens).
 *   k, v       [B, Hkv, cap, D] bf16 prompt caches; rows [0, S) are read.
 *   keep_idx   [B, Hkv, keep_ld] int32 output; entries [0, B1) of each row are
 *              written (keep_ld >= B1; MT callers point it at their idx rows).
 *   k_out,v_out[B, Hkv, out_cap, D] bf16 compacted caches (rows [0, B1)
 *              written).  Both NULL = MT mask mode: only keep_idx is written.
 *   pooled_out optional [B, Hkv, S-W] fp32 pooled scores (NULL = skip); the
 *              ranking itself uses log2 of the scores, so scores below the
 *              fp32 range (written here as 0) still rank exactly.
 *   ws         workspace of rkv_snap_evict_workspace() bytes.
 * k/v and k_out/v_out must not overlap.
 * Errors: RKV_ERR_INVALID_ARG for NULL or misaligned pointers, a pointer that
 * is not device memory (q_obs, k, keep_idx, ws, the outputs, and v when the
 * call compacts) and the size rules above; RKV_ERR_WORKSPACE for a missing or
 * short workspace; RKV_ERR_CUDA if a launch fails.
 */
rkv_status rkv_snap_evict(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v,
                          int64_t cap, int64_t S, int32_t pool_kernel, int32_t n_sink, int64_t B1,
                          float scale, int32_t* keep_idx, int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap,
                          float* pooled_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 1 for a batch whose rows hold prompts of different lengths, each with
 * its own keep count (ragged batch).  [RocketKV digest, 方法细节: SnapKV in
 * stage 1, GQA group-level token selection, pooling kernel size 63, per
 * request]  Same computation, arguments and results as rkv_snap_evict for
 * every batch row b on its own prompt of S_b tokens and keep count B1_b:
 * window = the row's last W tokens (q_obs[b] holds their queries), prefix
 * [0, S_b - W), keep[b, h, 0:B1_b] ascending, compacted rows [0, B1_b).  A row
 * with S_b <= W, or B1_b >= S_b, keeps all its S_b tokens.
 *   S_rows   [B] int32 DEVICE array of prompt lengths; S_max >= every entry
 *            sizes the launch (entries are clamped into [1, S_max]).
 *   B1_rows  [B] int32 DEVICE array of keep counts; B1_max >= every entry
 *            (entries are clamped into [min(W + sinks, hi), hi] with hi =
 *            min(S_b, B1_max)); B1_max >= min(S_max, W + n_sink + 1).
 *   k, v     [B, Hkv, cap, D] with S_max <= cap; row b's tokens are rows [0, S_b).
 *   pooled_out optional [B, Hkv, S_max - W] fp32: entries [0, S_b - W) of row b
 *            (not written for a row that keeps all its tokens).
 *   ws       rkv_snap_evict_workspace(d, S_max, W) bytes.
 * keep_ld and out_cap bound B1_max as in rkv_snap_evict; entries of keep and
 * of the compacted caches past a row's B1_b are not written.  A clamped
 * length or keep count sets bit 1 of the device error word.
 */
rkv_status rkv_snap_evict_ragged(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v,
                                 int64_t cap, const int32_t* S_rows, int64_t S_max, int32_t pool_kernel,
                                 int32_t n_sink, const int32_t* B1_rows, int64_t B1_max, float scale,
                                 int32_t* keep_idx, int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap,
                                 float* pooled_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Stage 1 over a paged prompt cache.  [RocketKV digest, 方法细节: SnapKV in
 * stage 1, per request, over a cache held in pages]  Same computation and
 * results as rkv_snap_evict_ragged, with each batch row's prompt K/V rows held
 * in pages of `page` rows shared by the whole batch:
 *   k_pages,v_pages [num_pages, Hkv, page, D] bf16 (16-byte aligned);
 *   block_table     [B, bt_stride] int32 DEVICE array: prompt rows
 *                   j*page .. j*page + page-1 of batch row b (every KV head)
 *                   are page block_table[b, j]; bt_stride * page >= S_max;
 *                   page ids are clamped into [0, num_pages) and a clamped id
 *                   sets bit 1 of the device error word;
 *   page            rows per page: a power of two in [8, 128];
 *   S_rows, B1_rows per-row prompt lengths and keep counts as in
 *                   rkv_snap_evict_ragged, or NULL: every row has S_max / B1_max.
 * The compacted caches k_out / v_out (when set) are dense [B, Hkv, out_cap, D]:
 * rkv_compact_kt_paged can move them into pages of the decode pool.
 */
rkv_status rkv_snap_evict_paged(rkv_dims d, const void* q_obs, int32_t W, const void* k_pages, const void* v_pages,
                                int64_t num_pages, int32_t page, const int32_t* block_table, int64_t bt_stride,
                                const int32_t* S_rows, int64_t S_max, int32_t pool_kernel, int32_t n_sink,
                                const int32_t* B1_rows, int64_t B1_max, float scale, int32_t* keep_idx,
                                int64_t keep_ld, void* k_out, void* v_out, int64_t out_cap, float* pooled_out,
                                void* ws, size_t ws_bytes, void* stream);

/*
 * Stage-1 eviction for callers that cannot allocate device memory.  The
 * paper has no counterpart to this entry point; it exists for serving
 * engines whose memory pool owns all device memory and for plugin hooks that
 * run inside another framework's step, where a cudaMalloc can fail or
 * synchronise the device.
 * Same operation, arguments and results as rkv_snap_evict, minus ws/ws_bytes:
 * the scratch is a fixed 32 MiB array of device memory inside this library,
 * held on every GPU that loads the library's device code until the process
 * exits.  Shapes whose rkv_snap_evict_workspace() exceeds 32 MiB return
 * RKV_ERR_WORKSPACE with a message giving both sizes.  It calls no cudaMalloc
 * or cudaFree.  The first call on a device, made with that device current,
 * looks up the array's device address (cudaGetSymbolAddress); make that first
 * call before any stream capture.  Devices 0-63 are served (others get
 * RKV_ERR_UNSUPPORTED).  Each device has its own copy of the array, so calls
 * on different devices are independent; every call on one device uses that
 * device's copy, so calls on one device that can overlap (different streams,
 * or several host threads) race, and the caller must serialise them.  No
 * part of the scratch needs to start at zero: each call writes all it reads.
 */
rkv_status rkv_snap_evict_noalloc(rkv_dims d, const void* q_obs, int32_t W, const void* k, const void* v,
                                  int64_t cap, int64_t S, int32_t pool_kernel, int32_t n_sink, int64_t B1,
                                  float scale, int32_t* keep_idx, int64_t keep_ld, void* k_out, void* v_out,
                                  int64_t out_cap, float* pooled_out, void* stream);

/*
 * Stage-1 compaction with the KT cache built on the way.  [RocketKV digest,
 * 方法细节: stage 1 permanently drops the evicted tokens; HSA step 1 keeps
 * per-page elementwise Kmax / Kmin of the keys]
 * For every (batch b, KV head h) and i < B1:
 *   k_out[b,h,i] = k[b,h,keep_idx[b,h,i]],  v_out[b,h,i] = v[b,h,keep_idx[b,h,i]];
 * and for every block j of blk consecutive compacted rows (the last one
 * partial), over its rows [j*blk, min(B1, (j+1)*blk)):
 *   kt[b,h,0,c,j] = max k_out[.,c],  kt[b,h,1,c,j] = min k_out[.,c].
 * Equal to rkv_snap_evict's compaction followed by rkv_build_kt on the
 * compacted cache (bit for bit), in one pass over the kept rows; run
 * rkv_snap_evict in mask mode (k_out = v_out = NULL) first to get keep_idx.
 * Arguments
 *   k, v       [B, Hkv, cap, D] bf16 prompt caches (16-byte aligned), each in
 *              device memory or in page-locked host memory: a host-resident
 *              cache is read in place over the host link, so only its kept
 *              rows cross it (stage 1 needs all of K but none of V).
 *   keep_idx   [B, Hkv, keep_ld] int32 rows to keep (entries are clamped into
 *              [0, cap)); keep_ld >= B1.
 *   k_out,v_out[B, Hkv, out_cap, D] bf16 compacted caches, B1 <= out_cap;
 *              must not overlap k, v.
 *   kt         [B, Hkv, 2, D, nblk_cap] bf16 (16-byte aligned), nblk_cap a
 *              multiple of 8 and >= ceil(B1 / blk); columns [0, ceil(B1/blk))
 *              are written.
 * Errors: RKV_ERR_INVALID_ARG for NULL or misaligned pointers, k or v in
 * memory the device cannot reach (pageable host memory included), and the
 * size rules above; RKV_ERR_CUDA if the launch fails.
 */
rkv_status rkv_compact_kt(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                          int64_t keep_ld, int64_t B1, void* k_out, void* v_out, int64_t out_cap, int32_t blk, void* kt,
                          int64_t nblk_cap, void* stream);

/*
 * rkv_compact_kt writing the compacted rows into pages: row i of batch row b
 * (for every KV head h) goes to slot i % blk of page block_table[b, i / blk]:
 *   k_pages[page, h, i % blk] = k[b, h, keep_idx[b, h, i]], likewise for v;
 * KT as rkv_compact_kt (per (b, h), logical block order); k and v as there
 * (device or page-locked host memory).
 *   k_pages,v_pages [num_pages, Hkv, blk, D] bf16 pools (16-byte aligned).
 *   block_table     [B, bt_stride] int32 DEVICE array, bt_stride >= ceil(B1/blk);
 *                   page ids are clamped into [0, num_pages).
 * Errors as rkv_compact_kt.
 */
rkv_status rkv_compact_kt_paged(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                                int64_t keep_ld, int64_t B1, void* k_pages, void* v_pages, int64_t num_pages,
                                const int32_t* block_table, int64_t bt_stride, int32_t blk, void* kt,
                                int64_t nblk_cap, void* stream);

/*
 * KT cache build.  [RocketKV digest, 方法细节: HSA step 1 -- tokens grouped
 * into pages along the sequence, elementwise Kmax and Kmin per page stored
 * aligned along the head dimension]
 * For block j (tokens j*blk .. min(n, (j+1)*blk)-1) and channel c:
 *   kt[b,h,0,c,j] = max of k[b,h,row(t),c],  kt[b,h,1,c,j] = min of the same,
 * row(t) = t (idx == NULL) or idx[b,h,t] (MT candidate rows).
 * Writes blocks [0, ceil(n/blk)); requires ceil(n/blk) <= nblk_cap, n <= cap.
 */
rkv_status rkv_build_kt(rkv_dims d, const void* k, int64_t cap, int64_t n, const int32_t* idx,
                        int64_t idx_cap, int32_t blk, void* kt, int64_t nblk_cap, void* stream);

/*
 * Append one decoded token per (b, h) and update the KT cache.  [RocketKV
 * digest, 方法细节: HSA step 1 -- the auxiliary storage is updated whenever a
 * new key is generated]
 *   k[b,h,row] = k_new[b,h], v[b,h,row] = v_new[b,h]   ([B, Hkv, D] bf16);
 *   candidate n joins block n/blk: a new block starts from k_new, otherwise
 *   Kmax = max(Kmax, k_new), Kmin = min(Kmin, k_new);
 *   MT (idx != NULL): idx[b,h,n] = row.  Non-MT: pass row == n, idx = NULL.
 * The caller's n becomes n+1 after the call.
 */
rkv_status rkv_append_kv(rkv_dims d, const void* k_new, const void* v_new, void* k, void* v, int64_t cap,
                         int64_t n, int64_t row, int32_t* idx, int64_t idx_cap, void* kt,
                         int64_t nblk_cap, int32_t blk, void* stream);

/*
 * Stage 2: one HSA decode step, optionally fused with the step's append.
 * [RocketKV digest, 方法细节: HSA steps 1-3 and Algorithm 1]
 * With k_new/v_new ([B, Hkv, D] bf16) the token is first appended as candidate
 * n -- k[b,h,n] = k_new, v[b,h,n] = v_new and its KT block updated exactly as
 * rkv_append_kv does -- and the step attends the n+1 candidates; with both
 * NULL it attends the first n.  For every (b, KV head h), with the group's
 * queries q_g and N the attended count:
 *   i1   = top-k1 channels of sum_g |q_g| (equal values: lower channel first);
 *   qbar = sum_g q_g;  P[c] = Kmax[c] if qbar[c] >= 0 else Kmin[c];
 *   s[j] = sum_{c in i1} qbar[c] * P[c, j] for blocks j < nblk = ceil(N/blk);
 *   i2   = top-k2 blocks of s (equal: lower block first; all if k2 >= nblk);
 *   out[b, g] = softmax(q_g . k_t * scale) weighted sum of v_t over the valid
 *               tokens t < N of the blocks in i2 (fp32 output [B, Hq, D]).
 * Arguments
 *   k, v       [B, Hkv, cap, D] bf16 compacted caches, rows [0, n) valid.
 *   kt         KT cache covering [0, n); nblk_cap must be a multiple of 8.
 *   sel_blocks optional [B, Hkv, k2] int32: i2 ascending, -1 padded.
 *   sel_channels optional [B, Hkv, k1] int32: i1 ascending.
 * Requires 1 <= N <= cap, ceil(N/blk) <= nblk_cap, 1 <= k1 <= D, k2 >= 1,
 * 1 <= blk <= 128 (RKV_ERR_UNSUPPORTED otherwise), ceil(N/blk) <= 8192.
 * Block sizes that are multiples of 8 stream the selected K/V blocks with TMA;
 * other sizes (1 gives token-level selection) gather the rows one by one.
 * No workspace: split partials are combined on chip.
 * The launch may overlap the tail of the previous kernel on the stream
 * (programmatic dependent launch); it reads no input before that kernel ends.
 */
rkv_status rkv_hsa_decode(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n, void* kt,
                          int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale, float* out,
                          int32_t* sel_blocks, int32_t* sel_channels, const void* k_new, const void* v_new,
                          void* stream);

/*
 * RocketKV-MT decode step.  [RocketKV digest, 方法细节: RocketKV-MT -- all KV
 * tokens stay in memory, stage 2 selects only among the stage-1 survivors
 * plus newly generated tokens]
 * Same as rkv_hsa_decode over the candidate sequence t = 0 .. N-1 whose key
 * and value rows are k[b,h,idx[b,h,t]] and v[b,h,idx[b,h,t]] (full caches);
 * kt must be built over that sequence (rkv_build_kt with the same idx).  With
 * k_new/v_new the token is first written to cache row `row` and becomes
 * candidate n (idx[b,h,n] = row).
 */
rkv_status rkv_hsa_decode_mt(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int32_t* idx,
                             int64_t idx_cap, int64_t n, void* kt, int64_t nblk_cap, int32_t blk, int32_t k1,
                             int32_t k2, float scale, float* out, int32_t* sel_blocks, int32_t* sel_channels,
                             const void* k_new, const void* v_new, int64_t row, void* stream);

/*
 * RocketKV-MT, the reading over fixed blocks of the full cache.  [RocketKV
 * digest, 方法细节: RocketKV-MT -- every token stays in memory; stage 2
 * chooses among the N surviving input tokens plus the newly generated ones]
 * The pages leave open whether stage 2's blocks run over the survivors'
 * sequence (rkv_hsa_decode_mt) or over the full cache; these three calls
 * build the second reading.  Rows [0, n_prompt) of the full cache are the
 * prompt that stage 1 filtered; row r < n_prompt is a candidate when bit r of
 * the mask is set, and every row r >= n_prompt (decoded after that prompt)
 * is a candidate.
 *   mask  [B, Hkv, mask_ld] uint32 DEVICE array, bit r = word r / 32, bit
 *         r % 32; mask_ld >= ceil(n_prompt / 32); 4-byte aligned.
 *
 * rkv_keep_mask: mask bits [0, n_prompt) = the rows listed in keep_idx[b,h,
 * 0:B1] (the keep list of rkv_snap_evict in mask mode); entries outside
 * [0, n_prompt) are ignored.
 */
rkv_status rkv_keep_mask(rkv_dims d, const int32_t* keep_idx, int64_t keep_ld, int64_t B1, int64_t n_prompt,
                         uint32_t* mask, int64_t mask_ld, void* stream);

/*
 * KT over fixed blocks of the full cache, candidate rows only: for block j,
 * Kmax / Kmin over the candidate rows of [j*blk, min(n, (j+1)*blk)); a block
 * without candidates stores zeros.  Layout and size rules as rkv_build_kt
 * (no idx); n_prompt <= n <= cap.
 */
rkv_status rkv_build_kt_masked(rkv_dims d, const void* k, int64_t cap, int64_t n, const uint32_t* mask,
                               int64_t mask_ld, int64_t n_prompt, int32_t blk, void* kt, int64_t nblk_cap,
                               void* stream);

/*
 * HSA decode step of that reading.  Same arguments and rules as rkv_hsa_decode
 * (n = rows of the full cache in use, the fused append writes row n, which is
 * a candidate), plus the mask and n_prompt <= n.  Per (b, h):
 *   bounds  Kmax / Kmin of block j over its candidate rows (the fused append
 *           starts a block's bounds when it holds no earlier candidate);
 *   s[j]    Algorithm 1's score, -inf for a block without candidates, +inf
 *           for the block of the newest row N-1 when it holds a candidate;
 *   i2      top-k2 of s as rkv_hsa_decode (equal: lower block first);
 *   out     attention over the candidate rows of the blocks in i2.
 * Errors as rkv_hsa_decode, plus RKV_ERR_INVALID_ARG for a NULL or misaligned
 * mask, n_prompt outside [0, min(n, cap)] or mask_ld < ceil(n_prompt / 32).
 */
rkv_status rkv_hsa_decode_mt_masked(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n,
                                    const uint32_t* mask, int64_t mask_ld, int64_t n_prompt, void* kt,
                                    int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale, float* out,
                                    int32_t* sel_blocks, int32_t* sel_channels, const void* k_new, const void* v_new,
                                    void* stream);

/*
 * e4m3 (FP8) storage of the compacted cache.  Not on the pages: a storage
 * option that halves the bytes of each decode step (the pages' KV-size
 * formula counts one byte per element for FP8).  A code has 1 sign bit, 4
 * exponent bits (bias 7) and 3 mantissa bits; there are no infinities,
 * S.1111.111 is NaN and the largest magnitude is 448.  A stored row's value
 * is code * scale, with fp32 scales per (b, h) that the caller chooses:
 *   k_scale, v_scale  [B, Hkv] fp32 DEVICE arrays (4-byte aligned).
 * rkv_compact_kt_fp8: rkv_compact_kt writing codes: k_out[b,h,i] =
 * code(k[b,h,keep_idx[b,h,i]] / k_scale[b,h]) (the quotient in fp32, nearest
 * even, magnitudes past 448 saturated), likewise v_out with v_scale; the KT
 * cache holds, per block, the max / min of the key codes' values, stored as
 * codes (exact).  k, v as rkv_compact_kt (bf16, device or page-locked host).
 *   k_out, v_out  [B, Hkv, out_cap, D] uint8 codes (16-byte aligned).
 *   kt            [B, Hkv, 2, D, nblk_cap] uint8 codes, nblk_cap a multiple of 16.
 * Errors as rkv_compact_kt, plus NULL or misaligned scales.
 */
rkv_status rkv_compact_kt_fp8(rkv_dims d, const void* k, const void* v, int64_t cap, const int32_t* keep_idx,
                              int64_t keep_ld, int64_t B1, const float* k_scale, const float* v_scale, void* k_out,
                              void* v_out, int64_t out_cap, int32_t blk, void* kt, int64_t nblk_cap, void* stream);

/*
 * HSA decode step over an e4m3 cache (k, v [B, Hkv, cap, D] and kt
 * [B, Hkv, 2, D, nblk_cap] uint8 codes from rkv_compact_kt_fp8).  Same rules
 * and results as rkv_hsa_decode, with the block scores taken on the KT codes'
 * values (the positive K scale does not change their order) and attention
 * over the rows' values code * scale.  The fused append stores
 * code(k_new / k_scale) and code(v_new / v_scale) at row n and folds the key's
 * code into its block.  Requires blk a multiple of 8 (RKV_ERR_UNSUPPORTED
 * otherwise) and nblk_cap a multiple of 16.
 */
rkv_status rkv_hsa_decode_fp8(rkv_dims d, const void* q, void* k, void* v, int64_t cap, int64_t n,
                              const float* k_scale, const float* v_scale, void* kt, int64_t nblk_cap, int32_t blk,
                              int32_t k1, int32_t k2, float scale, float* out, int32_t* sel_blocks,
                              int32_t* sel_channels, const void* k_new, const void* v_new, void* stream);

/*
 * HSA decode step for a batch whose rows hold different numbers of candidates
 * (ragged batch).  [RocketKV digest, 方法细节: HSA steps 1-3 and Algorithm 1,
 * per request]  Same computation, arguments and results as rkv_hsa_decode,
 * except that batch row b attends its own N_b = n_rows[b] (+1 with the fused
 * append) candidates: blocks, k2 (capped at row b's block count), the
 * appended row index (n_rows[b]) and the KT column it updates are per row.
 *   n_rows     [B] int32 DEVICE array, candidates before the step's append; it
 *              is read when the kernel starts (after the previous kernel on the
 *              stream has finished), so a graph can replay with new lengths.
 *              The library does not update it.
 *   n_max      host upper bound of n_rows: sizes the launch and is checked like
 *              rkv_hsa_decode's n (n_max (+1) <= cap, ceil(n_max (+1) / blk) <=
 *              nblk_cap).  An entry outside [1, n_max] is clamped into it and
 *              sets bit 1 of the device error word.
 */
rkv_status rkv_hsa_decode_ragged(rkv_dims d, const void* q, void* k, void* v, int64_t cap, const int32_t* n_rows,
                                 int64_t n_max, void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2,
                                 float scale, float* out, int32_t* sel_blocks, int32_t* sel_channels,
                                 const void* k_new, const void* v_new, void* stream);

/*
 * HSA decode step over paged K/V caches.  [RocketKV digest, 方法细节: HSA steps
 * 1-3 and Algorithm 1; a page is one HSA block]  Same computation, arguments
 * and results as rkv_hsa_decode_ragged, except that the K and V rows live in
 * pools of pages of blk rows shared by every batch row:
 *   k_pages,v_pages [num_pages, Hkv, blk, D] bf16 (16-byte aligned);
 *   block_table     [B, bt_stride] int32 DEVICE array: logical block j of batch
 *                   row b (its tokens j*blk .. j*blk+blk-1) is page
 *                   block_table[b, j] of the pools, for every KV head;
 *   n_rows          [B] int32 DEVICE array of candidates before the append, or
 *                   NULL: every row has n_max.
 * With the fused append the token goes to slot n % blk of page
 * block_table[b, n / blk], which the caller must have assigned.  KT stays
 * per (b, h) in logical block order, as for the dense caches.  Page ids out
 * of [0, num_pages) are clamped and set bit 1 of the device error word.
 * Requires n_max (+1) <= bt_stride * blk and the limits of rkv_hsa_decode.
 */
rkv_status rkv_hsa_decode_paged(rkv_dims d, const void* q, void* k_pages, void* v_pages, int64_t num_pages,
                                const int32_t* block_table, int64_t bt_stride, const int32_t* n_rows, int64_t n_max,
                                void* kt, int64_t nblk_cap, int32_t blk, int32_t k1, int32_t k2, float scale,
                                float* out, int32_t* sel_blocks, int32_t* sel_channels, const void* k_new,
                                const void* v_new, void* stream);

/*
 * Diagnostics for the bounded waits of the HSA decode kernels (every
 * rkv_hsa_decode* call made after it, from any host thread).  limit_ns > 0
 * shortens each bounded wait from 1 s to limit_ns (at least 1000); extra_bytes
 * (at most 4096) is added to the byte count that each CTA's block-score
 * barrier expects, bytes that no copy ever delivers, so that wait runs out
 * while every real copy still completes: the kernel then goes on with the
 * scores it has received, finishes, and sets bit 0 of the device error word.
 * rkv_debug_set_wait(0, 0) restores normal operation.  Host only.
 */
rkv_status rkv_debug_set_wait(uint64_t limit_ns, uint32_t extra_bytes);

/*
 * Read and clear the library's device error word (synchronises the device).
 * Bit 0: a bounded wait for an asynchronous copy gave up in some kernel.
 * Bit 1: a per-row length, keep count or page id read from device memory was
 *        out of range (it was clamped).
 * Returns RKV_ERR_TIMEOUT if any bit was set, RKV_OK otherwise.
 */
rkv_status rkv_read_device_flags(uint32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* RKV_H */
