// Stage 1 of RocketKV: SnapKV eviction at the end of prefill.
//
// Method: "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV
// Cache Compression" (papercache digest), section 方法细节: SnapKV selects the
// prompt tokens most attended by an observation window at the prompt tail;
// scores are aggregated per GQA group (Ada-KV style) so the group shares one
// token set; a 1-D pooling of kernel 63 keeps neighbours of the chosen tokens.
// "RocketKV Guide" (aifetchly blog), Stage 1: window of 32 queries, softmax
// scale 1/sqrt(D).
//
// Kernels (all per (batch row, KV head) "pair"):
//   snap_pass<1>  row softmax statistics (max, sum) of every window query over
//                 its causal key range, per key chunk;
//   snap_pass<2>  per prefix key, the sum over the group's window rows of the
//                 normalised probabilities (column sums of P), per row group;
//   snap_pool     sum of row-group partials in fixed order, then max-pool;
//   snap_select   exact top-k of the pooled scores (radix select on an
//                 order-preserving key, equal keys: lower index first) written
//                 in ascending index order, plus sinks and the window;
//   snap_pool_select  the two above fused in one CTA per pair when the prefix
//                 fits shared memory (up to 1024 x 32 positions);
//   snap_compact  gather of the kept K and V rows (skipped in MT mask mode).
// The two score passes stream K with 3-D TMA tiles (128-byte swizzle) through
// a 4-stage mbarrier ring and run the contraction on tcgen05.mma into TMEM.
#include "rkv_common.cuh"
#include "rkv_internal.h"

#include <algorithm>
#include <mutex>

namespace rkv {

static __device__ unsigned int g_snap_err = 0;

// Full cluster barrier: release this CTA's prior writes (shared and global
// memory) to every CTA of the cluster, and acquire theirs.
// 4-byte asynchronous copy global -> shared (no register staging)
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Loads from another CTA's shared memory (an address from mapa).
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

namespace {

// Score passes on the 5th-generation tensor core.  One CTA = one (pair, row
// group, key chunk).  Warp 0 streams K tiles (128 keys x 128 dims, two
// 64-dim TMA boxes with 128-byte swizzle) through a 4-stage ring; warp 1
// issues tcgen05.mma into one of two TMEM accumulators; warps 2-5 (one per
// TMEM lane quadrant) drain the accumulators.
//   pass 1: D[128 query rows x 128 keys] = Q K^T; each epilogue thread owns a
//           query row and keeps its online softmax (max, sum) over the keys.
//           Groups of more than 128 window rows take 256 per CTA (two MMAs per
//           key tile into the two halves of a 256-column buffer, each epilogue
//           set draining one half of every tile), so the keys are read once per
//           256 rows instead of once per 128.
//   pass 2: D[128 keys x Ng query rows] = K Q^T; each epilogue thread owns a
//           key and sums exp2(logit - lse(row)) over the rows in registers.
constexpr int T_KEYS = 128;                       // keys per tile
constexpr int T_NST = 4;                          // smem ring depth (3 measured 1 % slower on the 32K layer)
constexpr int T_NT = 320;                         // producer, MMA, two sets of 4 epilogue warps
constexpr int P_CHUNK = 2048;                     // keys per work item (smaller when that leaves SMs idle)
constexpr int P1_ROWS = 128;                      // query rows per pass-1 MMA (M); a CTA takes one or two
constexpr int P2_ROWS = 256;                      // query rows per pass-2 CTA (MMA N, max)
constexpr uint32_t T_KTILE = T_KEYS * 256;        // 32 KB: two 16 KB k-blocks
constexpr uint32_t T_QMAX = P2_ROWS * 256;        // 64 KB

struct PassArgs {
  int64_t S, L;                    // L = S - W prefix keys (per-row lengths: the maxima)
  const int32_t* S_rows;           // [B] prompt length of each batch row, or nullptr (all rows S)
  const int32_t* bt;               // paged prompt cache: [B, bt_stride] page of each logical page, or nullptr
  int64_t bt_stride, num_pages;
  int32_t page_shift;              // log2 of the rows per page (pages hold 8 .. 128 rows)
  int32_t Hq, Hkv, G, W, R, RG1, RG2, nchunk1, nq2;
  int32_t p1rows;                  // query rows per pass-1 CTA: 128, or 256 for groups of more than 128 rows
  int32_t pairs, nchunk2;
  int32_t chunk;                   // keys per work item: P_CHUNK, halved down to 2 tiles for small jobs
  float scale_log2;
  float2* stats;                   // [pairs][R][nchunk1]
  float* scores;                   // [pairs][RG2][L]
};

struct TcSmem {                    // lives after the operand tiles
  uint64_t full[T_NST], empty[T_NST];
  uint64_t tfull[2], tempty[2];
  uint64_t qbar, qfree;            // Q tile loaded / no longer read by the MMAs
  uint32_t tmem_base;
  int32_t abort_flag;
  __align__(16) float nlse[P2_ROWS];   // pass 2: -log2(sum) of every query row
  float2 part[128];                // pass 1: (max, sum) of the second epilogue set, per row
};
// 1024 bytes of slack to align the base, the operand tiles, then the barriers and row data
constexpr uint32_t T_SMEM = 1024 + T_QMAX + T_NST * T_KTILE + (uint32_t)((sizeof(TcSmem) + 127) / 128 * 128);

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                        unsigned int* err) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// OR of p over the 256 epilogue threads (named barrier 1), the same in every one.
__device__ __forceinline__ bool epi_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}

// One batch row's stage-1 lengths.  Without per-row arrays they are the
// call's own S and B1.  Per-row entries are clamped into range: S_b into
// [1, S_max]; B1_b into [min(W + sinks, hi), hi] with hi = min(S_b, B1_max)
// (an entry at or past S_b keeps the whole row and is no error).  `bad` marks
// a clamped entry.
struct RowPlan {
  int S, L, sinks, B1;
  int64_t ntop;                    // prefix positions chosen by the top-k
  bool all, bad;                   // every token kept; an entry was out of range
};
__device__ __forceinline__ RowPlan row_plan(const int32_t* S_rows, const int32_t* B1_rows, int b, int64_t S_max,
                                            int64_t B1_max, int W, int n_sink) {
  RowPlan p;
  p.bad = false;
  int64_t S = S_max;
  if (S_rows) {
    const int64_t r = S_rows[b];
    S = min(max(r, (int64_t)1), S_max);
    p.bad |= S != r;
  }
  const int w = (int)min((int64_t)W, S);
  p.S = (int)S;
  p.L = (int)(S - w);
  p.sinks = min(n_sink, p.L);
  int64_t B1 = B1_max;
  if (B1_rows) {
    const int64_t r = B1_rows[b];
    const int64_t hi = min(S, B1_max), lo = min((int64_t)w + p.sinks, hi);
    B1 = min(max(r, lo), hi);
    p.bad |= B1 != r && !(r >= S && B1 == S);
  }
  p.all = B1 >= S || p.L <= 0;
  if (p.all) B1 = S;
  p.B1 = (int)B1;
  p.ntop = max((int64_t)0, B1 - w - p.sinks);
  return p;
}

// Prompt length of pair `pair`'s batch row.
__device__ __forceinline__ int64_t pair_S(const PassArgs& a, int pair) {
  return a.S_rows ? min(max((int64_t)a.S_rows[pair / a.Hkv], (int64_t)1), a.S) : a.S;
}

// One work item = (pair, row group, key chunk of a.chunk keys).  The grid is
// persistent: CTA c takes the contiguous items [c*n/grid, (c+1)*n/grid), so
// the K stream, the MMAs and the epilogue run across item boundaries without
// draining; the Q tile is reloaded only when (pair, row group) changes.
struct PassItem {
  int pair, rg, chunk, ntiles;
  int64_t j0;
};
template <int PASS>
__device__ __forceinline__ PassItem pass_item(const PassArgs& a, int item) {
  const int nchunk = PASS == 1 ? a.nchunk1 : a.nchunk2;
  const int RGp = PASS == 1 ? a.RG1 : a.RG2;
  PassItem it;
  it.chunk = item % nchunk;
  const int t2 = item / nchunk;
  it.rg = t2 % RGp;
  it.pair = t2 / RGp;
  // (a batch row shorter than the longest has empty items past its own length)
  const int64_t Sp = pair_S(a, it.pair);
  const int64_t kend = (PASS == 1) ? Sp : max(Sp - (int64_t)a.W, (int64_t)0);
  it.j0 = (int64_t)it.chunk * a.chunk;
  const int64_t j1 = min(kend, it.j0 + (int64_t)a.chunk);
  it.ntiles = j1 > it.j0 ? (int)((j1 - it.j0 + T_KEYS - 1) / T_KEYS) : 0;
  return it;
}

// Pass 2 walks a CTA's items backwards: with the same partition as pass 1 (one
// row group per pair), the K chunks a CTA read last in pass 1 are still in L2.
template <int PASS>
__device__ __forceinline__ int item_at(int ib, int ie, int ii) {
  return PASS == 2 ? ie - 1 - (ii - ib) : ii;
}

template <int PASS, bool WIDE = false>
__global__ void __launch_bounds__(T_NT, 1) snap_pass_kernel(const __grid_constant__ CUtensorMap tmK,
                                                            const __grid_constant__ CUtensorMap tmQ,
                                                            const PassArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sQ = smem;                                   // 2 k-blocks of nq rows x 128 B
  uint8_t* sK = smem + T_QMAX;                          // T_NST stages of 2 k-blocks x 128 keys x 128 B
  TcSmem& ts = *reinterpret_cast<TcSmem*>(smem + T_QMAX + T_NST * T_KTILE);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr bool wide = PASS == 1 && WIDE;             // pass 1 with two 128-row MMAs per tile (256 rows)
  const int nq = PASS == 1 ? (wide ? 2 * P1_ROWS : P1_ROWS) : a.nq2;   // Q tile rows (pass 2: MMA N)
  const int ncols = PASS == 1 ? T_KEYS : nq;                            // accumulator columns per MMA
  const int bcols = wide ? 2 * T_KEYS : ncols;                          // columns per buffer
  const uint32_t tcols = PASS == 1 ? (wide ? 512u : 256u) : (nq <= 64 ? 128u : (nq <= 128 ? 256u : 512u));
  const int nitems = a.pairs * (PASS == 1 ? a.RG1 * a.nchunk1 : a.RG2 * a.nchunk2);
  const int ib = (int)((int64_t)blockIdx.x * nitems / gridDim.x);
  const int ie = (int)((int64_t)(blockIdx.x + 1) * nitems / gridDim.x);
  unsigned int* err = &g_snap_err;
  volatile int32_t* abort_flag = &ts.abort_flag;

  if (tid == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmQ);
    for (int s = 0; s < T_NST; ++s) {
      mbar_init(&ts.full[s], 1);
      mbar_init(&ts.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ts.tfull[i], 1);
      mbar_init(&ts.tempty[i], wide ? 256 : 128);   // (wide pass 1: both epilogue sets drain every buffer)
    }
    mbar_init(&ts.qbar, 1);
    mbar_init(&ts.qfree, 1);
    ts.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ts.tmem_base, tcols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ts.tmem_base;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      int T = 0, nload = 0, key = -1;
      for (int ii = ib; ii < ie && !*abort_flag; ++ii) {
        const PassItem it = pass_item<PASS>(a, item_at<PASS>(ib, ie, ii));
        const int k = it.pair * (PASS == 1 ? a.RG1 : a.RG2) + it.rg;
        if (k != key) {
          // the MMAs of the previous Q tile have completed before it is overwritten
          if (nload > 0 && !tc_wait(&ts.qfree, (nload - 1) & 1, abort_flag, err)) break;
          const int b = it.pair / a.Hkv, hk = it.pair % a.Hkv;
          const int qrow = (b * a.Hq + hk * a.G) * a.W + it.rg * (PASS == 1 ? nq : P2_ROWS);
          mbar_arrive_expect_tx(&ts.qbar, (uint32_t)nq * 256u);
          for (int h = 0; h < 2; ++h)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                "%3}], [%4];" ::"r"(smem_u32(sQ + h * nq * 128)),
                "l"(reinterpret_cast<uint64_t>(&tmQ)), "r"(h * 64), "r"(qrow), "r"(smem_u32(&ts.qbar))
                : "memory");
          ++nload;
          key = k;
        }
        for (int t = 0; t < it.ntiles; ++t, ++T) {
          const int s = T % T_NST;
          if (T >= T_NST && !tc_wait(&ts.empty[s], ((T / T_NST) & 1) ^ 1, abort_flag, err)) break;
          mbar_arrive_expect_tx(&ts.full[s], T_KTILE);
          const int y = (int)(it.j0 + (int64_t)t * T_KEYS);
          if (a.bt) {
            // paged prompt: one box per page of the tile (a (page, KV head) slab of
            // the pool), each channel half; rows of the swizzled tile continue across pages
            const int b = it.pair / a.Hkv, hk = it.pair - b * a.Hkv;
            const int lp0 = y >> a.page_shift, npg = T_KEYS >> a.page_shift;
            const int32_t* btr = a.bt + (size_t)b * a.bt_stride;
            for (int i = 0; i < npg; ++i) {
              const int lp = lp0 + i;
              const int id = lp < a.bt_stride ? __ldg(btr + lp) : 0;
              const int idc = min(max(id, 0), (int)a.num_pages - 1);
              if (idc != id && lp < a.bt_stride) atomicOr(err, ERR_BAD_LENGTH);
              const uint32_t off = ((uint32_t)i << a.page_shift) * 128u;
              tma_load_3d(sK + s * T_KTILE + off, &tmK, 0, 0, idc * a.Hkv + hk, &ts.full[s]);
              tma_load_3d(sK + s * T_KTILE + T_KTILE / 2 + off, &tmK, 64, 0, idc * a.Hkv + hk, &ts.full[s]);
            }
          } else {
            tma_load_3d(sK + s * T_KTILE, &tmK, 0, y, it.pair, &ts.full[s]);
            tma_load_3d(sK + s * T_KTILE + T_KTILE / 2, &tmK, 64, y, it.pair, &ts.full[s]);
          }
        }
      }
      // every load issued has landed before the CTA can leave (bounded)
      for (int t = max(0, T - T_NST); t < T; ++t) mbar_wait(&ts.full[t % T_NST], (t / T_NST) & 1, err);
      if (nload > 0) mbar_wait(&ts.qbar, (nload - 1) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA --
    if (lane == 0) {
      const uint32_t idesc = PASS == 1 ? idesc_bf16_f32(128, T_KEYS) : idesc_bf16_f32(128, nq);
      int T = 0, nload = 0, key = -1;
      bool ok = true;
      for (int ii = ib; ii < ie && ok; ++ii) {
        const PassItem it = pass_item<PASS>(a, item_at<PASS>(ib, ie, ii));
        const int k = it.pair * (PASS == 1 ? a.RG1 : a.RG2) + it.rg;
        if (k != key) {
          if (nload > 0) tc_commit(&ts.qfree);        // arrives once every MMA issued so far is done
          if (!tc_wait(&ts.qbar, nload & 1, abort_flag, err)) break;
          ++nload;
          key = k;
        }
        for (int t = 0; t < it.ntiles; ++t, ++T) {
          const int s = T % T_NST, buf = T & 1;
          if (!tc_wait(&ts.full[s], (T / T_NST) & 1, abort_flag, err)) { ok = false; break; }
          if (T >= 2 && !tc_wait(&ts.tempty[buf], ((T >> 1) & 1) ^ 1, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kt = smem_u32(sK + s * T_KTILE), qt = smem_u32(sQ);
          const uint32_t d = tbase + (uint32_t)(buf * bcols);
#pragma unroll
          for (int kk8 = 0; kk8 < 8; ++kk8) {
            const int kb = kk8 >> 2, kk = kk8 & 3;
            const uint64_t kdesc = sdesc_k_sw128(kt + kb * (T_KTILE / 2) + kk * 32);
            const uint64_t qdesc = sdesc_k_sw128(qt + kb * nq * 128 + kk * 32);
            if (PASS == 1) {
              tc_mma_bf16(d, qdesc, kdesc, idesc, kk8 > 0);
              // rows 128-255 of the Q tile (16 KB further into each k-block) into the second half of the buffer
              if (wide) tc_mma_bf16(d + T_KEYS, sdesc_k_sw128(qt + kb * nq * 128 + 128 * 128 + kk * 32), kdesc, idesc,
                                    kk8 > 0);
            } else {
              tc_mma_bf16(d, kdesc, qdesc, idesc, kk8 > 0);
            }
          }
          tc_commit(&ts.empty[s]);
          tc_commit(&ts.tfull[buf]);
        }
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue --
    // Two sets of four warps; set e drains TMEM buffer e, i.e. the tiles T of the
    // CTA's stream with T % 2 == e (wide pass 1: set e drains rows 128 e .. of
    // every tile, from the half e of that tile's buffer).
    const int eset = (warp - 2) >> 2;                // 0 or 1
    const int quad = warp & 3;                       // TMEM lanes 32*quad .. +31
    const int r_loc = 32 * quad + lane;              // TMEM lane of this thread
    const int etid = (warp - 2) * 32 + lane;         // 0 .. 255 over both sets
    const uint32_t lane_addr = tbase + ((uint32_t)(32 * quad) << 16) + (uint32_t)(eset * ncols);
    const uint32_t lane_base = tbase + ((uint32_t)(32 * quad) << 16) + (uint32_t)(eset * T_KEYS);   // (wide)
    int T0 = 0, key = -1;                            // first tile of the item in the CTA's stream
    for (int ii = ib; ii < ie; ++ii) {
      const PassItem it = pass_item<PASS>(a, item_at<PASS>(ib, ie, ii));
      const int j032 = (int)it.j0;
      const int pair = it.pair;
      const int S32 = (int)pair_S(a, pair), L32 = max(S32 - a.W, 0);   // this row's prompt and prefix
      const int row0 = it.rg * (PASS == 1 ? nq : P2_ROWS);
      const int tfirst = wide ? 0 : ((T0 & 1) == eset ? 0 : 1);   // this set's first tile of the item
      const int tstep = wide ? 1 : 2;
      if (PASS == 1) {
        const int r = row0 + (wide ? P1_ROWS * eset : 0) + r_loc;   // query row in the group
        const bool rvalid = r < a.R;
        const int lim = S32 - a.W + (rvalid ? (r % a.W) : 0);     // last key this row attends
        float m = neg_inf(), l = 0.f;
        for (int t = tfirst; t < it.ntiles; t += tstep) {
          const int T = T0 + t;
          const int bf = wide ? (T & 1) : eset;         // this tile's buffer
          const uint32_t la = wide ? lane_base + (uint32_t)(bf * bcols) : lane_addr;
          // the warp gives up together: the TMEM loads below are warp-collective
          if (!__all_sync(0xffffffffu, tc_wait(&ts.tfull[bf], (T >> 1) & 1, abort_flag, err))) break;
          tc_fence_after();
          // online softmax over the tile's four 32-key chunks; the next chunk's
          // TMEM load is in flight while one is reduced (64 value registers)
          const int jt = j032 + t * T_KEYS;
          const bool full_tile = jt + T_KEYS <= S32 - a.W;   // every row attends every key of the tile
          const int jmax = min(S32 - 1, lim) - jt;           // last attended column of the tile
          float va[32], vb[32];
          tmem_ld32(la, va);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float* cur = (c & 1) ? vb : va;
            if (c < 3) tmem_ld32(la + 32 * (c + 1), (c & 1) ? va : vb);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            float mn;
            if (full_tile) {
              // the maximum of the raw logits scales to the maximum of the scaled ones (scale > 0)
              float x0 = fmax3(cur[0], cur[1], cur[2]), x1 = fmax3(cur[3], cur[4], cur[5]);
#pragma unroll
              for (int i = 6; i < 30; i += 4) {
                x0 = fmax3(x0, cur[i], cur[i + 1]);
                x1 = fmax3(x1, cur[i + 2], cur[i + 3]);
              }
              x0 = fmax3(x0, x1, fmaxf(cur[30], cur[31]));
              mn = fmaxf(m, x0 * a.scale_log2);
              const float2 sc = make_float2(a.scale_log2, a.scale_log2), nm = make_float2(-mn, -mn);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 x = fma_f2(make_float2(cur[i], cur[i + 1]), sc, nm);
                acc[(i >> 1) & 3] = add_f2(acc[(i >> 1) & 3], make_float2(ex2_ftz(x.x), ex2_ftz(x.y)));
              }
            } else {
              float tm = neg_inf();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float x = (32 * c + i <= jmax) ? cur[i] * a.scale_log2 : neg_inf();
                cur[i] = x;
                tm = fmaxf(tm, x);
              }
              mn = fmaxf(m, tm);
              if (mn != neg_inf()) {
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                  acc[(i >> 1) & 3] =
                      add_f2(acc[(i >> 1) & 3], make_float2(ex2_ftz(cur[i] - mn), ex2_ftz(cur[i + 1] - mn)));
              }
            }
            const float2 s01 = add_f2(add_f2(acc[0], acc[1]), add_f2(acc[2], acc[3]));
            if (mn != neg_inf()) {
              l = (m == neg_inf() ? 0.f : l * ex2_ftz(m - mn)) + (s01.x + s01.y);
              m = mn;
            }
            if (c < 3) tmem_wait_ld();
          }
          tc_fence_before();
          mbar_arrive(&ts.tempty[bf]);
        }
        if (wide) {
          if (rvalid) a.stats[((size_t)pair * a.R + r) * a.nchunk1 + it.chunk] = make_float2(m, l);
        } else {
          // the two sets drained alternate tiles of the same rows: merge
          if (eset == 1) ts.part[r_loc] = make_float2(m, l);
          asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight epilogue warps
          if (eset == 0) {
            const float2 o = ts.part[r_loc];
            const float mn = fmaxf(m, o.x);
            const float ls =
                (m == neg_inf() ? 0.f : l * exp2f(m - mn)) + (o.x == neg_inf() ? 0.f : o.y * exp2f(o.x - mn));
            if (rvalid) a.stats[((size_t)pair * a.R + r) * a.nchunk1 + it.chunk] = make_float2(mn, ls);
          }
        }
      } else {
        const int k = pair * a.RG2 + it.rg;
        if (k != key) {
          key = k;
          asm volatile("bar.sync 1, 256;" ::: "memory");   // both sets are done with the old normalisers
          // negated log2-domain normaliser of every query row (rows past R:
          // -inf -> weight 0), combined from pass 1's per-chunk (max, sum); tpr
          // adjacent threads share a row and load its chunk statistics eight at a time
          const int tpr = 256 / nq;                      // nq is a multiple of 32: 1, 2, 4 or 8
          const int i = etid / tpr, p = etid - i * tpr;
          const int r = row0 + i;
          float M = neg_inf(), Ls = 0.f;
          if (r < a.R) {
            const float2* st = a.stats + ((size_t)pair * a.R + r) * a.nchunk1;
            for (int c0 = p; c0 < a.nchunk1; c0 += 8 * tpr) {
              float2 v[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int c = c0 + u * tpr;
                v[u] = c < a.nchunk1 ? st[c] : make_float2(neg_inf(), 0.f);
              }
              float mb = M;
#pragma unroll
              for (int u = 0; u < 8; ++u) mb = fmaxf(mb, v[u].x);
              if (mb != neg_inf()) {
                Ls = (M == neg_inf()) ? 0.f : Ls * exp2f(M - mb);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  if (v[u].x != neg_inf()) Ls += v[u].y * exp2f(v[u].x - mb);
                M = mb;
              }
            }
          }
          for (int o = 1; o < tpr; o <<= 1) {
            const float Mo = __shfl_xor_sync(0xffffffffu, M, o), Lo = __shfl_xor_sync(0xffffffffu, Ls, o);
            const float Mn = fmaxf(M, Mo);
            if (Mn != neg_inf())
              Ls = ((M == neg_inf()) ? 0.f : Ls * exp2f(M - Mn)) + ((Mo == neg_inf()) ? 0.f : Lo * exp2f(Mo - Mn));
            M = Mn;
          }
          if (p == 0) ts.nlse[i] = (r < a.R) ? -(M + log2f(Ls)) : neg_inf();
          asm volatile("bar.sync 1, 256;" ::: "memory");   // the eight epilogue warps
        }
        for (int t = tfirst; t < it.ntiles; t += 2) {
          const int T = T0 + t;
          // the warp gives up together: the TMEM loads below are warp-collective
          if (!__all_sync(0xffffffffu, tc_wait(&ts.tfull[eset], (T >> 1) & 1, abort_flag, err))) break;
          tc_fence_after();
          // the key's score is written as log2 of the sum of its probabilities,
          // sum_c 2^(y_c) with y_c = logit * scale - lse_c (log2 units).  A plain
          // fp32 sum is exact to about 2^-17 relative while it stays above 2^-100
          // (flushed terms are below 2^-126 each, at most 512 of them); a warp with
          // a smaller sum re-reads its accumulator and takes a log-sum-exp over
          // 32-row chunks instead, so scores far below the fp32 range keep their rank
          const float2 sc = make_float2(a.scale_log2, a.scale_log2);
          const float4* nl4 = reinterpret_cast<const float4*>(ts.nlse);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          auto sum32 = [&](const float* v, int c0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 nl = nl4[(c0 + i) >> 2];   // same address across the warp: broadcast
              const float2 x0 = fma_f2(make_float2(v[i], v[i + 1]), sc, make_float2(nl.x, nl.y));
              const float2 x1 = fma_f2(make_float2(v[i + 2], v[i + 3]), sc, make_float2(nl.z, nl.w));
              acc[(i >> 2) & 3] = add_f2(acc[(i >> 2) & 3], make_float2(ex2_ftz(x0.x), ex2_ftz(x0.y)));
              acc[((i >> 2) + 2) & 3] = add_f2(acc[((i >> 2) + 2) & 3], make_float2(ex2_ftz(x1.x), ex2_ftz(x1.y)));
            }
          };
          for (int c0 = 0; c0 < nq; c0 += 64) {        // nq is a multiple of 32
            float v[2][32];
            const bool two = c0 + 32 < nq;
            tmem_ld32(lane_addr + c0, v[0]);
            if (two) tmem_ld32(lane_addr + c0 + 32, v[1]);
            tmem_wait_ld();
            sum32(v[0], c0);
            if (two) sum32(v[1], c0 + 32);
          }
          const float2 s01 = add_f2(add_f2(acc[0], acc[1]), add_f2(acc[2], acc[3]));
          const float lin = s01.x + s01.y;
          float lm = neg_inf(), ls = 0.f;
          if (__any_sync(0xffffffffu, lin < 0x1p-100f)) {
            auto lse32 = [&](float* v, int c0) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 nl = nl4[(c0 + i) >> 2];
                const float2 x0 = fma_f2(make_float2(v[i], v[i + 1]), sc, make_float2(nl.x, nl.y));
                const float2 x1 = fma_f2(make_float2(v[i + 2], v[i + 3]), sc, make_float2(nl.z, nl.w));
                v[i] = x0.x;
                v[i + 1] = x0.y;
                v[i + 2] = x1.x;
                v[i + 3] = x1.y;
              }
              float x0 = fmax3(v[0], v[1], v[2]), x1 = fmax3(v[3], v[4], v[5]);
#pragma unroll
              for (int i = 6; i < 30; i += 4) {
                x0 = fmax3(x0, v[i], v[i + 1]);
                x1 = fmax3(x1, v[i + 2], v[i + 3]);
              }
              const float mn = fmaxf(lm, fmax3(x0, x1, fmaxf(v[30], v[31])));
              if (mn == neg_inf()) return;               // rows past the group (or all masked)
              const float2 nm = make_float2(-mn, -mn);
              float2 e[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 d = add_f2(make_float2(v[i], v[i + 1]), nm);
                e[(i >> 1) & 3] = add_f2(e[(i >> 1) & 3], make_float2(ex2_ftz(d.x), ex2_ftz(d.y)));
              }
              const float2 t01 = add_f2(add_f2(e[0], e[1]), add_f2(e[2], e[3]));
              ls = (lm == neg_inf() ? 0.f : ls * ex2_ftz(lm - mn)) + (t01.x + t01.y);
              lm = mn;
            };
            for (int c0 = 0; c0 < nq; c0 += 32) {
              float v[32];
              tmem_ld32(lane_addr + c0, v);
              tmem_wait_ld();
              lse32(v, c0);
            }
          }
          if (lin >= 0x1p-100f) {
            lm = 0.f;
            ls = lin;
          }
          tc_fence_before();
          mbar_arrive(&ts.tempty[eset]);
          const int j = j032 + t * T_KEYS + r_loc;
          if (j < L32) a.scores[((size_t)pair * a.RG2 + it.rg) * a.L + j] = lm == neg_inf() ? neg_inf() : lm + log2f(ls);
        }
      }
      T0 += it.ntiles;
      // a barrier per item (part[] is free again) that also agrees on giving up
      if (epi_any(*abort_flag != 0)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, tcols);
  }
}

// log2(2^a + 2^b) for log2-domain scores (-inf is an empty sum).
__device__ __forceinline__ float log2_add(float a, float b) {
  const float m = fmaxf(a, b);
  if (m == neg_inf()) return m;
  return m + log2f(exp2f(a - m) + exp2f(b - m));
}

// Sum of the row-group partials (fixed order, log2 domain), then max-pool
// (clipped ends).  pooled_log gets log2 of the pooled scores (what the select
// ranks); pooled_out, if set, the scores themselves (0 below the fp32 range).
constexpr int POOL_TILE = 1024;
constexpr int POOL_MAX_HALF = 512;

__global__ void __launch_bounds__(256) snap_pool_kernel(const float* scores, int RG, int64_t Ls, int half,
                                                        float* pooled_log, float* pooled_out, const int32_t* S_rows,
                                                        int64_t S_max, int Hkv, int W) {
  __shared__ float tile[POOL_TILE + 2 * POOL_MAX_HALF];
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  // Ls: row stride of the score arrays (the longest prefix); L: this row's prefix
  const int64_t Sp = S_rows ? min(max((int64_t)S_rows[pair / Hkv], (int64_t)1), S_max) : S_max;
  const int64_t L = max(Sp - (int64_t)W, (int64_t)0);
  const int64_t j0 = (int64_t)blockIdx.x * POOL_TILE;
  const int span = POOL_TILE + 2 * half;
  for (int i = threadIdx.x; i < span; i += blockDim.x) {
    const int64_t j = j0 - half + i;
    float v = neg_inf();
    if (j >= 0 && j < L) {
      v = scores[((size_t)pair * RG) * Ls + j];
      for (int r = 1; r < RG; ++r) v = log2_add(v, scores[((size_t)pair * RG + r) * Ls + j]);
    }
    tile[i] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < POOL_TILE; i += blockDim.x) {
    const int64_t j = j0 + i;
    if (j >= L) break;
    float m = tile[i];
    for (int t = 1; t <= 2 * half; ++t) m = fmaxf(m, tile[i + t]);
    pooled_log[(size_t)pair * Ls + j] = m;
    if (pooled_out) pooled_out[(size_t)pair * Ls + j] = exp2f(m);
  }
}

// Exact top-ntop of pooled[n_sink, L) per pair; keep = sinks + winners
// (ascending) + window.  One CTA of 1024 threads per pair.
constexpr int SEL_NT = 1024;

__device__ __forceinline__ int block_excl_scan(bool flag, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    wsum[32 + lane] = incl - v;
    if (lane == 31) wsum[64] = incl;
  }
  __syncthreads();
  const int r = wsum[32 + warp] + __popc(bal & ((1u << lane) - 1u));
  total = wsum[64];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(SEL_NT) snap_select_kernel(const float* pooled, int64_t Ls, int64_t S_max,
                                                             int W0, int n_sink0, int64_t B1_max,
                                                             int32_t* keep, int64_t keep_ld, const int32_t* S_rows,
                                                             const int32_t* B1_rows, int Hkv) {
  __shared__ int hist[256];
  __shared__ int wsum[72];
  __shared__ uint32_t sh_digit;
  __shared__ int64_t sh_k;
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.x, tid = threadIdx.x;
  // this row's lengths (Ls: row stride of the pooled scores)
  const RowPlan rp = row_plan(S_rows, B1_rows, pair / Hkv, S_max, B1_max, W0, n_sink0);
  if (rp.bad && tid == 0) atomicOr(&g_snap_err, ERR_BAD_LENGTH);
  const int64_t L = rp.L, S = rp.S, B1 = rp.B1;
  const int W = (int)(S - L), n_sink = rp.sinks;
  const int64_t ntop = rp.ntop;
  const float* p = pooled + (size_t)pair * Ls;
  int32_t* out = keep + (size_t)pair * keep_ld;
  if (rp.all) {
    for (int64_t i = tid; i < S; i += SEL_NT) out[i] = (int32_t)i;
    return;
  }
  for (int i = tid; i < n_sink; i += SEL_NT) out[i] = i;
  for (int i = tid; i < W; i += SEL_NT) out[B1 - W + i] = (int32_t)(S - W + i);
  if (ntop <= 0) return;
  const int64_t ncand = L - n_sink;
  if (ntop >= ncand) {
    for (int64_t i = tid; i < ncand; i += SEL_NT) out[n_sink + i] = (int32_t)(n_sink + i);
    return;
  }
  // radix select of the ntop-th largest key, 8 bits at a time from the top
  uint32_t prefix = 0, mask = 0;
  int64_t k = ntop;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += SEL_NT) hist[i] = 0;
    __syncthreads();
    for (int64_t j = n_sink + tid; j < L; j += SEL_NT) {
      const uint32_t key = f2key(p[j]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // suffix sums over bins, 8 bins per lane, highest bins first
      int c[8];
      int s = 0;
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        c[u] = hist[tid * 8 + u];
        s += c[u];
      }
      // exclusive suffix sum over lanes (lanes above hold higher bins)
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (tid + o < 32) incl += t;
      }
      int above = incl - s;   // count in bins of higher lanes
      for (int u = 7; u >= 0; --u) {
        if (above < k && above + c[u] >= k) {
          sh_digit = (uint32_t)(tid * 8 + u);
          sh_k = k - above;
        }
        above += c[u];
      }
    }
    __syncthreads();
    prefix |= sh_digit << shift;
    mask |= 255u << shift;
    k = sh_k;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int64_t need_eq = k;   // how many keys equal to T are taken (lowest indices first)
  int64_t pos = n_sink, eq_taken = 0;
  for (int64_t base = n_sink; base < L; base += SEL_NT) {
    const int64_t j = base + tid;
    const uint32_t key = (j < L) ? f2key(p[j]) : 0u;
    const bool gt = (j < L) && key > T;
    const bool eq = (j < L) && key == T;
    int eq_total, take_total;
    const int eq_before = block_excl_scan(eq, wsum, eq_total);
    const bool take = gt || (eq && eq_taken + eq_before < need_eq);
    const int tpos = block_excl_scan(take, wsum, take_total);
    if (take) out[pos + tpos] = (int32_t)j;
    pos += take_total;
    eq_taken += eq_total;
  }
}

// Buckets of the bucket select, and the padded shared-memory index of entry u
// (one pad word per 32: threads reading entries 32 apart hit distinct banks).
constexpr int PS_NB = 1024;
__device__ __forceinline__ int ps_pad(int u) { return u + (u >> 5); }

// Pool + select for one pair over a cluster of NC CTAs (prefixes of up to
// 16 x 256 x (h + 1) positions; one CTA for up to 256 (h + 1)).  CTA r pools
// positions [r*PC, r*PC + PC), PC = 256 (h + 1), each thread E = h + 1
// consecutive outputs: the window of output a + i is window entries
// [a + i, a + i + 2h], of which [a + E - 1, a + 2E - 2] is common to all E
// outputs, the rest a suffix of [a, a + E - 2] and a prefix of
// [a + 2E - 1, a + 3E - 3] (the van Herk / Gil-Werman split).
// The pooled scores form runs of equal values, and the passes after pooling
// walk a thread's runs (keys are order-preserving integers of the pooled log2
// scores).  The bucket select then runs over the cluster with four cluster
// barriers: the key range; the 1024-bucket histograms (every CTA sums all of
// them); the counts of certainly taken positions and the members of a split
// boundary bucket (which every CTA ranks itself); and one before leaving, so
// no CTA exits while another reads its shared memory.  Each CTA writes its own
// taken positions at their places in the ascending keep list.  An equal or
// non-finite key range, or a split bucket of more than CL_MAXM members, sends
// the keys to global scratch, where CTA 0 runs a radix select over them.
constexpr int CL_NT = 256;
constexpr int CL_MAXM = 512;
constexpr int CL_MAXNC = 16;                    // (beyond 8 CTAs: where the GPU schedules such clusters)

// shared words of one cluster CTA's padded window of CL_NT (h + 1) + 2 (h + 1)
// scores; its CL_NT (h + 1) pooled scores follow (cl_smem_words in all)
__host__ __device__ inline int cl_key_words(int h) {
  const int U = (CL_NT + 2) * (h + 1);
  return ((U + U / 32 + 1) + 3) & ~3;
}
__host__ __device__ inline int cl_smem_words(int h) {
  const int P = CL_NT * (h + 1);
  return cl_key_words(h) + (((P + P / 32 + 1) + 3) & ~3);
}

struct __align__(16) ClSmem {
  uint32_t hist[PS_NB];            // this CTA's bucket counts
  uint32_t ghist[PS_NB];           // the cluster's (radix fallback: 256-digit counts)
  uint2 memb[CL_MAXM];             // this CTA's members of the split bucket (key, position)
  uint2 allm[CL_MAXM];             // every member of the cluster, in CTA order
  uint32_t taken[CL_NT];           // taken bits of this CTA's positions (at most CL_NT * 32)
  uint32_t mm[2];                  // this CTA's (min, max) candidate key
  uint32_t cnt[2];                 // this CTA's (certainly taken positions, members)
  uint32_t ctk[CL_MAXNC];          // taken members of each CTA
  uint32_t certv[CL_MAXNC];        // certainly taken positions of each CTA
  uint32_t msv[CL_MAXNC + 1];      // where each CTA's members start among all (the total last)
  uint32_t wsum[CL_NT / 32], wmin[CL_NT / 32], wmax[CL_NT / 32];
  int32_t sh[8];
};

// Exclusive prefix of a flag over the CTA's CL_NT threads; writes the total.
__device__ __forceinline__ int cl_excl_scan(bool f, uint32_t* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < CL_NT / 32; ++w) {
    const int v = (int)wsum[w];
    if (w < warp) pre += v;
    tot += v;
  }
  __syncthreads();
  total = tot;
  return pre + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(CL_NT) snap_pool_select_cl_kernel(const float* scores, int RG, int64_t Ls, int h,
                                                                     int64_t S_max, int W0, int n_sink0,
                                                                     int64_t B1_max, int32_t* keep, int64_t keep_ld,
                                                                     float* pooled_out, const int32_t* S_rows,
                                                                     const int32_t* B1_rows, int Hkv, int NC,
                                                                     uint32_t* key_scratch) {
  extern __shared__ __align__(16) uint32_t xs[];
  __shared__ ClSmem cs;
  pdl_wait();
  pdl_launch_dependents();
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RowPlan rp = row_plan(S_rows, B1_rows, pair / Hkv, S_max, B1_max, W0, n_sink0);
  if (rp.bad && tid == 0 && rank == 0) atomicOr(&g_snap_err, ERR_BAD_LENGTH);
  const int L = rp.L, S = rp.S, B1 = rp.B1, W = rp.S - rp.L, n_sink = rp.sinks;
  const int ntop = (int)rp.ntop;
  const int E = h + 1, PC = CL_NT * E;
  const int p0 = rank * PC;                       // this CTA's first position
  int32_t* out = keep + (size_t)pair * keep_ld;
  // (every decision below up to the select is the same in every CTA of the cluster)
  if (rp.all) {
    for (int i = rank * CL_NT + tid; i < S; i += NC * CL_NT) out[i] = i;
    return;
  }
  if (rank == 0) {
    for (int i = tid; i < n_sink; i += CL_NT) out[i] = i;
    for (int i = tid; i < W; i += CL_NT) out[B1 - W + i] = (int32_t)(S - W + i);
  }
  if (ntop <= 0 && !pooled_out) return;

  // This CTA's window of the row-group sums: padded coordinate u holds position
  // p0 + u - h, at ps_pad(u).  The per-thread phases below are loops over a
  // thread's E positions, kept rolled: straight-line code of this length does
  // not stay in the instruction cache, and every warp runs it once.
  const int Uloc = PC + 2 * E;
  {
    const float* sc = scores + (size_t)pair * RG * Ls;
    if (RG == 1) {
      // one asynchronous 4-byte copy per entry: every copy of a thread in flight at once
      for (int u = tid; u < Uloc; u += CL_NT) {
        const int j = p0 + u - h;
        if (j >= 0 && j < L) cp_async_4(smem_u32(&xs[ps_pad(u)]), sc + j);
        else xs[ps_pad(u)] = __float_as_uint(neg_inf());
      }
      cp_async_commit();
      cp_async_wait_all();
    } else {
      // several row groups: their log2 sums are added up on the way
      for (int u0 = tid; u0 < Uloc; u0 += 8 * CL_NT) {
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int j = p0 + u0 + t * CL_NT - h;
          v[t] = (u0 + t * CL_NT < Uloc && j >= 0 && j < L) ? __ldg(sc + j) : neg_inf();
        }
        for (int r = 1; r < RG; ++r) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int j = p0 + u0 + t * CL_NT - h;
            if (u0 + t * CL_NT < Uloc && j >= 0 && j < L) v[t] = log2_add(v[t], __ldg(sc + (size_t)r * Ls + j));
          }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int u = u0 + t * CL_NT;
          if (u < Uloc) xs[ps_pad(u)] = __float_as_uint(v[t]);
        }
      }
    }
  }
  __syncthreads();

  // max-pool of outputs [a, a + E) (the right prefix maxima wait in ko, the
  // pooled values replace them), and the runs of equal pooled values among this
  // thread's candidates (positions >= n_sink): a max-pool this wide leaves about
  // two runs per 32 positions, so the passes below walk runs, not positions
  const int al = tid * E, a = p0 + al;
  const bool mine = a < L;
  const int cnt_i = mine ? min(E, L - a) : 0;       // this thread's positions [a, a + cnt_i)
  const int i_lo = mine ? max(0, n_sink - a) : 0;   // its candidates start here
  // the pooled log2 score of position a + i sits at kr[kx(i)] (a padded run of ko)
  uint32_t* ko = xs + cl_key_words(h);
  uint32_t* kr = ko + ps_pad(al);
  const int alo = al & 31;
  auto kx = [alo](int i) { return i + ((alo + i) >> 5); };
  uint32_t runs = 0u;                               // bit i: candidate position a + i starts a run of equal values
  if (mine) {
    float m;
    float l = neg_inf();
    if (E == 32) {
      // blocks of 32 window entries are padded rows of 33 words: the left block
      // is row tid (entries 0-30), the middle row tid's entry 31 and row tid + 1
      // (0-30), the right row tid + 1's entry 31 and row tid + 2 (0-29)
      const uint32_t* r0 = xs + 33 * tid;
      const uint32_t* r1 = r0 + 33;
      const uint32_t* r2 = r0 + 66;
      float m0 = __uint_as_float(r0[31]), m1 = neg_inf();
      for (int k = 0; k < 30; k += 2) {
        m0 = fmaxf(m0, __uint_as_float(r1[k]));
        m1 = fmaxf(m1, __uint_as_float(r1[k + 1]));
      }
      m = fmax3(m0, m1, __uint_as_float(r1[30]));
      float r = __uint_as_float(r1[31]);
      kr[0] = __float_as_uint(neg_inf());
      for (int i = 1; i < 32; ++i) {
        kr[i] = __float_as_uint(r);
        r = fmaxf(r, __uint_as_float(r2[i - 1]));
      }
      uint32_t pnext = 0u;                          // pooled value bits of position i + 1
      for (int i = 31; i >= 0; --i) {
        const uint32_t pb = __float_as_uint(fmax3(__uint_as_float(kr[i]), l, m));
        kr[i] = pb;
        runs |= (pb != pnext ? 2u : 0u) << i;       // position i + 1 starts a run
        pnext = pb;
        if (i > 0) l = fmaxf(l, __uint_as_float(r0[i - 1]));
      }
    } else {
      auto X = [&](int u) { return __uint_as_float(xs[ps_pad(u)]); };
      float m0 = neg_inf(), m1 = neg_inf();
      for (int i = 0; i < E; i += 2) {
        m0 = fmaxf(m0, X(al + E - 1 + i));
        if (i + 1 < E) m1 = fmaxf(m1, X(al + E + i));
      }
      m = fmaxf(m0, m1);
      float r = neg_inf();
      for (int i = 0; i < E; ++i) {
        kr[kx(i)] = __float_as_uint(r);
        r = fmaxf(r, X(al + 2 * E - 1 + i));
      }
      uint32_t pnext = 0u;
      for (int i = E - 1; i >= 0; --i) {
        const uint32_t pb = __float_as_uint(fmax3(__uint_as_float(kr[kx(i)]), l, m));
        kr[kx(i)] = pb;
        runs |= (pb != pnext ? 2u : 0u) << i;
        pnext = pb;
        if (i > 0) l = fmaxf(l, X(al + i - 1));
      }
    }
  }
  if (pooled_out && mine) {
    float* po = pooled_out + (size_t)pair * Ls;
    for (int i = 0; i < cnt_i; ++i) po[a + i] = exp2f(__uint_as_float(kr[kx(i)]));
  }
  // runs within [i_lo, cnt_i), the first one starting at i_lo
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  {
    const uint32_t span = i_lo >= cnt_i ? 0u : (cnt_i >= 32 ? 0xffffffffu : ((1u << cnt_i) - 1u)) & ~((1u << i_lo) - 1u);
    runs = (runs | (i_lo < cnt_i ? 1u << i_lo : 0u)) & span;
    for (uint32_t rb = runs; rb; rb &= rb - 1u) {
      const uint32_t key = f2key(__uint_as_float(kr[kx(__ffs(rb) - 1)]));
      kmn = min(kmn, key);
      kmx = max(kmx, key);
    }
  }
  // the order-preserving key of position a + i
  auto key_at = [&](int i) { return f2key(__uint_as_float(kr[kx(i)])); };
  // the run starting at bit i of `rb` (lowest set bit) ends at the next set bit, or at cnt_i
  auto run_end = [&](uint32_t rest) { return rest ? __ffs(rest) - 1 : cnt_i; };
  if (ntop <= 0) return;                            // (the pooled scores were written above)
  if (ntop >= L - n_sink) {
    for (int i = i_lo; i < cnt_i; ++i) out[a + i] = a + i;
    return;
  }

  // ---- key range of the cluster
  kmn = __reduce_min_sync(0xffffffffu, kmn);
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  if (lane == 0) {
    cs.wmin[warp] = kmn;
    cs.wmax[warp] = kmx;
  }
  for (int i = tid; i < PS_NB; i += CL_NT) cs.hist[i] = 0u;
  cs.taken[tid] = 0u;
  if (tid < CL_MAXNC) cs.ctk[tid] = 0u;
  if (tid == 0) cs.sh[3] = 0;
  __syncthreads();
  if (tid == 0) {
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int w = 0; w < CL_NT / 32; ++w) {
      lo = min(lo, cs.wmin[w]);
      hi = max(hi, cs.wmax[w]);
    }
    cs.mm[0] = lo;
    cs.mm[1] = hi;
  }
  cluster_sync();                                   // (1) every CTA's range is published
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int c = 0; c < NC; ++c) {
    lo = min(lo, ld_cluster_u32(mapa(smem_u32(&cs.mm[0]), (uint32_t)c)));
    hi = max(hi, ld_cluster_u32(mapa(smem_u32(&cs.mm[1]), (uint32_t)c)));
  }
  auto kval = [](uint32_t key) { return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key); };
  const float vlo = kval(lo), width = kval(hi) - vlo;
  const float inv = (width > 0.f && isfinite(width)) ? __fdividef((float)PS_NB, width) : 0.f;
  auto bucket = [&](uint32_t key) { return max(0, min(PS_NB - 1, (int)((kval(key) - vlo) * inv))); };
  bool use_radix = inv == 0.f;
  int bb = 0, need = 0, m = 0;
  if (!use_radix) {
    // ---- histogram: one count per run of equal buckets along this thread's positions
    {
      for (uint32_t rb = runs; rb;) {
        const int i = __ffs(rb) - 1;
        rb &= rb - 1u;
        atomicAdd(&cs.hist[bucket(key_at(i))], (uint32_t)(run_end(rb) - i));
      }
    }
    __syncthreads();
    cluster_sync();                                 // (2) every CTA's histogram is complete
    for (int q = tid; q < PS_NB / 4; q += CL_NT) {
      uint4 acc = make_uint4(0u, 0u, 0u, 0u);
      for (int c = 0; c < NC; ++c) {
        const uint4 v = ld_cluster_v4(mapa(smem_u32(&cs.hist[4 * q]), (uint32_t)c));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      *reinterpret_cast<uint4*>(&cs.ghist[4 * q]) = acc;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds buckets 32l .. 32l+31; counts from the top bucket down find the
      // lane holding the ntop-th largest key (exactly one: ntop < the candidates),
      // then suffix sums over that lane's 32 buckets, one per lane, the bucket
      const uint4* h4 = reinterpret_cast<const uint4*>(&cs.ghist[32 * lane]);
      uint32_t sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = h4[q];
        sum += v.x + v.y + v.z + v.w;
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      const uint32_t above = incl - sum;
      const unsigned cross = __ballot_sync(0xffffffffu, above < (uint32_t)ntop && incl >= (uint32_t)ntop);
      const int lx = __ffs(cross) - 1;
      const uint32_t above_x = __shfl_sync(0xffffffffu, above, lx);
      const uint32_t ck = cs.ghist[32 * lx + lane];
      uint32_t sk = ck;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, sk, o);
        if (lane + o < 32) sk += t;
      }
      const uint32_t abv = above_x + sk - ck;
      if (abv < (uint32_t)ntop && abv + ck >= (uint32_t)ntop) {
        cs.sh[0] = 32 * lx + lane;
        cs.sh[1] = (int)((uint32_t)ntop - abv);
        cs.sh[2] = (int)ck;
      }
    }
    __syncthreads();
    bb = cs.sh[0];
    need = cs.sh[1];
    m = cs.sh[2];
    if (need < m && m > CL_MAXM) use_radix = true;   // the same in every CTA
  }
  if (!use_radix) {
    // ---- this CTA's certainly taken positions and its members of a split bucket
    const bool split = need < m;
    uint32_t cert = 0u;
    for (uint32_t rb = runs; rb;) {
      const int i = __ffs(rb) - 1;
      rb &= rb - 1u;
      const int e = run_end(rb);                    // positions [a + i, a + e) share one key
      const uint32_t key = key_at(i);
      const int bk = bucket(key);
      if (bk > bb || (bk == bb && !split)) {
        cert |= (e - i >= 32 ? 0xffffffffu : ((1u << (e - i)) - 1u)) << i;
      } else if (bk == bb) {
        const int base = atomicAdd(&cs.sh[3], e - i);
        for (int t = i; t < e; ++t) cs.memb[base + t - i] = make_uint2(key, (uint32_t)(a + t));
      }
    }
    const uint32_t wc = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(cert));
    if (lane == 0) cs.wsum[warp] = wc;
    __syncthreads();
    if (tid == 0) {
      uint32_t c = 0;
#pragma unroll
      for (int w = 0; w < CL_NT / 32; ++w) c += cs.wsum[w];
      cs.cnt[0] = c;
      cs.cnt[1] = (uint32_t)cs.sh[3];
    }
    cluster_sync();                                 // (3) counts and member lists are published
    if (warp == 0) {
      // lane c < NC fetches CTA c's counts; the members' start in CTA order by a scan
      uint32_t cc = 0u, mc = 0u;
      if (lane < NC) {
        cc = ld_cluster_u32(mapa(smem_u32(&cs.cnt[0]), (uint32_t)lane));
        mc = ld_cluster_u32(mapa(smem_u32(&cs.cnt[1]), (uint32_t)lane));
      }
      uint32_t inc = mc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (lane < NC) {
        cs.msv[lane] = inc - mc;
        cs.certv[lane] = cc;
      }
      if (lane == 31) cs.msv[CL_MAXNC] = inc;     // every member of the cluster
    }
    __syncthreads();
    const uint32_t mtot = cs.msv[CL_MAXNC];
    const uint32_t* ms = cs.msv;
    auto cta_of = [&](uint32_t i) {
      int c = 0;
      for (int u = 1; u < NC; ++u) c = i >= ms[u] ? u : c;
      return c;
    };
    // a taken member of the split bucket counts for its CTA, and marks its bit here
    auto take = [&](uint32_t i, uint32_t pos) {
      const int c = cta_of(i);
      atomicAdd(&cs.ctk[c], 1u);
      if (c == rank) {
        const int lp = (int)pos - p0;               // this CTA's local position
        atomicOr(&cs.taken[lp >> 5], 1u << (lp & 31));
      }
    };
    if (split) {
      // every member of the cluster, in CTA order, then each one's rank among them
      // (larger key first, equal keys by position)
      for (uint32_t i = tid; i < mtot; i += CL_NT) {
        const int c = cta_of(i);
        const uint32_t ad = mapa(smem_u32(&cs.memb[i - ms[c]]), (uint32_t)c);
        cs.allm[i] = make_uint2(ld_cluster_u32(ad), ld_cluster_u32(ad + 4u));
      }
      __syncthreads();
      if (mtot <= CL_NT / 4) {
        // four threads per member, each against a quarter of the others
        const uint32_t i = (uint32_t)tid >> 2, qd = (uint32_t)tid & 3u;
        uint2 me = make_uint2(0u, 0u);
        int rk = 0;
        if (i < mtot) {
          me = cs.allm[i];
          for (uint32_t u = qd; u < mtot; u += 4) {
            const uint2 o = cs.allm[u];
            rk += (o.x > me.x) || (o.x == me.x && o.y < me.y);
          }
        }
        rk += __shfl_xor_sync(0xffffffffu, rk, 1);
        rk += __shfl_xor_sync(0xffffffffu, rk, 2);
        if (i < mtot && qd == 0 && rk < need) take(i, me.y);
      } else {
        for (uint32_t i = tid; i < mtot; i += CL_NT) {
          const uint2 me = cs.allm[i];
          int rk = 0;
          for (uint32_t u = 0; u < mtot; ++u) {
            const uint2 o = cs.allm[u];
            rk += (o.x > me.x) || (o.x == me.x && o.y < me.y);
          }
          if (rk < need) take(i, me.y);
        }
      }
      __syncthreads();
    }
    // taken positions of the CTAs before this one, then this CTA's in ascending order
    int pos = n_sink;
    for (int c = 0; c < rank; ++c) pos += (int)cs.certv[c] + (split ? (int)cs.ctk[c] : 0);
    uint32_t tk = cert;
    if (split && cnt_i > 0) {
      // bits [al, al + E) of the taken map (at most two words)
      const uint64_t w2 = ((uint64_t)cs.taken[min((al >> 5) + 1, CL_NT - 1)] << 32) | cs.taken[al >> 5];
      tk |= (uint32_t)(w2 >> (al & 31)) & (E == 32 ? 0xffffffffu : ((1u << E) - 1u));
    }
    const uint32_t cnt = (uint32_t)__popc(tk);
    uint32_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) cs.wsum[warp] = inc;
    __syncthreads();
    pos += (int)(inc - cnt);
    for (int w = 0; w < warp; ++w) pos += (int)cs.wsum[w];
    const int pend = n_sink + ntop;                 // (exactly ntop are taken; the bound guards the row)
    for (uint32_t bits = tk; bits && pos < pend; bits &= bits - 1u) out[pos++] = a + (__ffs(bits) - 1);
    cluster_sync();                                 // (4) no CTA leaves while another reads its shared memory
    return;
  }

  // ---- radix fallback: the keys in global scratch, CTA 0 selects over them
  uint32_t* ks = key_scratch + (size_t)pair * Ls;
  for (int i = i_lo; i < cnt_i; ++i) ks[a + i] = key_at(i);
  cluster_sync();                                   // keys visible; every remote read done
  if (rank != 0) return;
  uint32_t prefix = 0, mask = 0;
  int k = ntop;
  for (int shift = 24; shift >= 0; shift -= 8) {
    cs.ghist[tid] = 0u;                             // (CL_NT == 256 digits)
    __syncthreads();
    for (int j = n_sink + tid; j < L; j += CL_NT) {
      const uint32_t key = ks[j];
      if ((key & mask) == prefix) atomicAdd(&cs.ghist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      int c[8];
      int sum = 0;
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        c[u] = (int)cs.ghist[lane * 8 + u];
        sum += c[u];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      int above = incl - sum;
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        if (above < k && above + c[u] >= k) {
          cs.sh[4] = lane * 8 + u;
          cs.sh[5] = k - above;
        }
        above += c[u];
      }
    }
    __syncthreads();
    prefix |= (uint32_t)cs.sh[4] << shift;
    mask |= 255u << shift;
    k = cs.sh[5];
    __syncthreads();
  }
  // keys > T are taken, and the first k keys equal to T in position order
  const uint32_t T = prefix;
  int pos = n_sink, eq_taken = 0;
  for (int base = n_sink; base < L; base += CL_NT) {
    const int j = base + tid;
    const uint32_t key = j < L ? ks[j] : 0u;
    const bool gt = j < L && key > T, eq = j < L && key == T;
    int eq_tot, take_tot;
    const int eq_before = cl_excl_scan(eq, cs.wsum, eq_tot);
    const bool take = gt || (eq && eq_taken + eq_before < k);
    const int tpos = cl_excl_scan(take, cs.wsum, take_tot);
    if (take && pos + tpos < n_sink + ntop) out[pos + tpos] = j;
    pos += take_tot;
    eq_taken += eq_tot;
  }
}

// K_c[i] = K[keep[i]], V_c[i] = V[keep[i]].
__global__ void __launch_bounds__(256) snap_compact_kernel(const bf16* k, const bf16* v, int64_t cap,
                                                           const int32_t* keep, int64_t keep_ld, int64_t B1_max,
                                                           bf16* ko, bf16* vo, int64_t out_cap, const int32_t* S_rows,
                                                           const int32_t* B1_rows, int64_t S_max, int Hkv, int W,
                                                           int n_sink, const int32_t* bt, int64_t bt_stride,
                                                           int64_t num_pages, int page_shift) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  const int64_t B1 = row_plan(S_rows, B1_rows, pair / Hkv, S_max, B1_max, W, n_sink).B1;
  const int b = pair / Hkv, hk = pair - b * Hkv;
  for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x) {
    const int64_t row = (int64_t)blockIdx.x * 32 + i / 16;
    const int ch = i % 16;
    if (row >= B1) break;
    const int64_t src = min(max((int64_t)keep[(size_t)pair * keep_ld + row], (int64_t)0), cap - 1);
    // dense: row src of the pair; paged: slot src % page of page bt[b, src / page] (cap = rows a row's pages cover)
    size_t e;
    if (bt) {
      const int64_t pg = min(max((int64_t)bt[(size_t)b * bt_stride + (src >> page_shift)], (int64_t)0), num_pages - 1);
      e = (((size_t)pg * Hkv + hk) << page_shift) + (size_t)(src & ((1 << page_shift) - 1));
    } else {
      e = (size_t)pair * cap + src;
    }
    const uint4 kv = *reinterpret_cast<const uint4*>(k + e * HD + ch * 8);
    const uint4 vv = *reinterpret_cast<const uint4*>(v + e * HD + ch * 8);
    *reinterpret_cast<uint4*>(ko + ((size_t)pair * out_cap + row) * HD + ch * 8) = kv;
    *reinterpret_cast<uint4*>(vo + ((size_t)pair * out_cap + row) * HD + ch * 8) = vv;
  }
}

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

int snap_num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  });
  return n;
}

}  // namespace

// Keys per work item of the score passes: P_CHUNK, halved (down to two tiles)
// while the pass-1 items would not cover the GPU's 152 SMs; a function of the
// shape alone, so the workspace query and the launch agree on any device.
int snap_chunk_keys(int64_t pairs, int64_t S, int64_t rg1) {
  int c = P_CHUNK;
  while (c > 2 * T_KEYS && pairs * rg1 * ((S + c - 1) / c) < 152) c >>= 1;
  return c;
}

size_t snap_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t S, int32_t W) {
  const int64_t pairs = (int64_t)B * Hkv;
  const int G = Hq / Hkv;
  const int64_t R = (int64_t)G * W;
  const int64_t RG = (R + P2_ROWS - 1) / P2_ROWS;
  const int64_t L = std::max<int64_t>(S - W, 0);
  const int64_t p1 = R > P1_ROWS ? 2 * P1_ROWS : P1_ROWS;
  const int chunk = snap_chunk_keys(pairs, S, (R + p1 - 1) / p1);
  const int64_t nchunk1 = (S + chunk - 1) / chunk;
  return al256((size_t)pairs * R * nchunk1 * sizeof(float2)) + al256((size_t)pairs * RG * L * sizeof(float)) +
         al256((size_t)pairs * L * sizeof(float));
}

int snap_pass2_rows(int32_t G, int32_t W) { return std::min(P2_ROWS, (G * W + 31) & ~31); }
int snap_pass1_rows(int32_t G, int32_t W) { return G * W > P1_ROWS ? 2 * P1_ROWS : P1_ROWS; }

// CTAs of the cluster pool + select for prefix length L and half window h:
// 1..max_nc when it applies (the separate pool + select takes longer prefixes
// and windows wider than 63)
int pool_select_cl_ctas(int64_t L, int h, int max_nc) {
  const int E = h + 1;
  if (L <= 0 || E > 32) return 0;
  const int64_t nq = (L + E - 1) / E;
  const int64_t nc = (nq + CL_NT - 1) / CL_NT;
  return nc <= max_nc ? (int)nc : 0;
}


// Launch as clusters of nc CTAs along x, with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, unsigned nc,
                               cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

cudaError_t snap_launch(const SnapArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmQ1, const CUtensorMap* tmQ2,
                        cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess, cl_attr_err = cudaSuccess;
  static int cl_max = 8;                          // largest cluster of the pool + select
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(snap_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, T_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(snap_pass_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, T_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(snap_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, T_SMEM);
    // (the window and keys of half width 31 plus the static select state pass the default 48 KB)
    cl_attr_err = cudaFuncSetAttribute(snap_pool_select_cl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       cl_smem_words(31) * 4);
    // clusters of up to 16 CTAs where the GPU schedules them (prefixes of up to
    // 4096 pooling groups in one kernel), else the portable 8
    if (cl_attr_err == cudaSuccess &&
        cudaFuncSetAttribute(snap_pool_select_cl_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CL_MAXNC, 1, 1);
      cfg.blockDim = dim3(CL_NT, 1, 1);
      cfg.dynamicSmemBytes = (size_t)cl_smem_words(31) * 4u;
      int cmax = 0;
      if (cudaOccupancyMaxPotentialClusterSize(&cmax, snap_pool_select_cl_kernel, &cfg) == cudaSuccess)
        cl_max = std::max(8, std::min(cmax, CL_MAXNC));
      else
        cudaGetLastError();                       // (a refused query leaves no error behind)
    } else if (cl_attr_err == cudaSuccess) {
      cudaGetLastError();
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int pairs = a.B * a.Hkv;
  // (per-row lengths: S and B1 are the maxima, W the window of rows longer than it)
  const bool ragged = a.S_rows != nullptr || a.B1_rows != nullptr || a.bt != nullptr;
  const int W = ragged ? a.W : (int)std::min<int64_t>(a.W, a.S);
  const int64_t L = std::max<int64_t>(a.S - W, 0);
  const bool keep_all = !ragged && (a.B1 >= a.S || L <= 0);
  const int n_sink = (int)std::max<int64_t>(0, std::min<int64_t>(a.n_sink, L));
  if (!keep_all && L > 0) {
    PassArgs p;
    p.S = a.S;
    p.L = L;
    p.S_rows = a.S_rows;
    p.bt = a.bt;
    p.bt_stride = a.bt_stride;
    p.num_pages = a.num_pages;
    p.page_shift = a.page_shift;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.G;
    p.W = W;
    p.R = a.G * W;
    p.p1rows = snap_pass1_rows(a.G, W);
    p.RG1 = (p.R + p.p1rows - 1) / p.p1rows;
    p.RG2 = (p.R + P2_ROWS - 1) / P2_ROWS;
    p.nq2 = snap_pass2_rows(a.G, W);
    p.chunk = snap_chunk_keys(pairs, a.S, p.RG1);
    p.nchunk1 = (int)((a.S + p.chunk - 1) / p.chunk);
    p.scale_log2 = a.scale_log2;
    uint8_t* w = reinterpret_cast<uint8_t*>(a.ws);
    p.stats = reinterpret_cast<float2*>(w);
    w += al256((size_t)pairs * p.R * p.nchunk1 * sizeof(float2));
    p.scores = reinterpret_cast<float*>(w);
    w += al256((size_t)pairs * p.RG2 * L * sizeof(float));
    float* pooled_log = reinterpret_cast<float*>(w);   // log2 pooled scores (separate pool + select)

    p.pairs = pairs;
    p.nchunk2 = (int)((L + p.chunk - 1) / p.chunk);
    // persistent grids: one CTA per SM (the ring and Q tile fill the shared memory)
    const int items1 = pairs * p.RG1 * p.nchunk1, items2 = pairs * p.RG2 * p.nchunk2;
    cudaError_t e = launch_pdl(p.p1rows > P1_ROWS ? snap_pass_kernel<1, true> : snap_pass_kernel<1>,
                               dim3((unsigned)std::min(items1, snap_num_sms())), dim3(T_NT),
                               T_SMEM, st, *tmK, *tmQ1, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(snap_pass_kernel<2>, dim3((unsigned)std::min(items2, snap_num_sms())), dim3(T_NT), T_SMEM, st,
                   *tmK, *tmQ2, p);
    if (e != cudaSuccess) return e;
    const int half = (int)(a.pool / 2);
    const int cl_nc = cl_attr_err == cudaSuccess ? pool_select_cl_ctas(L, half, cl_max) : 0;
    if (cl_nc > 0) {
      e = launch_cluster_pdl(snap_pool_select_cl_kernel, dim3((unsigned)cl_nc, pairs), dim3(CL_NT),
                             (size_t)cl_smem_words(half) * 4u, (unsigned)cl_nc, st, (const float*)p.scores, (int)p.RG2,
                             (int64_t)L, half, (int64_t)a.S, (int)W, (int)a.n_sink, (int64_t)a.B1, a.keep,
                             (int64_t)a.keep_ld, a.pooled_out, a.S_rows, a.B1_rows, (int)a.Hkv, cl_nc,
                             reinterpret_cast<uint32_t*>(pooled_log));
      if (e != cudaSuccess) return e;
    } else {
      e = launch_pdl(snap_pool_kernel, dim3((unsigned)((L + POOL_TILE - 1) / POOL_TILE), pairs), dim3(256), 0, st,
                     (const float*)p.scores, (int)p.RG2, (int64_t)L, half, pooled_log, a.pooled_out, a.S_rows,
                     (int64_t)a.S, (int)a.Hkv, (int)W);
      if (e != cudaSuccess) return e;
      e = launch_pdl(snap_select_kernel, dim3(pairs), dim3(SEL_NT), 0, st, (const float*)pooled_log, (int64_t)L,
                     (int64_t)a.S, (int)W, (int)a.n_sink, (int64_t)a.B1, a.keep, (int64_t)a.keep_ld, a.S_rows,
                     a.B1_rows, (int)a.Hkv);
      if (e != cudaSuccess) return e;
    }
  } else {
    // every token of every row kept: keep = 0..S_b-1
    cudaError_t e = launch_pdl(snap_select_kernel, dim3(pairs), dim3(SEL_NT), 0, st, (const float*)nullptr, (int64_t)0,
                               (int64_t)a.S, (int)W, n_sink, (int64_t)a.B1, a.keep, (int64_t)a.keep_ld, a.S_rows,
                               a.B1_rows, (int)a.Hkv);
    if (e != cudaSuccess) return e;
  }
  if (a.k_out) {
    cudaError_t e = launch_pdl(snap_compact_kernel, dim3((unsigned)((a.B1 + 31) / 32), pairs), dim3(256), 0, st,
                               reinterpret_cast<const bf16*>(a.k), reinterpret_cast<const bf16*>(a.v), (int64_t)a.cap,
                               (const int32_t*)a.keep, (int64_t)a.keep_ld, (int64_t)a.B1,
                               reinterpret_cast<bf16*>(a.k_out), reinterpret_cast<bf16*>(a.v_out), (int64_t)a.out_cap,
                               a.S_rows, a.B1_rows, (int64_t)a.S, (int)a.Hkv, (int)W, (int)a.n_sink, a.bt,
                               (int64_t)a.bt_stride, (int64_t)a.num_pages, (int)a.page_shift);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

unsigned int snap_take_device_error() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_snap_err, sizeof(v)) != cudaSuccess) return ~0u;
  cudaMemcpyToSymbol(g_snap_err, &z, sizeof(z));
  return v;
}

}  // namespace rkv
