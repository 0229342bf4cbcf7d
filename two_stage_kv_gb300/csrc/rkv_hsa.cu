// Stage 2 of RocketKV: one Hybrid Sparse Attention decode step per launch,
// optionally fused with the append of the step's new key/value.
//
// Method: "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV
// Cache Compression" (papercache digest), section 方法细节, HSA steps 1-3 and
// Algorithm 1 (top-k1 channels of the group sum of |q|, sign of the group sum
// of q, sign-selected Kmax/Kmin page scores, top-k2 pages, exact attention over
// the selected pages; the Kmax/Kmin store is updated when a key is generated);
// RocketKV-MT for the candidate-restricted variant.
//
// GB300 design.  One thread-block cluster of `ns` CTAs (256 threads each) per
// (batch row, KV head), ns chosen so the grid fits in one wave.  CTA r:
//   0. at launch prefetches, with one 2-D TMA box, every KT row (Kmax and Kmin
//      of all 128 channels) of its share of the blocks, [r*cpr, r*cpr + cpr);
//      the KT rows do not depend on the query, so the load overlaps step A
//      (shares wider than 128 blocks gather the chosen rows in step B instead);
//   A. loads the group's G query rows and forms sum|q| and sum q per channel in
//      fp32 with an error-free TwoSum check (an inexact sum sends the whole CTA
//      to an fp64 path, so the channel decision is the exact-arithmetic one),
//      then picks the top-k1 channels by rank (two threads count, for each
//      channel, the channels ahead of it);
//   B. folds the appended key into its block, scores its own blocks in fp32
//      and sends every score, and each warp's score bounds, to every CTA of
//      the cluster with st.async, counted on the receivers' mbarriers;
//   C. picks the top-k2 blocks and lists them in ascending order (every CTA of
//      the cluster computes the same list);
//   D. TMA-loads the K and V rows of its share of the blocks into 128-byte-
//      swizzled shared tiles (rows past n read as zero; one mbarrier per
//      block), computes S^T = K Q^T per 16-token step on bf16 mma.sync (tokens
//      on the M side, G <= 8 heads per 8-wide N tile), a CTA-wide softmax in
//      fp32, and O^T = V^T P^T with each warp owning 16 output dimensions (P
//      is split into bf16 hi + lo, so PV keeps ~16 mantissa bits);
//   E. sends its partial (max, sum, O) for each head with st.async to the CTA
//      that owns the head, whose mbarrier counts the bytes; the owner combines
//      the ns partials and writes fp32 outputs.
// Both top-k steps are exact (larger first, equal values: lower index).  For
// the blocks, a 256-bucket histogram over [min, max] finds the bucket holding the k-th value
// and only that bucket's members are ranked pairwise; a radix select on an
// order-preserving key takes over for degenerate value sets.  No global
// scratch and no atomics on the data path; the cross-CTA waits are one
// hardware cluster barrier at launch and bounded mbarrier waits.
#include "rkv_common.cuh"
#include "rkv_internal.h"

#include <algorithm>
#include <mutex>

namespace rkv {

static __device__ unsigned int g_hsa_err = 0;

namespace {

constexpr int NT = 256;                 // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int PART_STRIDE = HD + 2;     // O[128], max, sum
constexpr int MAX_ROUND_ROWS = 128;     // K/V rows staged per round (8 steps of 16 tokens)
constexpr uint32_t KT_TILE_BUDGET = 32 * 1024;
constexpr int NBUCKET = NT;             // one histogram bucket per thread
constexpr int MEMBER_MAX = 512;         // boundary-bucket members ranked pairwise

struct FixedSmem {
  bf16 qs[16][HD + 8];          // query rows (padded: conflict-free ldmatrix), rows >= G are zero
  bf16 knew[HD];                // appended key / value of this pair (e4m3 storage: its code values)
  uint8_t knew8[HD];            // e4m3 storage: codes of the appended key / value
  uint8_t vnew8[HD];
  bf16 vnew[HD];
  float qsel[HD];               // group-summed q of the kept channels, ascending channel
  int32_t rowoff[HD];           // KT row (0..2*HD) of each kept channel
  alignas(16) float asum[HD];   // sum_g |q_g| per channel (fp32, exact)
  float qbar32[HD];
  uint64_t akey64[HD];          // fp64 fallback
  double qbar64[HD];
  alignas(16) int32_t hist[4 * 256];   // bucket histogram; the radix fallback uses 4 x 256
  int32_t members[MEMBER_MAX];
  float wmin[NWARP], wmax[NWARP];
  alignas(16) int32_t wsum[2 * NWARP];
  int32_t misc[8];
  float wmaxh[NWARP][16];       // per-warp head maxima of a round
  float wsumh[NWARP][16];       // per-warp head probability sums of a round
  uint32_t pfrag[MAX_ROUND_ROWS / 16][2][4][32];   // P^T B fragments per 16-token step, head tile, hi/lo
  float mrun[16], lrun[16];
  uint64_t mbar[MAX_ROUND_ROWS / 8];    // one per staged block
  uint64_t ebar;                        // partials of the heads this CTA owns (phase E)
  uint64_t ktbar;                       // KT prefetch (phase B)
  uint64_t sbar;                        // every block score and score bound of the cluster (phase B)
  float2 rbound[8 * NWARP];             // (min, max) of the scores of each warp of each CTA
  uint32_t relig[MAX_ROUND_ROWS / 32];  // masked MT: candidate rows of the staged round
};

// Inverse of f2key.
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Block-wide exclusive scan of a flag.  Returns the prefix, writes the total.
__device__ __forceinline__ int scan1(bool f, int32_t* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    const int v = wsum[w];
    if (w < warp) pre += v;
    tot += v;
  }
  __syncthreads();
  total = tot;
  return pre + __popc(bal & ((1u << lane) - 1u));
}

// Exact top-k of keys[0, n) by MSB-first radix select on order-preserving keys
// (equal keys: lower index first); writes flag[0, n).
__device__ void radix_topk(const uint32_t* keys, int n, int k, uint8_t* flag, FixedSmem& fs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 4 * 256; i += NT) fs.hist[i] = 0;
  __syncthreads();
  uint32_t prefix = 0, mask = 0;
  int kk = k;
  for (int p = 0; p < 4; ++p) {
    const int shift = 24 - 8 * p;
    int32_t* h = fs.hist + 256 * p;
    for (int base = 0; base < n; base += NT) {
      const int j = base + tid;
      const uint32_t key = j < n ? keys[j] : 0u;
      const bool act = (j < n) && ((key & mask) == prefix);
      const unsigned am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const unsigned d = (key >> shift) & 255u;
        const unsigned m = __match_any_sync(am, d);
        if (lane == __ffs(m) - 1) atomicAdd(&h[d], __popc(m));
      }
    }
    __syncthreads();
    if (warp == 0) {
      int cnt[8];
      int s = 0;
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        cnt[u] = h[lane * 8 + u];
        s += cnt[u];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      int above = incl - s;
#pragma unroll
      for (int u = 7; u >= 0; --u) {
        if (above < kk && above + cnt[u] >= kk) {
          fs.misc[4] = lane * 8 + u;
          fs.misc[5] = kk - above;
        }
        above += cnt[u];
      }
    }
    __syncthreads();
    prefix |= (uint32_t)fs.misc[4] << shift;
    mask |= 255u << shift;
    kk = fs.misc[5];
    __syncthreads();
  }
  const uint32_t T = prefix;
  int eq_taken = 0;
  for (int base = 0; base < n; base += NT) {
    const int j = base + tid;
    const uint32_t key = j < n ? keys[j] : 0u;
    const bool eq = (j < n) && key == T;
    int eq_tot;
    const int eq_before = scan1(eq, fs.wsum, eq_tot);
    if (j < n) flag[j] = (key > T) || (eq && eq_taken + eq_before < kk);
    eq_taken += eq_tot;
  }
  __syncthreads();
}

// Exact top-k (0 < k < n) of vals[0, n), listed: sel[0, k) = the indices of
// the k largest values in ascending order, equal values taken in ascending
// index order.  mn / mx are the minimum and maximum of vals.
//
// A 256-bucket histogram over [mn, mx] locates the bucket holding the k-th
// value; every warp reads the whole histogram and finds that bucket on its
// own (no block barrier for the search).  Usually that bucket is taken whole
// and the chosen values are simply those in it or above; otherwise its
// members are ranked pairwise.  Degenerate value sets (equal, non-finite
// range, a crowded boundary bucket) go to a radix select on order-preserving
// keys, which overwrites vals.  fs.hist must be zero on entry and fs.misc[3]
// zero; both are left dirty (one call per launch).
__device__ void topk_list(float* vals, int n, int k, float mn, float mx, uint8_t* flag, int32_t* sel, FixedSmem& fs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float width = mx - mn;
  bool fallback = !(width > 0.f) || !isfinite(width);
  // (any monotone map of the scores to buckets gives the same exact selection,
  // so the scale need not be correctly rounded)
  const float inv = fallback ? 0.f : __fdividef((float)NBUCKET, width);
  // (clamped at both ends: -inf / +inf entries of the masked multi-turn reading)
  auto bucket = [&](float s) { return max(0, min(NBUCKET - 1, (int)((s - mn) * inv))); };
  int bb = 0, need = 0, m = 0;
  if (!fallback) {
    if (n <= 2 * NT) {
      // both of this thread's scores read before either count is added
      const float v0 = tid < n ? vals[tid] : 0.f, v1 = tid + NT < n ? vals[tid + NT] : 0.f;
      if (tid < n) atomicAdd(&fs.hist[bucket(v0)], 1);
      if (tid + NT < n) atomicAdd(&fs.hist[bucket(v1)], 1);
    } else {
      for (int j = tid; j < n; j += NT) atomicAdd(&fs.hist[bucket(vals[j])], 1);
    }
    __syncthreads();
    // lane l holds buckets 8l .. 8l+7; counts from the top bucket down
    const int4 h0 = *reinterpret_cast<const int4*>(&fs.hist[8 * lane]);
    const int4 h1 = *reinterpret_cast<const int4*>(&fs.hist[8 * lane + 4]);
    const int cnt[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    int s = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) s += cnt[u];
    int incl = s;   // this lane's buckets and every higher lane's
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    int above = incl - s;
    int found = -1, fneed = 0, fm = 0;
#pragma unroll
    for (int u = 7; u >= 0; --u) {
      if (above < k && above + cnt[u] >= k) {
        found = 8 * lane + u;
        fneed = k - above;
        fm = cnt[u];
      }
      above += cnt[u];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, found >= 0)) - 1;   // exactly one lane
    bb = __shfl_sync(0xffffffffu, found, src);
    need = __shfl_sync(0xffffffffu, fneed, src);
    m = __shfl_sync(0xffffffffu, fm, src);
    fallback = m > MEMBER_MAX;                      // the same in every warp
  }
  if (!fallback) {
    if (need < m) {
      // the boundary bucket is split: rank its members
      for (int j = tid; j < n; j += NT)
        if (bucket(vals[j]) == bb) fs.members[atomicAdd(&fs.misc[3], 1)] = j;
      __syncthreads();
      for (int i = tid; i < m; i += NT) {
        const int j = fs.members[i];
        const float sv = vals[j];
        int rk = 0;
        for (int i2 = 0; i2 < m; ++i2) {
          const int j2 = fs.members[i2];
          const float s2 = vals[j2];
          rk += (s2 > sv) || (s2 == sv && j2 < j);
        }
        flag[j] = rk < need ? 1 : 0;
      }
      __syncthreads();
    }
    auto chosen = [&](int j) -> bool {
      if (j >= n) return false;
      const int bk = bucket(vals[j]);
      return bk > bb || (bk == bb && (need == m || flag[j] != 0));
    };
    if (n <= 2 * NT) {
      // thread t lists blocks 2t and 2t+1: in-warp positions from two ballots,
      // warp offsets from one exchange
      const bool f0 = chosen(2 * tid), f1 = chosen(2 * tid + 1);
      const unsigned b0 = __ballot_sync(0xffffffffu, f0), b1 = __ballot_sync(0xffffffffu, f1);
      const unsigned lt = (1u << lane) - 1u;
      if (lane == 0) fs.wsum[warp] = __popc(b0) + __popc(b1);
      __syncthreads();
      const int4 w0 = *reinterpret_cast<const int4*>(&fs.wsum[0]);
      const int4 w1 = *reinterpret_cast<const int4*>(&fs.wsum[4]);
      const int pre = __popc(b0 & lt) + __popc(b1 & lt) + (warp > 0 ? w0.x : 0) + (warp > 1 ? w0.y : 0) +
                      (warp > 2 ? w0.z : 0) + (warp > 3 ? w0.w : 0) + (warp > 4 ? w1.x : 0) + (warp > 5 ? w1.y : 0) +
                      (warp > 6 ? w1.z : 0);
      if (f0 && pre < k) sel[pre] = 2 * tid;
      if (f1 && pre + (int)f0 < k) sel[pre + (int)f0] = 2 * tid + 1;
    } else {
      int out = 0;
      for (int base = 0; base < n; base += NT) {
        const int j = base + tid;
        const bool f = chosen(j);
        int tot;
        const int pre = scan1(f, fs.wsum, tot);
        if (f && out + pre < k) sel[out + pre] = j;
        out += tot;
      }
    }
  } else {
    uint32_t* keys = reinterpret_cast<uint32_t*>(vals);
    __syncthreads();
    for (int j = tid; j < n; j += NT) keys[j] = f2key(vals[j]);
    __syncthreads();
    radix_topk(keys, n, k, flag, fs);
    int out = 0;
    for (int base = 0; base < n; base += NT) {
      const int j = base + tid;
      const bool f = j < n && flag[j];
      int tot;
      const int pre = scan1(f, fs.wsum, tot);
      if (f && out + pre < k) sel[out + pre] = j;
      out += tot;
    }
  }
}

// Exact top-k (0 < k < n <= 2 * NT) of vals[0, n), listed: sel[0, k) = the
// indices of the k largest values in ascending order, equal values taken in
// ascending index order.  mn < mx are the finite minimum and maximum of the
// finite values (infinite values clamp to the end buckets).  Thread t owns
// blocks 2t and 2t+1 for the whole selection.
//   1. a 256-bucket histogram over [mn, mx] (any monotone map keeps the exact
//      order between buckets); every warp then finds the bucket holding the
//      k-th value on its own;
//   2. blocks above that bucket are chosen; when the bucket is split, each
//      warp lists its members (in block order) in shared memory;
//   3. every warp ranks all members itself (at most 64: one or two per lane),
//      so each thread knows the list position of its blocks without another
//      exchange, and writes them.
// Returns true when the list was written (three CTA barriers in all, the last
// one left to the caller).  Returns false for a split bucket of more than 64
// members, having written nothing and left fs.hist zero for the general select.
// fs.hist must be zero on entry.
__device__ bool topk_small(const float* vals, int n, int k, float mn, float mx, int32_t* sel, FixedSmem& fs) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // (any monotone map of the scores to buckets gives the same exact selection)
  const float inv = __fdividef((float)NBUCKET, mx - mn);
  const int j0 = 2 * tid;
  const bool ok0 = j0 < n, ok1 = j0 + 1 < n;
  float2 v = make_float2(0.f, 0.f);
  // (the score array holds n rounded up to 8 entries: the pair word stays inside it)
  if (ok0) v = *reinterpret_cast<const float2*>(vals + j0);
  const int b0 = ok0 ? max(0, min(NBUCKET - 1, (int)((v.x - mn) * inv))) : -1;
  const int b1 = ok1 ? max(0, min(NBUCKET - 1, (int)((v.y - mn) * inv))) : -1;
  if (ok0) atomicAdd(&fs.hist[b0], 1);
  if (ok1) atomicAdd(&fs.hist[b1], 1);
  __syncthreads();
  int bb, need, m;
  {
    // lane l holds buckets 8l .. 8l+7; counts from the top bucket down
    const int4 h0 = *reinterpret_cast<const int4*>(&fs.hist[8 * lane]);
    const int4 h1 = *reinterpret_cast<const int4*>(&fs.hist[8 * lane + 4]);
    const int cnt[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    int tot = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) tot += cnt[u];
    int incl = tot;   // this lane's buckets and every higher lane's
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    int above = incl - tot;
    int found = -1, fneed = 0, fm = 0;
#pragma unroll
    for (int u = 7; u >= 0; --u) {
      if (above < k && above + cnt[u] >= k) {
        found = 8 * lane + u;
        fneed = k - above;
        fm = cnt[u];
      }
      above += cnt[u];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, found >= 0)) - 1;   // exactly one lane
    bb = __shfl_sync(0xffffffffu, found, src);
    need = __shfl_sync(0xffffffffu, fneed, src);
    m = __shfl_sync(0xffffffffu, fm, src);
  }
  const bool split = need < m;             // the same in every warp
  if (split && m > 64) {
    __syncthreads();                       // every warp has read the histogram
    fs.hist[tid] = 0;
    __syncthreads();
    return false;
  }
  const unsigned lt = (1u << lane) - 1u;
  const bool c0 = b0 > bb || (b0 == bb && !split), c1 = b1 > bb || (b1 == bb && !split);
  const unsigned bc0 = __ballot_sync(0xffffffffu, c0), bc1 = __ballot_sync(0xffffffffu, c1);
  const bool m0 = split && b0 == bb, m1 = split && b1 == bb;
  int mp = 0;                              // this warp's members in lower lanes
  if (split) {
    const unsigned bm0 = __ballot_sync(0xffffffffu, m0), bm1 = __ballot_sync(0xffffffffu, m1);
    mp = __popc(bm0 & lt) + __popc(bm1 & lt);
    if (m0) fs.members[warp * 64 + mp] = j0;
    if (m1) fs.members[warp * 64 + mp + (m0 ? 1 : 0)] = j0 + 1;
    if (lane == 0) fs.wsum[NWARP + warp] = __popc(bm0) + __popc(bm1);
  }
  if (lane == 0) fs.wsum[warp] = __popc(bc0) + __popc(bc1);
  __syncthreads();
  int pre = __popc(bc0 & lt) + __popc(bc1 & lt);
  {
    const int4 w0 = *reinterpret_cast<const int4*>(&fs.wsum[0]);
    const int4 w1 = *reinterpret_cast<const int4*>(&fs.wsum[4]);
    pre += (warp > 0 ? w0.x : 0) + (warp > 1 ? w0.y : 0) + (warp > 2 ? w0.z : 0) + (warp > 3 ? w0.w : 0) +
           (warp > 4 ? w1.x : 0) + (warp > 5 ? w1.y : 0) + (warp > 6 ? w1.z : 0);
  }
  bool f0 = c0, f1 = c1;
  if (split) {
    // members in block order: warp w's list starts at ms[w]
    const int4 q0 = *reinterpret_cast<const int4*>(&fs.wsum[NWARP]);
    const int4 q1 = *reinterpret_cast<const int4*>(&fs.wsum[NWARP + 4]);
    const int mc[NWARP] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    int ms[NWARP];
    int acc = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
      ms[w] = acc;
      acc += mc[w];
    }
    // lane l ranks members l and l + 32 against every member
    int jm[2];
    float sm[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      int w = 0;
#pragma unroll
      for (int u = 1; u < NWARP; ++u) w = i >= ms[u] ? u : w;
      jm[h] = i < m ? fs.members[w * 64 + (i - ms[w])] : 0x7fffffff;
      sm[h] = i < m ? vals[jm[h]] : 0.f;
    }
    int rk[2] = {0, 0};
    for (int i2 = 0; i2 < m; ++i2) {
      const int sl = i2 & 31;
      const float s2 = __shfl_sync(0xffffffffu, i2 < 32 ? sm[0] : sm[1], sl);
      const int j2 = __shfl_sync(0xffffffffu, i2 < 32 ? jm[0] : jm[1], sl);
#pragma unroll
      for (int h = 0; h < 2; ++h) rk[h] += (s2 > sm[h]) || (s2 == sm[h] && j2 < jm[h]);
    }
    const unsigned win0 = __ballot_sync(0xffffffffu, lane < m && rk[0] < need);
    const unsigned win1 = __ballot_sync(0xffffffffu, lane + 32 < m && rk[1] < need);
    // chosen members before this thread's blocks (global member index < g)
    const int g = ms[warp] + mp;
    const int below = g <= 32 ? __popc(g == 32 ? win0 : (win0 & ((1u << g) - 1u)))
                              : __popc(win0) + __popc(g == 64 ? win1 : (win1 & ((1u << (g - 32)) - 1u)));
    pre += below;
    auto won = [&](int gi) { return gi < 32 ? ((win0 >> gi) & 1u) != 0 : ((win1 >> (gi - 32)) & 1u) != 0; };
    if (m0) f0 = won(g);
    if (m1) f1 = won(g + (m0 ? 1 : 0));
  }
  if (f0 && pre < k) sel[pre] = j0;
  if (f1 && pre + (int)f0 < k) sel[pre + (int)f0] = j0 + 1;
  return true;
}

// RAG: lengths read after the dependency wait (n_rows, or the call's n when
// n_rows is NULL); PG: K/V in pages of blk rows, [num_pages, Hkv, blk, D], found
// through a per-row block table (implies RAG); MK: the multi-turn reading over
// fixed blocks of the full cache, where only candidate rows (stage-1 survivors
// of the prompt, every row decoded after it) count: bounds, blocks without a
// candidate never chosen, the newest row's block always chosen, attention over
// candidate rows only.
// F8: k, v and kt hold e4m3 codes (value = code * the pair's scale); the
// bounds and scores are on code values, attention dequantizes through the
// logit and output scales.
template <bool MT, int NH, bool RAG, bool PG, bool MK = false, bool F8 = false, bool WF = false>
__global__ void __launch_bounds__(NT, 2) hsa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                           const __grid_constant__ CUtensorMap tmV,
                                                           const __grid_constant__ CUtensorMap tmKT,
                                                           const HsaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  FixedSmem& fs = *reinterpret_cast<FixedSmem*>(smem);
  bf16* kttile = reinterpret_cast<bf16*>(smem + a.off_tiles);          // phase B (dead before D)
  float* sval = reinterpret_cast<float*>(smem + a.off_scores);
  uint8_t* flag = reinterpret_cast<uint8_t*>(smem + a.off_flags);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + a.off_sel);
  int32_t* bt_s = reinterpret_cast<int32_t*>(smem + a.off_bt);         // paged: page of each block
  float* recv = reinterpret_cast<float*>(smem + a.off_recv);
  uint8_t* tK = smem + a.off_tiles;
  uint8_t* tV = tK + 2 * a.tile_half_bytes;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int ns = a.ns;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int pair = b * a.Hkv + hk;
  const int G = a.G;
  const bool app = a.k_new != nullptr;
  const int cpr = a.cpr;
  const int jlo = (int)rank * cpr;                       // blocks this CTA scores: [jlo, jhi)
  const bool spec = a.kt_spec != 0;
  // Lengths: launch constants, worked out while the previous kernel may still
  // run; with per-row lengths (RAG) they are redone from n_rows after the wait.
  int n_old = a.n;                                       // tokens before this step's append
  int n_tot = a.n + (app ? 1 : 0);                       // tokens attended
  int nb_new = app ? n_old / a.blk : -1;
  int nblk = a.nblk;
  int jhi = min(nblk, jlo + cpr);
  bool own_new = app && nb_new >= jlo && nb_new < jhi;   // this CTA holds the appended key's block

  // Prologue that touches no data of the previous kernel.
  if (tid == 0) {
    for (int i = 0; i < MAX_ROUND_ROWS / 8; ++i) mbar_init(&fs.mbar[i], 1);
    mbar_init(&fs.ebar, 1);
    mbar_init(&fs.ktbar, 1);
    mbar_init(&fs.sbar, 1);
    fence_mbar_init();
    // every CTA of the cluster sends its scores and its warps' score bounds to every
    // CTA (per-row lengths are only known after the dependency wait: armed below)
    if (!RAG) mbar_arrive_expect_tx(&fs.sbar, (uint32_t)(a.nblk * 4 + ns * NWARP * 8) + a.sbar_extra_tx);
    // every CTA of the cluster sends its (O, max, sum) of each head this CTA owns
    const int gmine = (int)rank < G ? (G - (int)rank + ns - 1) / ns : 0;
    if (gmine > 0) mbar_arrive_expect_tx(&fs.ebar, (uint32_t)(gmine * ns * PART_STRIDE * 4));
    if (!MT && a.tma_kv) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    if (spec) prefetch_tmap(&tmKT);
  }
  for (int i = tid; i < 4 * 256; i += NT) fs.hist[i] = 0;
  if (tid == 0) fs.misc[3] = 0;
  if (tid < 16) {
    fs.mrun[tid] = neg_inf();
    fs.lrun[tid] = 0.f;
  }
  // The group's query rows and the appended key / value are read first after
  // the dependency wait: ask L2 for them now (a prefetch brings nothing into
  // the CTA, so it may run while the previous kernel still writes them).
  if (tid == 32) {
    prefetch_l2_bulk(reinterpret_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)hk * G) * HD,
                     (uint32_t)(G * HD * 2));
    if (app) {
      prefetch_l2_bulk(a.k_new + (size_t)pair * HD, HD * 2);
      prefetch_l2_bulk(a.v_new + (size_t)pair * HD, HD * 2);
    }
  }
  // every CTA of the cluster must have started before a DSMEM store reaches it;
  // the matching wait (start of phase B) precedes the first remote store (phase B)
  cluster_arrive_relaxed();
  pdl_wait();
  pdl_launch_dependents();
  if (RAG) {
    // this batch row's length, clamped into [1, the call's maximum] (an entry out
    // of range raises ERR_BAD_LENGTH)
    const int nr = a.n_rows ? a.n_rows[b] : a.n;
    n_old = min(max(nr, 1), a.n);
    if (nr != n_old && tid == 0 && rank == 0) atomicOr(&g_hsa_err, ERR_BAD_LENGTH);
    n_tot = n_old + (app ? 1 : 0);
    nb_new = app ? n_old / a.blk : -1;
    nblk = (n_tot + a.blk - 1) / a.blk;
    jhi = min(nblk, jlo + cpr);
    own_new = app && nb_new >= jlo && nb_new < jhi;
    // (a remote byte count arriving before this arrival is fine: the phase needs both)
    if (tid == 0) mbar_arrive_expect_tx(&fs.sbar, (uint32_t)(nblk * 4 + ns * NWARP * 8) + a.sbar_extra_tx);
  }
  if (PG) {
    // this row's block table (published by the barriers of phase A); a page id out
    // of range is clamped and raises ERR_BAD_LENGTH
    const int32_t* btr = a.block_table + (size_t)b * a.bt_stride;
    for (int j = tid; j < nblk; j += NT) {
      const int pg = btr[j];
      const int pc = min(max(pg, 0), (int)a.num_pages - 1);
      if (pg != pc && rank == 0) atomicOr(&g_hsa_err, ERR_BAD_LENGTH);
      bt_s[j] = pc;
    }
  }
  // KT rows do not depend on the query: with the prefetch, all 2*D rows of this
  // CTA's blocks are in flight while the channels are chosen
  if (spec && tid == 0 && jhi > jlo) {
    mbar_arrive_expect_tx(&fs.ktbar, (uint32_t)(2 * HD * cpr * (F8 ? 1 : 2)));
    tma_load_2d(kttile, &tmKT, jlo, pair * 2 * HD, &fs.ktbar);
  }
  // the CTA holding the appended key's block persists its KT column; without
  // the prefetch it fetches the old column now and writes the new one at the end
  const uint32_t* mrow = MK ? a.mask + (size_t)pair * a.mask_ld : nullptr;
  // the appended key starts its block's bounds when the block holds no earlier
  // candidate, and widens them otherwise
  bool fresh_new = (a.blk_shift >= 0 ? (n_old & (a.blk - 1)) : n_old % a.blk) == 0;
  if (MK && own_new && !fresh_new) fresh_new = !cand_any(mrow, a.n_prompt, (int64_t)nb_new * a.blk, n_old);
  bf16 kt_old = __float2bfloat16(0.f);
  bf16* kt_col = nullptr;
  uint8_t kt_old8 = 0;
  uint8_t* kt_col8 = nullptr;
  if (own_new) {
    const int m = tid >> 7, c = tid & (HD - 1);    // 256 threads = {max, min} x 128 channels
    const size_t o = ((size_t)pair * 2 * HD + m * HD + c) * a.nblk_cap + nb_new;
    if (F8) {
      kt_col8 = reinterpret_cast<uint8_t*>(a.kt) + o;
      if (!spec && !fresh_new) kt_old8 = *kt_col8;
    } else {
      kt_col = reinterpret_cast<bf16*>(a.kt) + o;
      if (!spec && !fresh_new) kt_old = *kt_col;
    }
  }
  // e4m3 storage: dequantization scales of this pair
  const float k_sc = F8 ? __ldg(a.k_scale + pair) : 1.f;
  const float v_sc = F8 ? __ldg(a.v_scale + pair) : 1.f;

  // ---------------------------------------------------------------- A ------
  {
    const bf16* qg = reinterpret_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)hk * G) * HD;
    const int r = tid >> 4, c = tid & 15;          // 256 threads = 16 rows x 16 chunks
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < G) val = *reinterpret_cast<const uint4*>(qg + (size_t)r * HD + c * 8);
    *reinterpret_cast<uint4*>(&fs.qs[r][c * 8]) = val;
    if (app && tid < 32) {
      const bf16* src = (tid < 16 ? a.k_new : a.v_new) + (size_t)pair * HD + (tid & 15) * 8;
      bf16* dst = (tid < 16 ? fs.knew : fs.vnew) + (tid & 15) * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
  }
  __syncthreads();
  if (F8 && app) {
    // the appended key / value as stored: codes of x / scale, and their values
    const int c = tid & (HD - 1);
    bf16* src = tid < HD ? fs.knew : fs.vnew;
    const uint16_t code = e4m3x2_from_f32(__fdiv_rn(bf2f(src[c]), tid < HD ? k_sc : v_sc), 0.f);
    (tid < HD ? fs.knew8 : fs.vnew8)[c] = (uint8_t)(code & 0xFF);
    src[c] = __float2bfloat16_rn(e4m3x2_to_f32(code).x);   // read after the barriers of phase A
  }
  bool inexact = false;
  if (tid < HD) {
    float sa = 0.f, sq = 0.f;
    for (int g = 0; g < G; ++g) {
      const float x = bf2f(fs.qs[g][tid]);
      float e1, e2;
      sa = two_sum(sa, fabsf(x), e1);
      sq = two_sum(sq, x, e2);
      inexact |= (e1 != 0.f) | (e2 != 0.f);
    }
    fs.asum[tid] = sa;
    fs.qbar32[tid] = sq;
  }
  const bool use64 = __syncthreads_or(inexact) != 0;
  if (app && rank == 0) {
    // Persist the appended token now (cache row, MT candidate index): this launch
    // never reads that row from memory (its tiles take the token from shared
    // memory, TMA reads past the old length return zero, gathers stop below it),
    // so the store leaves the tail of the launch.
    if (F8 && tid < 16) {
      // 128 code bytes per row: threads 0-7 the key, 8-15 the value
      uint8_t* dst = (tid < 8 ? reinterpret_cast<uint8_t*>(a.k) : reinterpret_cast<uint8_t*>(a.v)) +
                     ((size_t)pair * a.cap + (size_t)n_old) * HD + (tid & 7) * 16;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>((tid < 8 ? fs.knew8 : fs.vnew8) + (tid & 7) * 16);
    } else if (!F8 && tid < 32) {
      bf16* dst = (tid < 16 ? reinterpret_cast<bf16*>(a.k) : reinterpret_cast<bf16*>(a.v)) +
                  (PG ? (((size_t)bt_s[nb_new] * a.Hkv + hk) * a.blk + (size_t)(n_old % a.blk))
                      : (size_t)pair * a.cap + (MT ? a.row : (int64_t)n_old)) * HD + (tid & 15) * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>((tid < 16 ? fs.knew : fs.vnew) +
                                                                        (tid & 15) * 8);
    }
    if (MT && tid == 32) a.idx_w[(size_t)pair * a.idx_cap + n_old] = (int32_t)a.row;
  }
  // Top-k1 channels by rank: channel c = tid / 2 is taken when fewer than k1
  // channels have a larger sum, or an equal sum and a lower index.  The two
  // threads of a channel count the even and the odd groups of four channels.
  // Both CTAs of an SM run this count at once, so it is kept to one compare
  // per channel: the sums are >= +0, so "v >= mine" is "v > below" with below
  // the next float under mine, and a group of four channels wholly below c
  // compares against below (equal sums count), any other group against mine;
  // the group holding c then adds its lower-index ties on its own.  The
  // counts are kept in fp32 (exact up to 2^24): a compare feeding a float
  // select and add issues far faster here than one turned into an integer.
  const int c = tid >> 1, hc = tid & 1;
  int rk = 0;
  if (!use64) {
    if (a.k1 < HD) {
      const float mine = fs.asum[c];
      const int mbits = __float_as_int(mine);
      const float below = mbits > 0 ? __int_as_float(mbits - 1) : -1.f;
      const float4* a4 = reinterpret_cast<const float4*>(fs.asum);
      float f0 = 0.f, f1 = 0.f;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        const int q4 = 2 * i + hc;                 // the two halves hit different banks
        const float4 v = a4[q4];
        const float t = (4 * q4 + 3 < c) ? below : mine;
        f0 += (v.x > t ? 1.f : 0.f) + (v.y > t ? 1.f : 0.f);
        f1 += (v.z > t ? 1.f : 0.f) + (v.w > t ? 1.f : 0.f);
      }
      const int qc = c >> 2;
      if ((qc & 1) == hc)
        for (int j = 4 * qc; j < c; ++j) f0 += fs.asum[j] == mine ? 1.f : 0.f;
      rk = (int)(f0 + f1);
    }
  } else {
    // rare: some group sum needs more than fp32's 24 bits; redo every channel in fp64
    if (tid < HD) {
      double sa = 0.0, sq = 0.0;
      for (int g = 0; g < G; ++g) {
        const double x = (double)bf2f(fs.qs[g][tid]);
        sa += fabs(x);
        sq += x;
      }
      fs.akey64[tid] = (uint64_t)__double_as_longlong(sa);   // non-negative: orders like integers
      fs.qbar64[tid] = sq;
    }
    __syncthreads();
    if (a.k1 < HD) {
      const uint64_t mine = fs.akey64[c];
      for (int j = hc; j < HD; j += 2) {
        const uint64_t o = fs.akey64[j];
        rk += (o > mine) || (o == mine && j < c);
      }
    }
  }
  rk += __shfl_xor_sync(0xffffffffu, rk, 1);
  {
    // the kept channels in ascending order
    const bool take = hc == 0 && rk < a.k1;
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    if (lane == 0) fs.wsum[warp] = __popc(bal);
    __syncthreads();
    int pos = __popc(bal & ((1u << lane) - 1u));
    {
      const int4 w0 = *reinterpret_cast<const int4*>(&fs.wsum[0]);
      const int4 w1 = *reinterpret_cast<const int4*>(&fs.wsum[4]);
      pos += (warp > 0 ? w0.x : 0) + (warp > 1 ? w0.y : 0) + (warp > 2 ? w0.z : 0) + (warp > 3 ? w0.w : 0) +
             (warp > 4 ? w1.x : 0) + (warp > 5 ? w1.y : 0) + (warp > 6 ? w1.z : 0);
    }
    if (take) {
      // (fp64 only on the rare inexact path: this GPU's fp64 rate is low)
      float qf;
      bool nonneg;
      if (use64) {
        const double qb = fs.qbar64[c];
        qf = (float)qb;
        nonneg = qb >= 0.0;
      } else {
        qf = fs.qbar32[c];
        nonneg = qf >= 0.f;
      }
      fs.qsel[pos] = qf;
      fs.rowoff[pos] = (nonneg ? 0 : HD) + c;     // Kmax when the group sum is >= 0
      if (rank == 0 && a.sel_channels) a.sel_channels[(size_t)pair * a.k1 + pos] = c;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- B ------
  // CTA `rank` scores blocks [jlo, jhi) and sends every score (and the min / max
  // of each warp's scores) to every CTA of the cluster with st.async; each CTA
  // then holds all nblk scores once its sbar completes.  A score is the fp32
  // sum over the k1 chosen channels of qbar * (Kmax or Kmin), four threads per
  // block pair splitting the channels.
  const int k1 = a.k1;
  float smn = __int_as_float(0x7f800000), smx = neg_inf();
  cluster_wait_acquire();      // every CTA of the cluster has started and armed its barriers
  {
    const uint32_t sbar_local = smem_u32(&fs.sbar);
    const uint32_t sval_local = smem_u32(sval);
    const int bc = spec ? cpr : a.kt_chunk;          // columns per tile (multiple of 8; of 16 for e4m3)
    const int cg = tid & 3, bp = tid >> 2;           // channel group, block pair within a 128-block span
    // with k1 <= 32 each thread's channels (i = cg + 4u) are read into registers
    // now, so the tile reads below do not wait on them one by one
    constexpr int KC = 8;
    const bool kfast = k1 <= 4 * KC;
    int rowv[KC];
    float qv[KC];
#pragma unroll
    for (int u = 0; u < KC; ++u) {
      const int i = cg + 4 * u;
      const bool ok = kfast && i < k1;
      rowv[u] = ok ? (spec ? fs.rowoff[i] : i) : 0;   // row 0 with weight 0 adds +0
      qv[u] = ok ? fs.qsel[i] : 0.f;
    }
    if (MK) {
      // which of this CTA's blocks hold a candidate (read after the barrier before scoring)
      for (int j = jlo + tid; j < jhi; j += NT)
        flag[j] = cand_any(mrow, a.n_prompt, (int64_t)j * a.blk, min((int64_t)(j + 1) * a.blk, (int64_t)n_tot)) ? 1
                                                                                                                : 0;
    }
    for (int cb0 = jlo; cb0 < jhi; cb0 += bc) {
      const int nb_here = min(bc, jhi - cb0);
      if (spec) {
        if (!mbar_wait(&fs.ktbar, 0, &g_hsa_err, a.wait_ns)) mbar_wait(&fs.ktbar, 0, &g_hsa_err, a.wait_ns);
        if (own_new) {
          // fold the appended key into its block in every KT row and persist the column
          const int col = nb_new - cb0;
          const int m = tid >> 7, c = tid & (HD - 1);
          if (F8) {
            uint8_t& slot = reinterpret_cast<uint8_t*>(kttile)[(size_t)tid * bc + col];
            const float x = bf2f(fs.knew[c]), o = e4m3x2_to_f32(slot).x;
            if (fresh_new || (m == 1 ? (x < o) : (x > o))) slot = fs.knew8[c];
            *kt_col8 = slot;
          } else {
            const bf16 kv = fs.knew[c];
            bf16& slot = kttile[(size_t)tid * bc + col];
            if (fresh_new) {
              slot = kv;
            } else {
              const float x = bf2f(kv), o = bf2f(slot);
              if (m == 1 ? (x < o) : (x > o)) slot = kv;
            }
            *kt_col = slot;
          }
        }
      } else {
        if (cb0 > jlo) __syncthreads();              // the previous chunk's scores are done with the tile
        // 16-byte chunks: 8 bf16 entries, or 16 e4m3 codes
        const int per = F8 ? 16 : 8;
        const int n16 = (nb_here + per - 1) / per;
        for (int row = warp; row < k1; row += NWARP) {
          const size_t eb = F8 ? 1 : 2;
          const uint8_t* src = reinterpret_cast<const uint8_t*>(a.kt) +
                               (((size_t)pair * 2 * HD + fs.rowoff[row]) * a.nblk_cap + cb0) * eb;
          uint8_t* dst = reinterpret_cast<uint8_t*>(kttile) + (size_t)row * bc * eb;
          for (int ch = lane; ch < n16; ch += 32) cp_async_16(smem_u32(dst + ch * 16), src + ch * 16);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        if (own_new && nb_new >= cb0 && nb_new < cb0 + nb_here) {
          const int col = nb_new - cb0;
          const bool fresh = fresh_new;
          for (int i = tid; i < k1; i += NT) {
            const int ro = fs.rowoff[i];
            const bf16 kv = fs.knew[ro & (HD - 1)];
            if (F8) {
              uint8_t& slot = reinterpret_cast<uint8_t*>(kttile)[(size_t)i * bc + col];
              const float x = bf2f(kv), o = e4m3x2_to_f32(slot).x;
              if (fresh || (ro >= HD ? (x < o) : (x > o))) slot = fs.knew8[ro & (HD - 1)];
            } else {
              bf16& slot = kttile[(size_t)i * bc + col];
              if (fresh) {
                slot = kv;
              } else {
                const float x = bf2f(kv), o = bf2f(slot);
                if (ro >= HD ? (x < o) : (x > o)) slot = kv;
              }
            }
          }
        }
      }
      __syncthreads();
      const uint32_t* tile32 = reinterpret_cast<const uint32_t*>(kttile);
      const int pitch = bc / 2;
      for (int jb = 0; jb < nb_here; jb += 128) {      // warp-uniform trip count
        const int jp = (jb >> 1) + bp;
        const bool live = 2 * jp < nb_here;
        const int jpc = live ? jp : 0;
        float s0 = 0.f, s1 = 0.f;
        if (kfast) {
#pragma unroll
          for (int u = 0; u < KC; ++u) {
            if (F8) {
              // two blocks' codes per 16-bit word, row pitch bc bytes
              const float2 f = e4m3x2_to_f32(reinterpret_cast<const uint16_t*>(kttile)[rowv[u] * pitch + jpc]);
              s0 = fmaf(qv[u], f.x, s0);
              s1 = fmaf(qv[u], f.y, s1);
            } else {
              const uint32_t v = tile32[rowv[u] * pitch + jpc];
              s0 = fmaf(qv[u], bf16_lo(v), s0);
              s1 = fmaf(qv[u], bf16_hi(v), s1);
            }
          }
        } else {
          for (int i = cg; i < k1; i += 4) {
            const int row = spec ? fs.rowoff[i] : i;
            const float q = fs.qsel[i];
            if (F8) {
              const float2 f = e4m3x2_to_f32(reinterpret_cast<const uint16_t*>(kttile)[(size_t)row * pitch + jpc]);
              s0 = fmaf(q, f.x, s0);
              s1 = fmaf(q, f.y, s1);
            } else {
              const uint32_t v = tile32[(size_t)row * pitch + jpc];
              s0 = fmaf(q, bf16_lo(v), s0);
              s1 = fmaf(q, bf16_hi(v), s1);
            }
          }
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        s0 = (s0 == 0.f) ? 0.f : s0;     // -0 -> +0
        s1 = (s1 == 0.f) ? 0.f : s1;
        const int j = cb0 + 2 * jp;
        const bool v0 = live, v1 = live && 2 * jp + 1 < nb_here;
        bool f0 = v0, f1 = v1;                       // finite scores (the bucket range)
        if (MK) {
          // a block without a candidate scores -inf, the newest row's block +inf
          const int tail = (n_tot - 1) / a.blk;
          const float pinf = __int_as_float(0x7f800000);
          if (v0) s0 = !flag[j] ? neg_inf() : (j == tail ? pinf : s0);
          if (v1) s1 = !flag[j + 1] ? neg_inf() : (j + 1 == tail ? pinf : s1);
          f0 = v0 && isfinite(s0);
          f1 = v1 && isfinite(s1);
        }
        if (f0) {
          smn = fminf(smn, s0);
          smx = fmaxf(smx, s0);
        }
        if (f1) {
          smn = fminf(smn, s1);
          smx = fmaxf(smx, s1);
        }
        if (cg < 2 && (cg == 0 ? v0 : v1)) {
          const float sv = cg == 0 ? s0 : s1;
          const uint32_t off = 4u * (uint32_t)(j + cg);
          for (int d = 0; d < ns; ++d) st_async_f32(mapa(sval_local + off, d), sv, mapa(sbar_local, d));
        }
      }
    }
    smn = key2f(__reduce_min_sync(0xffffffffu, f2key(smn)));
    smx = key2f(__reduce_max_sync(0xffffffffu, f2key(smx)));
    if (lane < ns) {
      const uint32_t off = smem_u32(&fs.rbound[(int)rank * NWARP + warp]);
      st_async_v2f32(mapa(off, lane), smn, smx, mapa(sbar_local, lane));
    }
    if (!mbar_wait(&fs.sbar, 0, &g_hsa_err, a.wait_ns)) mbar_wait(&fs.sbar, 0, &g_hsa_err, a.wait_ns);
    {
      // every warp combines the ns * NWARP (<= 64) bounds, two per lane
      const int nb = ns * NWARP;
      const float2 r0 = lane < nb ? fs.rbound[lane] : make_float2(__int_as_float(0x7f800000), neg_inf());
      const float2 r1 = lane + 32 < nb ? fs.rbound[lane + 32] : make_float2(__int_as_float(0x7f800000), neg_inf());
      smn = fminf(r0.x, r1.x);
      smx = fmaxf(r0.y, r1.y);
      smn = key2f(__reduce_min_sync(0xffffffffu, f2key(smn)));
      smx = key2f(__reduce_max_sync(0xffffffffu, f2key(smx)));
    }
  }

  // ---------------------------------------------------------------- C ------
  const int k2e = RAG ? min(a.k2, nblk) : a.k2e;
  if (k2e >= nblk) {
    for (int j = tid; j < nblk; j += NT) sel[j] = j;
  } else {
    const bool done = nblk <= 2 * NT && smx > smn && isfinite(smx - smn) &&
                      topk_small(sval, nblk, k2e, smn, smx, sel, fs);
    if (!done) topk_list(sval, nblk, k2e, smn, smx, flag, sel, fs);
  }
  __syncthreads();

  // ---------------------------------------------------------------- D ------
  // Q as the B operand of S^T = K Q^T: heads 8*ht .. 8*ht+7, all 8 k-steps.
  uint32_t qb[NH][8][2];
#pragma unroll
  for (int ht = 0; ht < NH; ++ht)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      ldsm_x4(smem_u32(&fs.qs[8 * ht + (lane & 7)][(4 * j + (lane >> 3)) * 8]), qb[ht][2 * j][0], qb[ht][2 * j][1],
              qb[ht][2 * j + 1][0], qb[ht][2 * j + 1][1]);
  // O^T accumulator of this warp's 16 output dimensions: dims 16*warp + lane/4 (+8),
  // heads 8*ht + 2*(lane%4) + {0, 1}
  // (the narrow-group kernel keeps the lo part of P in its own accumulator,
  // halving the chain of dependent mma in the PV step)
  constexpr bool SPLIT = NH == 1;
  float acc[NH][4], accl[NH][4];
#pragma unroll
  for (int ht = 0; ht < NH; ++ht)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[ht][e] = accl[ht][e] = 0.f;
  // With several staging rounds per CTA (WF, narrow groups) every warp instead
  // runs its own online softmax over its own 16-token steps and accumulates O^T
  // over all 128 dimensions (acc8[dt]: dims 16*dt + lane/4 (+8), heads
  // 2*(lane%4) + {0, 1}); the CTA merges the eight warp partials once, after the
  // last round, so a round needs only its closing barrier.  Each warp reads only
  // its own K and V rows.
  constexpr bool WARP_FLASH = WF && NH == 1;
  float acc8[WARP_FLASH ? 8 : 1][4];
  float wm[2] = {neg_inf(), neg_inf()}, wl[2] = {0.f, 0.f};   // this warp's heads 2*(lane%4) + {0, 1}
#pragma unroll
  for (int i = 0; i < (WARP_FLASH ? 8 : 1); ++i) acc8[i][0] = acc8[i][1] = acc8[i][2] = acc8[i][3] = 0.f;

  const int chunk = RAG ? (k2e + ns - 1) / ns : a.chunk;   // blocks per CTA (at most the plan's chunk)
  const int s_lo = (int)rank * chunk;
  const int s_hi = min(k2e, s_lo + chunk);
  const uint32_t half = a.tile_half_bytes;
  const int blk = a.blk;
  const int bsh = a.blk_shift;
  // x / blk for x >= 0 (a shift for power-of-two blocks: this sits on the chain)
  auto divb = [bsh, blk](int x) { return bsh >= 0 ? x >> bsh : x / blk; };
  uint32_t phase = 0;
  unsigned int* err = &g_hsa_err;
  const int g4 = lane >> 2, t4 = lane & 3;
  // K/V rows arrive by TMA (block rows contiguous, blk a multiple of 8) or are
  // gathered row by row with cp.async (MT candidate rows, or other block sizes)
  const bool gat = MT || a.tma_kv == 0;

  const float sl2 = a.scale_log2 * k_sc;        // logits in log2 units (e4m3: times the K scale)
  for (int r0 = s_lo; r0 < s_hi; r0 += a.slots_round) {
    const int nsl = min(a.slots_round, s_hi - r0);
    const int rows = nsl * blk;
    const int nsteps = (rows + 15) / 16;
    const int rows16 = nsteps * 16;
    if (!gat) {
      {
        // The copies are spread over all warps: one warp issuing them all serialises them.
        // The region was last read through the generic proxy before a barrier (write
        // after read), so no proxy fence is needed.
        if (warp == 0)
          for (int s = lane; s < nsl; s += 32)
            mbar_arrive_expect_tx(&fs.mbar[s], (uint32_t)blk * 128u * (F8 ? 2u : 4u));
        __syncwarp();
        if (F8) {
          // code rows (128 bytes, unswizzled) into the hi half of the K and V
          // tiles, converted in place by the warp that owns the rows
          const int part = warp & 1;
          for (int s = (warp >> 1) + 4 * lane; s < nsl; s += 128) {
            const uint32_t off = (uint32_t)s * blk * 128u;
            tma_load_3d((part ? tV : tK) + half + off, part ? &tmV : &tmK, 0, sel[r0 + s] * blk, pair, &fs.mbar[s]);
          }
        } else {
          const int part = warp & 3;                   // K lo, K hi, V lo, V hi
          for (int s = (warp >> 2) + 2 * lane; s < nsl; s += 64) {
            // dense: rows sel*blk.. of the pair's cache; paged: the whole (page, head) slab
            const int y = PG ? 0 : sel[r0 + s] * blk;
            const int z = PG ? bt_s[sel[r0 + s]] * a.Hkv + hk : pair;
            const uint32_t off = (uint32_t)s * blk * 128u + (uint32_t)(part & 1) * half;
            tma_load_3d(((part >> 1) ? tV : tK) + off, (part >> 1) ? &tmV : &tmK, (part & 1) * 64, y, z,
                        &fs.mbar[s]);
          }
        }
      }
    } else {
      const bf16* kb = reinterpret_cast<const bf16*>(a.k) + (PG ? (size_t)0 : (size_t)pair * a.cap * HD);
      const bf16* vb = reinterpret_cast<const bf16*>(a.v) + (PG ? (size_t)0 : (size_t)pair * a.cap * HD);
      const int32_t* ib = MT ? a.idx + (size_t)pair * a.idx_cap : nullptr;
      for (int i = tid; i < rows * 16; i += NT) {
        const int r = i >> 4, ch = i & 15;
        const int slot = divb(r);
        const int t = sel[r0 + slot] * blk + (r - slot * blk);
        const uint32_t o = (uint32_t)(ch >> 3) * half + swz128(r, ch & 7);
        if (t < n_old) {
          // row of token t: MT candidate row, paged (page, head) slab row, or t itself
          const int64_t prow = MT ? min(max((int64_t)ib[t], (int64_t)0), a.cap - 1)
                               : PG ? ((int64_t)bt_s[divb(t)] * a.Hkv + hk) * blk + (t - divb(t) * blk) : (int64_t)t;
          cp_async_16(smem_u32(tK) + o, kb + prow * HD + ch * 8);
          cp_async_16(smem_u32(tV) + o, vb + prow * HD + ch * 8);
        } else if (t == n_old && app) {
          *reinterpret_cast<uint4*>(tK + o) = *reinterpret_cast<const uint4*>(fs.knew + ch * 8);
          *reinterpret_cast<uint4*>(tV + o) = *reinterpret_cast<const uint4*>(fs.vnew + ch * 8);
        } else {
          *reinterpret_cast<uint4*>(tK + o) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(tV + o) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
    }
    // Rows [rows, rows16) of both tiles enter the last 16-token step with P = 0: keep them finite.
    for (int i = tid; i < (rows16 - rows) * 32; i += NT) {
      const int r = rows + (i >> 5), ch = (i >> 1) & 15;
      *reinterpret_cast<uint4*>(((i & 1) ? tV : tK) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7)) =
          make_uint4(0, 0, 0, 0);
    }
    if (MK && tid < MAX_ROUND_ROWS) {
      // candidate rows of this round, one bit per staged row
      bool e = false;
      if (tid < rows) {
        const int slot = divb(tid);
        const int t = sel[r0 + slot] * blk + (tid - slot * blk);
        e = t < n_tot && (t >= a.n_prompt || ((__ldg(mrow + (t >> 5)) >> (t & 31)) & 1u) != 0);
      }
      const unsigned bm = __ballot_sync(0xffffffffu, e);
      if (lane == 0) fs.relig[warp] = bm;
    }
    if (gat) cp_async_wait_all();
    // cp.async rows and zero rows come from every thread; TMA rows are waited for per slot
    if (gat || rows16 != rows || MK) __syncthreads();

    // --- S^T = K Q^T for the warp's 16-token step, masked and in log2 units
    const int c0 = warp * 16;
    const bool has_step = c0 < rows;
    float x[NH][4];
#pragma unroll
    for (int ht = 0; ht < NH; ++ht) x[ht][0] = x[ht][1] = x[ht][2] = x[ht][3] = neg_inf();
    if (has_step) {
      if (!gat) {
        const int sa = divb(c0), sb = min(divb(c0 + 15), nsl - 1);
        for (int s = sa; s <= sb; ++s)
          if (!mbar_wait(&fs.mbar[s], phase, err, a.wait_ns)) mbar_wait(&fs.mbar[s], phase, err, a.wait_ns);
        if (F8) {
          // this warp's 16 key and value rows: codes (row r at byte r*128 of each
          // tile's hi half) to bf16 code values in the swizzled tiles, in place
          // (all reads first); other warps read the value rows only after the
          // barriers before the PV step
          uint4 cv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int q = lane + 32 * (i & 3), r = c0 + (q >> 3), cb = q & 7;
            const uint8_t* src = (i < 4 ? tK : tV) + half + (uint32_t)r * 128u + cb * 16;
            cv[i] = r < rows ? *reinterpret_cast<const uint4*>(src) : make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int q = lane + 32 * (i & 3), r = c0 + (q >> 3), cb = q & 7;
            if (r >= rows) continue;
            const uint32_t w[4] = {cv[i].x, cv[i].y, cv[i].z, cv[i].w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int ch8 = 2 * cb + hh;               // 8 channels per bf16 chunk
              const uint4 o = make_uint4(e4m3x2_to_bf16x2((uint16_t)(w[2 * hh] & 0xFFFF)),
                                         e4m3x2_to_bf16x2((uint16_t)(w[2 * hh] >> 16)),
                                         e4m3x2_to_bf16x2((uint16_t)(w[2 * hh + 1] & 0xFFFF)),
                                         e4m3x2_to_bf16x2((uint16_t)(w[2 * hh + 1] >> 16)));
              *reinterpret_cast<uint4*>((i < 4 ? tK : tV) + (uint32_t)(ch8 >> 3) * half + swz128(r, ch8 & 7)) = o;
            }
          }
          __syncwarp();
        }
        if (app) {
          // the appended token lies past the tensor map's extent (read as zero): write it in
          for (int s = sa; s <= sb; ++s) {
            if (sel[r0 + s] != nb_new) continue;
            const int r = s * blk + (n_old - nb_new * blk);
            const int ch = lane & 15;
            const uint32_t o = (uint32_t)(ch >> 3) * half + swz128(r, ch & 7);
            uint8_t* dst = (lane < 16 ? tK : tV) + o;
            const bf16* src = (lane < 16 ? fs.knew : fs.vnew) + ch * 8;
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
          }
          __syncwarp();
        }
      }
      // NC independent accumulator chains over the 8 k-steps (a dependent mma
      // costs ~35 cycles here); two for the wide-group kernel (register room)
      constexpr int NC = NH == 1 ? 4 : 2;
      float st[NH][NC][4];
#pragma unroll
      for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int u = 0; u < NC; ++u) st[ht][u][0] = st[ht][u][1] = st[ht][u][2] = st[ht][u][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int r = c0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = ks * 2 + (lane >> 4);
        uint32_t ka[4];
        ldsm_x4(smem_u32(tK) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7), ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
        for (int ht = 0; ht < NH; ++ht) mma_bf16(st[ht][ks % NC], ka, qb[ht][ks][0], qb[ht][ks][1]);
      }
      // this lane: tokens c0 + lane/4 (e = 0, 1) and + 8 (e = 2, 3); heads 2(lane%4) + (e & 1)
      const int ta = c0 + g4, tb = ta + 8;
      const int sla = divb(ta), slb = divb(tb);
      bool va = ta < rows && sel[r0 + sla] * blk + (ta - sla * blk) < n_tot;
      bool vb = tb < rows && sel[r0 + slb] * blk + (tb - slb * blk) < n_tot;
      if (MK) {
        va = va && ((fs.relig[ta >> 5] >> (ta & 31)) & 1u) != 0;
        vb = vb && ((fs.relig[tb >> 5] >> (tb & 31)) & 1u) != 0;
      }
#pragma unroll
      for (int ht = 0; ht < NH; ++ht)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float sv = (NC == 4 ? (st[ht][0][e] + st[ht][1][e]) + (st[ht][2][NC == 4 ? e : 0] + st[ht][3 % NC][e])
                                    : st[ht][0][e] + st[ht][1][e]) * sl2;
          x[ht][e] = ((e < 2) ? va : vb) ? sv : neg_inf();
        }
    }
    if constexpr (WARP_FLASH) {
      // --- this warp's head maxima and probability sums (x = -inf off its step)
      float m0 = fmaxf(x[0][0], x[0][2]), m1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      }
      const float mn0 = fmaxf(wm[0], m0), mn1 = fmaxf(wm[1], m1);
      const float cr0 = (wm[0] == neg_inf()) ? 0.f : ex2_ftz(wm[0] - mn0);
      const float cr1 = (wm[1] == neg_inf()) ? 0.f : ex2_ftz(wm[1] - mn1);
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = (x[0][e] == neg_inf()) ? 0.f : ex2_ftz(x[0][e] - ((e & 1) ? mn1 : mn0));
      float s0 = p[0] + p[2], s1 = p[1] + p[3];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      wl[0] = wl[0] * cr0 + s0;
      wl[1] = wl[1] * cr1 + s1;
      wm[0] = mn0;
      wm[1] = mn1;
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        acc8[dt][0] *= cr0;
        acc8[dt][1] *= cr1;
        acc8[dt][2] *= cr0;
        acc8[dt][3] *= cr1;
      }
      if (has_step) {
        // --- O^T (all 128 dims) += V^T P^T over this warp's 16 tokens; P^T as the
        // B operand straight from registers (hi + lo bf16 parts)
        const uint32_t h0 = pack_bf16(p[0], p[1]), h1 = pack_bf16(p[2], p[3]);
        const uint32_t l0 = pack_bf16(p[0] - bf16_lo(h0), p[1] - bf16_hi(h0));
        const uint32_t l1 = pack_bf16(p[2] - bf16_lo(h1), p[3] - bf16_hi(h1));
        const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
        const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);
        const int r = c0 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          const int ch = 2 * dt + ((lane >> 3) & 1);
          uint32_t va4[4];
          ldsm_x4_t(smem_u32(tV) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7), va4[0], va4[1], va4[2], va4[3]);
          mma_bf16(acc8[dt], va4, bh0, bh1);
          mma_bf16(acc8[dt], va4, bl0, bl1);
        }
      }
    } else {
      // --- CTA-wide head maxima of this round
  #pragma unroll
      for (int ht = 0; ht < NH; ++ht) {
        float m0 = fmaxf(x[ht][0], x[ht][2]), m1 = fmaxf(x[ht][1], x[ht][3]);
  #pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
          m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
        }
        if (g4 == 0) {
          fs.wmaxh[warp][8 * ht + 2 * t4] = m0;
          fs.wmaxh[warp][8 * ht + 2 * t4 + 1] = m1;
        }
      }
      __syncthreads();
      float mnew[NH][2], corr[NH][2];
  #pragma unroll
      for (int ht = 0; ht < NH; ++ht)
  #pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 8 * ht + 2 * t4 + hh;
          float m = fs.mrun[h];
  #pragma unroll
          for (int w = 0; w < NWARP; ++w) m = fmaxf(m, fs.wmaxh[w][h]);
          const float mo = fs.mrun[h];
          mnew[ht][hh] = m;
          corr[ht][hh] = (mo == neg_inf()) ? 0.f : ex2_ftz(mo - m);
        }
      // --- probabilities, their head sums, and P^T fragments for every warp
  #pragma unroll
      for (int ht = 0; ht < NH; ++ht) {
        float p[4];
  #pragma unroll
        for (int e = 0; e < 4; ++e) p[e] = (x[ht][e] == neg_inf()) ? 0.f : ex2_ftz(x[ht][e] - mnew[ht][e & 1]);
        float s0 = p[0] + p[2], s1 = p[1] + p[3];
  #pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (g4 == 0) {
          fs.wsumh[warp][8 * ht + 2 * t4] = s0;
          fs.wsumh[warp][8 * ht + 2 * t4 + 1] = s1;
        }
        if (has_step) {
          const uint32_t h0 = pack_bf16(p[0], p[1]), h1 = pack_bf16(p[2], p[3]);
          const uint32_t l0 = pack_bf16(p[0] - bf16_lo(h0), p[1] - bf16_hi(h0));
          const uint32_t l1 = pack_bf16(p[2] - bf16_lo(h1), p[3] - bf16_hi(h1));
          uint32_t* pf = &fs.pfrag[warp][ht][0][0];
          pf[0 * 32 + lane] = movmatrix_trans(h0);
          pf[1 * 32 + lane] = movmatrix_trans(h1);
          pf[2 * 32 + lane] = movmatrix_trans(l0);
          pf[3 * 32 + lane] = movmatrix_trans(l1);
        }
      }
      __syncthreads();
      // --- running max / sum (threads < 16 keep the CTA copy) and rescale
      if (tid < 16) {
        float m = fs.mrun[tid];
  #pragma unroll
        for (int w = 0; w < NWARP; ++w) m = fmaxf(m, fs.wmaxh[w][tid]);
        const float c = (fs.mrun[tid] == neg_inf()) ? 0.f : ex2_ftz(fs.mrun[tid] - m);
        float l = fs.lrun[tid] * c;
  #pragma unroll
        for (int w = 0; w < NWARP; ++w) l += fs.wsumh[w][tid];
        fs.lrun[tid] = l;
        fs.mrun[tid] = m;
      }
  #pragma unroll
      for (int ht = 0; ht < NH; ++ht) {
        acc[ht][0] *= corr[ht][0];
        acc[ht][1] *= corr[ht][1];
        acc[ht][2] *= corr[ht][0];
        acc[ht][3] *= corr[ht][1];
        if (SPLIT) {
          accl[ht][0] *= corr[ht][0];
          accl[ht][1] *= corr[ht][1];
          accl[ht][2] *= corr[ht][0];
          accl[ht][3] *= corr[ht][1];
        }
      }
      // --- O^T (dims 16*warp .. +15) += V^T P^T over every 16-token step of the round
      for (int cs = 0; cs < nsteps; ++cs) {
        const int r = cs * 16 + (lane & 7) + (lane >> 4) * 8;
        const int ch = 2 * warp + ((lane >> 3) & 1);
        uint32_t va4[4];
        ldsm_x4_t(smem_u32(tV) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7), va4[0], va4[1], va4[2], va4[3]);
  #pragma unroll
        for (int ht = 0; ht < NH; ++ht) {
          const uint32_t* pf = &fs.pfrag[cs][ht][0][0];
          mma_bf16(acc[ht], va4, pf[0 * 32 + lane], pf[1 * 32 + lane]);
          mma_bf16(SPLIT ? accl[ht] : acc[ht], va4, pf[2 * 32 + lane], pf[3 * 32 + lane]);
        }
      }
    }
    phase ^= 1u;
    if (r0 + a.slots_round < s_hi) __syncthreads();   // tiles and fragments are reused by the next round
  }

  if (SPLIT) {
#pragma unroll
    for (int ht = 0; ht < NH; ++ht)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[ht][e] += accl[ht][e];
  }
  // ---------------------------------------------------------------- E ------
  // Partials go to the owner of each head (head g: CTA g % ns) with st.async,
  // which counts their bytes on the owner's ebar; only owners wait.
  // owner CTA and slot of head g (shifts for a power-of-two cluster: this is the tail)
  const int nsh = a.ns_shift;
  auto own_of = [nsh, ns](int g) { return nsh >= 0 ? g & (ns - 1) : g % ns; };
  auto slot_of = [nsh, ns](int g) { return nsh >= 0 ? g >> nsh : g / ns; };
  const int gown = slot_of(G + ns - 1);
  if constexpr (WARP_FLASH) {
    // Warp w leaves its O^T in its own K rows (bytes [2048 w, 2048 w + 2048) of
    // the lo half for dims 0-63, of the hi half for dims 64-127; no other warp
    // reads those rows after the last round) as [dim][G] floats, so a lane's two
    // heads are one 8-byte store and the merge reads consecutive words; its
    // (max, sum) per head go to wmaxh / wsumh.
    {
      const int g0 = 2 * t4;
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        float* rg = reinterpret_cast<float*>(tK + (dt < 4 ? 0u : half) + (uint32_t)warp * 2048u);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float* dst = rg + ((16 * dt + g4 + 8 * u) & 63) * G + g0;
          if ((G & 1) == 0 && g0 + 1 < G) {
            *reinterpret_cast<float2*>(dst) = make_float2(acc8[dt][2 * u], acc8[dt][2 * u + 1]);
          } else {
            if (g0 < G) dst[0] = acc8[dt][2 * u];
            if (g0 + 1 < G) dst[1] = acc8[dt][2 * u + 1];
          }
        }
      }
      if (g4 == 0) {
        fs.wmaxh[warp][2 * t4] = wm[0];
        fs.wmaxh[warp][2 * t4 + 1] = wm[1];
        fs.wsumh[warp][2 * t4] = wl[0];
        fs.wsumh[warp][2 * t4 + 1] = wl[1];
      }
    }
    __syncthreads();
    const uint32_t ebar_local = smem_u32(&fs.ebar);
    // thread t merges head g = t % G over dims t / G, t / G + NT / G, ...: the
    // head's owner, remote address and warp weights are worked out once
    const int gstep = NT / G;
    if (tid < gstep * G) {
      const int g = tid % G;
      float fw[NWARP], M = neg_inf(), L = 0.f;
#pragma unroll
      for (int w = 0; w < NWARP; ++w) {
        fw[w] = fs.wmaxh[w][g];
        M = fmaxf(M, fw[w]);
      }
#pragma unroll
      for (int w = 0; w < NWARP; ++w) {
        fw[w] = fw[w] == neg_inf() ? 0.f : ex2_ftz(fw[w] - M);   // a warp with no token of head g weighs 0
        L = fmaf(fw[w], fs.wsumh[w][g], L);
      }
      const int owner = own_of(g), gl = slot_of(g);
      const uint32_t rbase = mapa(smem_u32(recv + ((size_t)gl * ns + rank) * PART_STRIDE), owner);
      const uint32_t rbar = mapa(ebar_local, owner);
      for (int d = tid / G; d < HD; d += gstep) {
        const float* og = reinterpret_cast<const float*>(tK + (d < 64 ? 0u : half)) + (d & 63) * G + g;
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) O = fmaf(fw[w], og[w * 512], O);
        st_async_f32(rbase + 4u * d, O, rbar);
      }
      if (tid < G) st_async_v2f32(rbase + 4u * HD, M, L, rbar);
    }
  } else {
    const uint32_t ebar_local = smem_u32(&fs.ebar);
#pragma unroll
    for (int ht = 0; ht < NH; ++ht) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int g = 8 * ht + 2 * t4 + hh;
        if (g < G) {
          const int owner = own_of(g), gl = slot_of(g);
          const uint32_t base = mapa(smem_u32(recv + ((size_t)gl * ns + rank) * PART_STRIDE), owner);
          const uint32_t bar = mapa(ebar_local, owner);
          st_async_f32(base + 4u * (16 * warp + g4), acc[ht][hh], bar);
          st_async_f32(base + 4u * (16 * warp + g4 + 8), acc[ht][2 + hh], bar);
        }
      }
    }
    if (tid < G) {
      const int owner = own_of(tid), gl = slot_of(tid);
      const uint32_t base = mapa(smem_u32(recv + ((size_t)gl * ns + rank) * PART_STRIDE), owner);
      st_async_v2f32(base + 4u * HD, fs.mrun[tid], fs.lrun[tid], mapa(ebar_local, owner));
    }
  }
  if ((int)rank < G) {
    if (!mbar_wait(&fs.ebar, 0, err, a.wait_ns)) mbar_wait(&fs.ebar, 0, err, a.wait_ns);
  }
  for (int gl = 0; gl < gown; ++gl) {
    const int g = gl * ns + (int)rank;
    if (g >= G) break;
    const float* rp = recv + (size_t)gl * ns * PART_STRIDE;
    if (tid < HD) {
      // all loads first (ns <= 8), then the rescaled sums in rank order
      float mr[8], lr[8], vr[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        mr[r] = neg_inf();
        lr[r] = 0.f;
        vr[r] = 0.f;
        if (r < ns) {
          const float2 ml = *reinterpret_cast<const float2*>(rp + (size_t)r * PART_STRIDE + HD);
          mr[r] = ml.x;
          lr[r] = ml.y;
          vr[r] = rp[(size_t)r * PART_STRIDE + tid];
        }
      }
      float M = mr[0];
#pragma unroll
      for (int r = 1; r < 8; ++r) M = fmaxf(M, mr[r]);
      float A = 0.f, L = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float f = (mr[r] == neg_inf()) ? 0.f : ex2_ftz(mr[r] - M);
        A = fmaf(f, vr[r], A);
        L = fmaf(f, lr[r], L);
      }
      // (L >= 1: the partial holding the maximum contributes exp2(0); a fast
      // divide is within 2 ulp and keeps the IEEE divide off the launch's tail)
      const float y = __fdividef(A, L);
      a.out[((size_t)b * a.Hq + (size_t)hk * G + g) * HD + tid] = F8 ? y * v_sc : y;
    }
  }
  if (own_new && !spec) {
    const int m = tid >> 7, c = tid & (HD - 1);    // 256 threads = {max, min} x 128 channels
    const bf16 kv = fs.knew[c];
    if (F8) {
      const float x = bf2f(kv), o = e4m3x2_to_f32(kt_old8).x;
      if (fresh_new || (m == 1 ? (x < o) : (x > o))) *kt_col8 = fs.knew8[c];
    } else if (fresh_new) {
      *kt_col = kv;
    } else {
      const float x = bf2f(kv), o = bf2f(kt_old);
      if (m == 1 ? (x < o) : (x > o)) *kt_col = kv;
    }
  }
  if (rank == 0) {
    if (a.sel_blocks) {
      for (int j = tid; j < a.k2; j += NT) a.sel_blocks[(size_t)pair * a.k2 + j] = j < k2e ? sel[j] : -1;
    }
  }
}

int g_num_sms = 0;

}  // namespace

bool hsa_plan(HsaArgs& a) {
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  });
  const int n_tot = a.n + (a.k_new ? 1 : 0);
  a.nblk = (n_tot + a.blk - 1) / a.blk;
  a.k2e = std::min(a.k2, a.nblk);
  a.blk_shift = (a.blk & (a.blk - 1)) == 0 ? __builtin_ctz((unsigned)a.blk) : -1;
  const int pairs = a.B * a.Hkv;
  // one wave at two CTAs per SM, at most 8 CTAs per cluster, no more CTAs than blocks
  int ns = std::max(1, (2 * g_num_sms) / std::max(1, pairs));
  ns = std::min(ns, 8);
  ns = std::min(ns, a.k2e);
  a.ns = std::max(ns, 1);
  a.ns_shift = (a.ns & (a.ns - 1)) == 0 ? __builtin_ctz((unsigned)a.ns) : -1;
  a.chunk = (a.k2e + a.ns - 1) / a.ns;
  a.slots_round = std::max(1, std::min(a.chunk, MAX_ROUND_ROWS / a.blk));
  // several staging rounds per CTA on the plain streamed path with narrow groups:
  // per-warp online softmax (one barrier per round instead of three)
  a.wflash = (a.tma_kv && !a.f8 && !a.mask && !a.block_table && !a.n_rows && a.G <= 8 &&
              a.chunk * a.blk > MAX_ROUND_ROWS) ? 1 : 0;
  const int nblk8 = (a.nblk + 7) & ~7;
  // blocks scored per CTA; with at most HSA_SPEC_MAX_COLS of them every KT row of
  // the CTA's blocks is prefetched at launch, otherwise the chosen rows are
  // gathered in chunks after the channel choice
  // (e4m3 codes: 16 blocks per 16-byte KT chunk)
  const int cq = a.f8 ? 16 : 8;
  const uint32_t eb = a.f8 ? 1u : 2u;
  a.cpr = std::max(cq, (((a.nblk + a.ns - 1) / a.ns) + cq - 1) / cq * cq);
  a.kt_spec = a.cpr <= HSA_SPEC_MAX_COLS ? 1 : 0;
  int bc = a.cpr;
  if ((uint32_t)a.k1 * bc * eb > KT_TILE_BUDGET) bc = std::max(cq, (int)(KT_TILE_BUDGET / (eb * a.k1)) / cq * cq);
  a.kt_chunk = bc;
  const uint32_t kt_tile_bytes = a.kt_spec ? 2u * HD * a.cpr * eb : eb * a.k1 * bc;
  const int gown = (a.G + a.ns - 1) / a.ns;
  auto al = [](uint32_t x, uint32_t q) { return (x + q - 1) / q * q; };
  uint32_t off = al(sizeof(FixedSmem), 128);
  a.off_x = 0;
  a.off_scores = off;
  off = al(off + 4u * (uint32_t)nblk8, 16);
  a.off_flags = off;
  off = al(off + (uint32_t)nblk8, 16);
  a.off_sel = off;
  off = al(off + 4u * (uint32_t)std::max(a.k2e, 1), 16);
  a.off_bt = off;
  if (a.block_table) off = al(off + 4u * (uint32_t)nblk8, 16);
  a.off_recv = off;
  off = al(off + 4u * gown * a.ns * PART_STRIDE, 1024);
  a.off_tiles = off;                       // K/V tiles; the KT gather tile shares this region
  const uint32_t rows16 = al((uint32_t)(a.slots_round * a.blk), 16);
  // (per-warp softmax: every warp owns 16 rows of each half tile for its partial)
  a.tile_half_bytes = a.wflash ? (uint32_t)MAX_ROUND_ROWS * 128u : rows16 * 128u;
  off += std::max(4u * a.tile_half_bytes, al(kt_tile_bytes, 16));
  a.smem_bytes = off + 1024u;   // room to align the base to 1024 bytes
  return a.smem_bytes <= 227u * 1024u;
}

cudaError_t hsa_launch(const HsaArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmKT,
                       bool mt, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const void* ks[13] = {
        (const void*)hsa_decode_kernel<false, 1, false, false, false, false, true>,
        (const void*)hsa_decode_kernel<false, 1, false, false, false, true>,
        (const void*)hsa_decode_kernel<false, 2, false, false, false, true>,
        (const void*)hsa_decode_kernel<false, 1, false, false, true>,
        (const void*)hsa_decode_kernel<false, 2, false, false, true>,
        (const void*)hsa_decode_kernel<false, 1, false, false>, (const void*)hsa_decode_kernel<false, 2, false, false>,
        (const void*)hsa_decode_kernel<true, 1, false, false>, (const void*)hsa_decode_kernel<true, 2, false, false>,
        (const void*)hsa_decode_kernel<false, 1, true, false>, (const void*)hsa_decode_kernel<false, 2, true, false>,
        (const void*)hsa_decode_kernel<false, 1, true, true>, (const void*)hsa_decode_kernel<false, 2, true, true>};
    for (const void* k : ks) {
      attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (attr_err != cudaSuccess) break;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ns, a.Hkv, a.B);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // per-row lengths (ragged batches) take their own instantiation: the uniform
  // kernels keep every length a launch constant
  const bool wide = a.G > 8;
  auto kern = mt ? (wide ? hsa_decode_kernel<true, 2, false, false> : hsa_decode_kernel<true, 1, false, false>)
          : a.f8 ? (wide ? hsa_decode_kernel<false, 2, false, false, false, true>
                         : hsa_decode_kernel<false, 1, false, false, false, true>)
          : a.mask ? (wide ? hsa_decode_kernel<false, 2, false, false, true>
                           : hsa_decode_kernel<false, 1, false, false, true>)
          : a.block_table ? (wide ? hsa_decode_kernel<false, 2, true, true> : hsa_decode_kernel<false, 1, true, true>)
          : a.n_rows ? (wide ? hsa_decode_kernel<false, 2, true, false> : hsa_decode_kernel<false, 1, true, false>)
          : a.wflash ? hsa_decode_kernel<false, 1, false, false, false, false, true>
                     : (wide ? hsa_decode_kernel<false, 2, false, false> : hsa_decode_kernel<false, 1, false, false>);
  return cudaLaunchKernelEx(&cfg, kern, *tmK, *tmV, *tmKT, a);
}

unsigned int hsa_take_device_error() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_hsa_err, sizeof(v)) != cudaSuccess) return ~0u;
  cudaMemcpyToSymbol(g_hsa_err, &z, sizeof(z));
  return v;
}

}  // namespace rkv
