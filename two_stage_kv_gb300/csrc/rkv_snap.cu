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
//   snap_compact  gather of the kept K and V rows (skipped in MT mask mode).
// The two score passes stream K with 3-D TMA tiles (128-byte swizzle) through
// a 4-stage mbarrier ring and run Q K^T on bf16 mma.sync with fp32 accumulation.
#include "rkv_common.cuh"
#include "rkv_internal.h"

#include <algorithm>

namespace rkv {

static __device__ unsigned int g_snap_err = 0;

namespace {

constexpr int P_NT = 256;          // 8 warps x 16 query rows = 128 rows per CTA
constexpr int P_ROWS = 128;
constexpr int P_TILE = 64;         // keys per TMA tile
constexpr int P_NST = 4;           // pipeline depth
constexpr int P_CHUNK = 2048;      // keys per CTA
constexpr uint32_t P_HALF = P_TILE * 128;            // one 64-dim half of a tile
constexpr uint32_t P_STAGE = 2 * P_HALF;             // 16 KB
constexpr uint32_t P_SMEM = P_NST * P_STAGE + 2 * 8 * P_TILE * 4 + 64 + 1024;

struct PassArgs {
  const bf16* q_obs;
  int64_t S, L;                    // L = S - W prefix keys
  int32_t Hq, Hkv, G, W, R, RG, nchunk1;
  float scale_log2;
  float2* stats;                   // [pairs][R][nchunk1]
  float* scores;                   // [pairs][RG][L]
};

template <int PASS>
__global__ void __launch_bounds__(P_NT) snap_pass_kernel(const __grid_constant__ CUtensorMap tmK, const PassArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* tiles = smem;
  float* colsum = reinterpret_cast<float*>(smem + P_NST * P_STAGE);       // [2][8][64]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_NST * P_STAGE + 2 * 8 * P_TILE * 4);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.z, rg = blockIdx.y, chunk = blockIdx.x;
  const int b = pair / a.Hkv, hk = pair % a.Hkv;
  const int64_t kend = (PASS == 1) ? a.S : a.L;
  const int64_t j0 = (int64_t)chunk * P_CHUNK;
  const int64_t j1 = min(kend, j0 + (int64_t)P_CHUNK);
  const int ntiles = (int)((j1 - j0 + P_TILE - 1) / P_TILE);

  if (tid == 0) {
    prefetch_tmap(&tmK);
    for (int s = 0; s < P_NST; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) {
    for (int it = 0; it < min(P_NST, ntiles); ++it) {
      const int y = (int)(j0 + (int64_t)it * P_TILE);
      mbar_arrive_expect_tx(&full[it], P_STAGE);
      tma_load_3d(tiles + it * P_STAGE, &tmK, 0, y, pair, &full[it]);
      tma_load_3d(tiles + it * P_STAGE + P_HALF, &tmK, 64, y, pair, &full[it]);
    }
  }

  // Query A fragments of this warp's 16 rows (rows >= R are zero).
  const int rw = rg * P_ROWS + warp * 16;
  const int ra = rw + (lane >> 2), rb = ra + 8;
  const bf16* qbase = a.q_obs + ((size_t)b * a.Hq + (size_t)hk * a.G) * a.W * HD;
  uint32_t qa[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = ks * 16 + 2 * (lane & 3);
    qa[ks][0] = ra < a.R ? *reinterpret_cast<const uint32_t*>(qbase + (size_t)ra * HD + c) : 0u;
    qa[ks][1] = rb < a.R ? *reinterpret_cast<const uint32_t*>(qbase + (size_t)rb * HD + c) : 0u;
    qa[ks][2] = ra < a.R ? *reinterpret_cast<const uint32_t*>(qbase + (size_t)ra * HD + c + 8) : 0u;
    qa[ks][3] = rb < a.R ? *reinterpret_cast<const uint32_t*>(qbase + (size_t)rb * HD + c + 8) : 0u;
  }
  const bool va = ra < a.R, vb = rb < a.R;
  // last key each window row may attend (causal): S - W + (row mod W)
  const int64_t lima = a.S - a.W + (ra % a.W), limb = a.S - a.W + (rb % a.W);

  float m_a = neg_inf(), m_b = neg_inf(), l_a = 0.f, l_b = 0.f;   // pass 1
  float lse_a = __int_as_float(0x7f800000), lse_b = lse_a;         // pass 2 (log2 units)
  if (PASS == 2) {
    auto lse_of = [&](int r) {
      const float2* st = a.stats + ((size_t)pair * a.R + r) * a.nchunk1;
      float M = neg_inf();
      for (int c = 0; c < a.nchunk1; ++c) M = fmaxf(M, st[c].x);
      float Ls = 0.f;
      for (int c = 0; c < a.nchunk1; ++c)
        if (st[c].x != neg_inf()) Ls += st[c].y * exp2f(st[c].x - M);
      return M + log2f(Ls);
    };
    if (va) lse_a = lse_of(ra);
    if (vb) lse_b = lse_of(rb);
  }

  unsigned int* err = &g_snap_err;
  for (int it = 0; it < ntiles; ++it) {
    const int st = it % P_NST;
    if (!mbar_wait(&full[st], (uint32_t)((it / P_NST) & 1), err)) mbar_wait(&full[st], (uint32_t)((it / P_NST) & 1), err);
    const uint32_t tb = smem_u32(tiles + st * P_STAGE);
    const int64_t jt = j0 + (int64_t)it * P_TILE;

    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int r = nt * 8 + (lane & 7);
        const int ch = ks * 2 + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tb + (uint32_t)(ch >> 3) * P_HALF + swz128(r, ch & 7), b0, b1, b2, b3);
        mma_bf16(sc[nt], qa[ks], b0, b1);
        mma_bf16(sc[nt], qa[ks + 1], b2, b3);
      }
    }

    if (PASS == 1) {
      float xa[16], xb[16];
      float ma = neg_inf(), mb = neg_inf();
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t j = jt + nt * 8 + 2 * (lane & 3) + e;
          const float x0 = (va && j < a.S && j <= lima) ? sc[nt][e] * a.scale_log2 : neg_inf();
          const float x1 = (vb && j < a.S && j <= limb) ? sc[nt][2 + e] * a.scale_log2 : neg_inf();
          xa[nt * 2 + e] = x0;
          xb[nt * 2 + e] = x1;
          ma = fmaxf(ma, x0);
          mb = fmaxf(mb, x1);
        }
      }
      const float na = fmaxf(m_a, ma), nb = fmaxf(m_b, mb);
      float sa = 0.f, sb = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        sa += (xa[i] == neg_inf()) ? 0.f : exp2f(xa[i] - na);
        sb += (xb[i] == neg_inf()) ? 0.f : exp2f(xb[i] - nb);
      }
      l_a = ((m_a == neg_inf()) ? 0.f : l_a * exp2f(m_a - na)) + sa;
      l_b = ((m_b == neg_inf()) ? 0.f : l_b * exp2f(m_b - nb)) + sb;
      m_a = na;
      m_b = nb;
      __syncthreads();
    } else {
      float* cs = colsum + (it & 1) * 8 * P_TILE + warp * P_TILE;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t j = jt + nt * 8 + 2 * (lane & 3) + e;
          const bool kj = j < a.L;
          const float pa = (va && kj) ? exp2f(sc[nt][e] * a.scale_log2 - lse_a) : 0.f;
          const float pb = (vb && kj) ? exp2f(sc[nt][2 + e] * a.scale_log2 - lse_b) : 0.f;
          float s = pa + pb;
          s += __shfl_xor_sync(0xffffffffu, s, 4);
          s += __shfl_xor_sync(0xffffffffu, s, 8);
          s += __shfl_xor_sync(0xffffffffu, s, 16);
          v[e] = s;
        }
        if (lane < 4) {
          cs[nt * 8 + 2 * lane] = v[0];
          cs[nt * 8 + 2 * lane + 1] = v[1];
        }
      }
      __syncthreads();
      if (tid < P_TILE) {
        const float* c2 = colsum + (it & 1) * 8 * P_TILE;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += c2[w * P_TILE + tid];
        const int64_t j = jt + tid;
        if (j < a.L) a.scores[((size_t)pair * a.RG + rg) * a.L + j] = s;
      }
    }
    if (tid == 0 && it + P_NST < ntiles) {
      fence_proxy_async_smem();
      const int y = (int)(j0 + (int64_t)(it + P_NST) * P_TILE);
      mbar_arrive_expect_tx(&full[st], P_STAGE);
      tma_load_3d(tiles + st * P_STAGE, &tmK, 0, y, pair, &full[st]);
      tma_load_3d(tiles + st * P_STAGE + P_HALF, &tmK, 64, y, pair, &full[st]);
    }
  }

  if (PASS == 1) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      const float moa = __shfl_xor_sync(0xffffffffu, m_a, o), loa = __shfl_xor_sync(0xffffffffu, l_a, o);
      const float mob = __shfl_xor_sync(0xffffffffu, m_b, o), lob = __shfl_xor_sync(0xffffffffu, l_b, o);
      const float na = fmaxf(m_a, moa), nb = fmaxf(m_b, mob);
      l_a = ((m_a == neg_inf()) ? 0.f : l_a * exp2f(m_a - na)) + ((moa == neg_inf()) ? 0.f : loa * exp2f(moa - na));
      l_b = ((m_b == neg_inf()) ? 0.f : l_b * exp2f(m_b - nb)) + ((mob == neg_inf()) ? 0.f : lob * exp2f(mob - nb));
      m_a = na;
      m_b = nb;
    }
    if ((lane & 3) == 0) {
      if (va) a.stats[((size_t)pair * a.R + ra) * a.nchunk1 + chunk] = make_float2(m_a, l_a);
      if (vb) a.stats[((size_t)pair * a.R + rb) * a.nchunk1 + chunk] = make_float2(m_b, l_b);
    }
  }
}

// Sum of the row-group partials (fixed order), then max-pool (clipped ends).
constexpr int POOL_TILE = 1024;
constexpr int POOL_MAX_HALF = 512;

__global__ void __launch_bounds__(256) snap_pool_kernel(const float* scores, int RG, int64_t L, int half,
                                                        float* pooled) {
  __shared__ float tile[POOL_TILE + 2 * POOL_MAX_HALF];
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  const int64_t j0 = (int64_t)blockIdx.x * POOL_TILE;
  const int span = POOL_TILE + 2 * half;
  for (int i = threadIdx.x; i < span; i += blockDim.x) {
    const int64_t j = j0 - half + i;
    float v = neg_inf();
    if (j >= 0 && j < L) {
      v = 0.f;
      for (int r = 0; r < RG; ++r) v += scores[((size_t)pair * RG + r) * L + j];
    }
    tile[i] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < POOL_TILE; i += blockDim.x) {
    const int64_t j = j0 + i;
    if (j >= L) break;
    float m = tile[i];
    for (int t = 1; t <= 2 * half; ++t) m = fmaxf(m, tile[i + t]);
    pooled[(size_t)pair * L + j] = m;
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

__global__ void __launch_bounds__(SEL_NT) snap_select_kernel(const float* pooled, int64_t L, int64_t S, int W,
                                                             int n_sink, int64_t ntop, int64_t B1,
                                                             int32_t* keep, int64_t keep_ld) {
  __shared__ int hist[256];
  __shared__ int wsum[72];
  __shared__ uint32_t sh_digit;
  __shared__ int64_t sh_k;
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.x, tid = threadIdx.x;
  const float* p = pooled + (size_t)pair * L;
  int32_t* out = keep + (size_t)pair * keep_ld;
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

// K_c[i] = K[keep[i]], V_c[i] = V[keep[i]].
__global__ void __launch_bounds__(256) snap_compact_kernel(const bf16* k, const bf16* v, int64_t cap,
                                                           const int32_t* keep, int64_t keep_ld, int64_t B1,
                                                           bf16* ko, bf16* vo, int64_t out_cap) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  for (int i = threadIdx.x; i < 32 * 16; i += blockDim.x) {
    const int64_t row = (int64_t)blockIdx.x * 32 + i / 16;
    const int ch = i % 16;
    if (row >= B1) break;
    const int64_t src = min(max((int64_t)keep[(size_t)pair * keep_ld + row], (int64_t)0), cap - 1);
    const uint4 kv = *reinterpret_cast<const uint4*>(k + ((size_t)pair * cap + src) * HD + ch * 8);
    const uint4 vv = *reinterpret_cast<const uint4*>(v + ((size_t)pair * cap + src) * HD + ch * 8);
    *reinterpret_cast<uint4*>(ko + ((size_t)pair * out_cap + row) * HD + ch * 8) = kv;
    *reinterpret_cast<uint4*>(vo + ((size_t)pair * out_cap + row) * HD + ch * 8) = vv;
  }
}

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t snap_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int64_t S, int32_t W) {
  const int64_t pairs = (int64_t)B * Hkv;
  const int G = Hq / Hkv;
  const int64_t R = (int64_t)G * W;
  const int64_t RG = (R + P_ROWS - 1) / P_ROWS;
  const int64_t L = std::max<int64_t>(S - W, 0);
  const int64_t nchunk1 = (S + P_CHUNK - 1) / P_CHUNK;
  return al256((size_t)pairs * R * nchunk1 * sizeof(float2)) + al256((size_t)pairs * RG * L * sizeof(float)) +
         al256((size_t)pairs * L * sizeof(float));
}

cudaError_t snap_launch(const SnapArgs& a, const CUtensorMap* tmK, cudaStream_t st) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(snap_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(snap_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int pairs = a.B * a.Hkv;
  const int W = (int)std::min<int64_t>(a.W, a.S);
  const int64_t L = a.S - W;
  const bool keep_all = a.B1 >= a.S || L <= 0;
  if (!keep_all) {
    PassArgs p;
    p.q_obs = reinterpret_cast<const bf16*>(a.q_obs);
    p.S = a.S;
    p.L = L;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.G;
    p.W = W;
    p.R = a.G * W;
    p.RG = (p.R + P_ROWS - 1) / P_ROWS;
    p.nchunk1 = (int)((a.S + P_CHUNK - 1) / P_CHUNK);
    p.scale_log2 = a.scale_log2;
    uint8_t* w = reinterpret_cast<uint8_t*>(a.ws);
    p.stats = reinterpret_cast<float2*>(w);
    w += al256((size_t)pairs * p.R * p.nchunk1 * sizeof(float2));
    p.scores = reinterpret_cast<float*>(w);
    w += al256((size_t)pairs * p.RG * L * sizeof(float));
    float* pooled = a.pooled_out ? a.pooled_out : reinterpret_cast<float*>(w);

    cudaError_t e = launch_pdl(snap_pass_kernel<1>, dim3(p.nchunk1, p.RG, pairs), dim3(P_NT), P_SMEM, st, *tmK, p);
    if (e != cudaSuccess) return e;
    const int nchunk2 = (int)((L + P_CHUNK - 1) / P_CHUNK);
    e = launch_pdl(snap_pass_kernel<2>, dim3(nchunk2, p.RG, pairs), dim3(P_NT), P_SMEM, st, *tmK, p);
    if (e != cudaSuccess) return e;
    e = launch_pdl(snap_pool_kernel, dim3((unsigned)((L + POOL_TILE - 1) / POOL_TILE), pairs), dim3(256), 0, st,
                   (const float*)p.scores, (int)p.RG, (int64_t)L, (int)(a.pool / 2), pooled);
    if (e != cudaSuccess) return e;
    const int n_sink = (int)std::max<int64_t>(0, std::min<int64_t>(a.n_sink, L));
    const int64_t ntop = std::max<int64_t>(0, a.B1 - W - n_sink);
    e = launch_pdl(snap_select_kernel, dim3(pairs), dim3(SEL_NT), 0, st, (const float*)pooled, (int64_t)L,
                   (int64_t)a.S, (int)W, (int)n_sink, (int64_t)ntop, (int64_t)a.B1, a.keep, (int64_t)a.keep_ld);
    if (e != cudaSuccess) return e;
  } else {
    // every token kept: keep = 0..S-1 (B1 == S enforced by the caller)
    cudaError_t e = launch_pdl(snap_select_kernel, dim3(pairs), dim3(SEL_NT), 0, st, (const float*)nullptr, (int64_t)0,
                               (int64_t)a.S, (int)a.S, 0, (int64_t)0, (int64_t)a.B1, a.keep, (int64_t)a.keep_ld);
    if (e != cudaSuccess) return e;
  }
  if (a.k_out) {
    cudaError_t e = launch_pdl(snap_compact_kernel, dim3((unsigned)((a.B1 + 31) / 32), pairs), dim3(256), 0, st,
                               reinterpret_cast<const bf16*>(a.k), reinterpret_cast<const bf16*>(a.v), (int64_t)a.cap,
                               (const int32_t*)a.keep, (int64_t)a.keep_ld, (int64_t)a.B1,
                               reinterpret_cast<bf16*>(a.k_out), reinterpret_cast<bf16*>(a.v_out), (int64_t)a.out_cap);
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
