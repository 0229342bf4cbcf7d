// Stage 2 of RocketKV: one Hybrid Sparse Attention decode step per launch.
//
// Method: "RocketKV: Accelerating Long-Context LLM Inference via Two-Stage KV
// Cache Compression" (papercache digest), section 方法细节, HSA steps 2-3 and
// Algorithm 1 (top-k1 channels of the group sum of |q|, sign of the group sum
// of q, sign-selected Kmax/Kmin page scores, top-k2 pages, exact attention over
// the selected pages); RocketKV-MT for the candidate-restricted variant.
//
// GB300 design.  One thread-block cluster of `ns` CTAs (128 threads each) per
// (batch row, KV head).  Every CTA of the cluster:
//   A. loads the group's G query rows, forms sum|q| and sum q per channel in
//      fp64 (exact for bf16 inputs) and picks the k1 channels by rank;
//   B. scores its 1/ns slice of the blocks from the channel-major KT cache
//      (coalesced rows along the block axis) and broadcasts the scores to
//      every CTA of the cluster through distributed shared memory;
//   C. ranks its own slice against all scores (strict order: score, then
//      lower block index) and broadcasts the winners' ranks as slots;
//   D. TMA-loads the K and V rows of its share of the selected blocks into
//      128-byte-swizzled shared tiles, runs QK^T and PV with bf16 mma.sync
//      (G query rows padded to 16; P split into bf16 hi + lo so the PV product
//      keeps ~16 mantissa bits) and an online softmax in fp32;
//   E. merges its warps' partial (max, sum, acc), sends the per-head partial to
//      the CTA that owns that head, and the owners combine the ns partials and
//      write fp32 outputs.  No global scratch, no atomics, no inter-CTA spins:
//      the only cluster waits are hardware cluster barriers.
#include "rkv_common.cuh"
#include "rkv_internal.h"

#include <algorithm>

namespace rkv {

static __device__ unsigned int g_hsa_err = 0;

namespace {

constexpr int NT = 128;          // threads per CTA
constexpr int NWARP = NT / 32;
constexpr int PART_STRIDE = HD + 2;   // acc[128], max, sum
constexpr uint32_t FIXED_SMEM = 8192;
constexpr int MAX_ROUND_ROWS = 256;

// Fixed shared-memory region (first FIXED_SMEM bytes).
struct FixedSmem {
  bf16 qs[16][HD];            // 4096: query rows, rows >= G are zero
  uint64_t akey[HD];          // 1024: bits of sum|q| (non-negative doubles order like integers)
  double qbar[HD];            // 1024: sum q
  float qsel[HD];             //  512: qbar of the kept channels, ascending channel order
  int32_t rowoff[HD];         //  512: KT row (0..2D) of each kept channel
  uint64_t mbar[2];           //   16
  int32_t wcount[NWARP];      //   16
  int32_t nvalid[MAX_ROUND_ROWS / 8];  // valid tokens of each staged block
};
static_assert(sizeof(FixedSmem) <= FIXED_SMEM, "fixed smem");

template <bool MT>
__global__ void __launch_bounds__(NT) hsa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                        const __grid_constant__ CUtensorMap tmV,
                                                        const HsaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  FixedSmem& fs = *reinterpret_cast<FixedSmem*>(smem);
  uint32_t* skey = reinterpret_cast<uint32_t*>(smem + a.off_scores);
  int32_t* sel = reinterpret_cast<int32_t*>(smem + a.off_sel);
  float* part = reinterpret_cast<float*>(smem + a.off_part);
  float* recv = reinterpret_cast<float*>(smem + a.off_recv);
  uint8_t* tK = smem + a.off_tiles;
  uint8_t* tV = tK + 2 * a.tile_half_bytes;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int ns = a.ns;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int pair = b * a.Hkv + hk;
  const int G = a.G;

  // Every CTA of the cluster must have started before any DSMEM store lands
  // in it; the matching wait sits just before the first remote store.
  cluster_arrive_relaxed();

  if (!MT && tid == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }

  // ---------------------------------------------------------------- A ------
  {
    const bf16* qg = reinterpret_cast<const bf16*>(a.q) + ((size_t)b * a.Hq + (size_t)hk * G) * HD;
    for (int i = tid; i < 16 * (HD / 8); i += NT) {
      const int r = i / (HD / 8), c = i % (HD / 8);
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < G) val = *reinterpret_cast<const uint4*>(qg + (size_t)r * HD + c * 8);
      *reinterpret_cast<uint4*>(&fs.qs[r][c * 8]) = val;
    }
  }
  if (tid == 0) {
    mbar_init(&fs.mbar[0], 1);
    fence_mbar_init();
  }
  // pad the score keys up to a multiple of 4 with the smallest key
  {
    const int npad = (a.nblk + 3) & ~3;
    for (int j = a.nblk + tid; j < npad; j += NT) skey[j] = 0u;
  }
  __syncthreads();
  {
    const int c = tid;  // NT == HD: one thread per channel
    double sa = 0.0, sq = 0.0;
    for (int g = 0; g < G; ++g) {
      const double x = (double)bf2f(fs.qs[g][c]);
      sa += fabs(x);
      sq += x;
    }
    fs.akey[c] = (uint64_t)__double_as_longlong(sa);
    fs.qbar[c] = sq;
  }
  __syncthreads();
  {
    const int c = tid;
    const uint64_t mine = fs.akey[c];
    int rk = 0;
#pragma unroll 8
    for (int j = 0; j < HD; ++j) {
      const uint64_t o = fs.akey[j];
      rk += (o > mine) || (o == mine && j < c);
    }
    const bool take = rk < a.k1;
    const unsigned bal = __ballot_sync(0xffffffffu, take);
    if (lane == 0) fs.wcount[warp] = __popc(bal);
    __syncthreads();
    int pos = __popc(bal & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) pos += fs.wcount[w];
    if (take) {
      const double qb = fs.qbar[c];
      fs.qsel[pos] = (float)qb;
      fs.rowoff[pos] = (qb >= 0.0 ? 0 : HD) + c;   // Kmax if the group sum is >= 0
      if (rank == 0 && a.sel_channels) a.sel_channels[(size_t)pair * a.k1 + pos] = c;
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- B ------
  const int per = (a.nblk + ns - 1) / ns;
  const int lo = (int)rank * per;
  const int hi = min(a.nblk, lo + per);
  cluster_wait_acquire();   // pairs with the relaxed arrive at entry
  {
    const bf16* ktp = reinterpret_cast<const bf16*>(a.kt) + (size_t)pair * 2 * HD * a.nblk_cap;
    const int k1 = a.k1;
    for (int j = lo + tid; j < hi; j += NT) {
      float s = 0.f;
      int i = 0;
      for (; i + 8 <= k1; i += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = bf2f(ktp[(size_t)fs.rowoff[i + u] * a.nblk_cap + j]);
#pragma unroll
        for (int u = 0; u < 8; ++u) s = fmaf(fs.qsel[i + u], v[u], s);
      }
      for (; i < k1; ++i) s = fmaf(fs.qsel[i], bf2f(ktp[(size_t)fs.rowoff[i] * a.nblk_cap + j]), s);
      const uint32_t key = f2key(s);
      const uint32_t laddr = smem_u32(&skey[j]);
      for (int d = 0; d < ns; ++d) st_cluster_u32(mapa(laddr, d), key);
    }
  }
  cluster_sync();

  // ---------------------------------------------------------------- C ------
  {
    const int nq = (a.nblk + 3) >> 2;
    const uint4* sk4 = reinterpret_cast<const uint4*>(skey);
    for (int j = lo + tid; j < hi; j += NT) {
      const uint32_t mine = skey[j];
      int rk = 0;
      for (int o4 = 0; o4 < nq; ++o4) {
        const uint4 k4 = sk4[o4];
        const int o = o4 * 4;
        rk += (k4.x > mine) | ((k4.x == mine) & (o + 0 < j));
        rk += (k4.y > mine) | ((k4.y == mine) & (o + 1 < j));
        rk += (k4.z > mine) | ((k4.z == mine) & (o + 2 < j));
        rk += (k4.w > mine) | ((k4.w == mine) & (o + 3 < j));
      }
      if (rk < a.k2e) {
        const uint32_t laddr = smem_u32(&sel[rk]);
        for (int d = 0; d < ns; ++d) st_cluster_u32(mapa(laddr, d), (uint32_t)j);
      }
    }
  }
  cluster_sync();

  // ---------------------------------------------------------------- D ------
  // Query A fragments (16 rows x 128 dims) for the 8 k-steps.
  uint32_t qa[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int col = ks * 16 + (lane >> 4) * 8;
    ldsm_x4(smem_u32(&fs.qs[row][col]), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
  }

  float m_run[2] = {neg_inf(), neg_inf()};
  float l_run[2] = {0.f, 0.f};
  float acc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int s_lo = (int)rank * a.chunk;
  const int s_hi = min(a.k2e, s_lo + a.chunk);
  const uint32_t half = a.tile_half_bytes;
  const int blk = a.blk;
  uint32_t phase = 0;
  unsigned int* err = &g_hsa_err;

  for (int r0 = s_lo; r0 < s_hi; r0 += a.slots_round) {
    const int nsl = min(a.slots_round, s_hi - r0);
    const int rows = nsl * blk;
    const int rows16 = (rows + 15) & ~15;
    if (tid < nsl) fs.nvalid[tid] = min(blk, a.n - sel[r0 + tid] * blk);
    if (!MT) {
      if (tid == 0) {
        if (r0 != s_lo) fence_proxy_async_smem();
        mbar_arrive_expect_tx(&fs.mbar[0], (uint32_t)nsl * blk * 128u * 4u);
        for (int s = 0; s < nsl; ++s) {
          const int y = sel[r0 + s] * blk;
          const uint32_t off = (uint32_t)s * blk * 128u;
          tma_load_3d(tK + off, &tmK, 0, y, pair, &fs.mbar[0]);
          tma_load_3d(tK + half + off, &tmK, 64, y, pair, &fs.mbar[0]);
          tma_load_3d(tV + off, &tmV, 0, y, pair, &fs.mbar[0]);
          tma_load_3d(tV + half + off, &tmV, 64, y, pair, &fs.mbar[0]);
        }
      }
    } else {
      const bf16* kb = reinterpret_cast<const bf16*>(a.k) + (size_t)pair * a.cap * HD;
      const bf16* vb = reinterpret_cast<const bf16*>(a.v) + (size_t)pair * a.cap * HD;
      const int32_t* ib = a.idx + (size_t)pair * a.idx_cap;
      for (int i = tid; i < rows * 16; i += NT) {
        const int r = i >> 4, ch = i & 15;
        const int slot = r / blk;
        const int t = sel[r0 + slot] * blk + (r - slot * blk);
        const uint32_t o = (uint32_t)(ch >> 3) * half + swz128(r, ch & 7);
        if (t < a.n) {
          const int64_t prow = min(max((int64_t)ib[t], (int64_t)0), a.cap - 1);
          cp_async_16(smem_u32(tK) + o, kb + prow * HD + ch * 8);
          cp_async_16(smem_u32(tV) + o, vb + prow * HD + ch * 8);
        } else {
          *reinterpret_cast<uint4*>(tK + o) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(tV + o) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
    }
    // Rows [rows, rows16) of the V tile feed the last PV step with P = 0; keep them finite.
    for (int i = tid; i < (rows16 - rows) * 16; i += NT) {
      const int r = rows + (i >> 4), ch = i & 15;
      *reinterpret_cast<uint4*>(tV + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7)) = make_uint4(0, 0, 0, 0);
    }
    if (!MT) {
      if (!mbar_wait(&fs.mbar[0], phase, err)) mbar_wait(&fs.mbar[0], phase, err);
      phase ^= 1u;
    } else {
      cp_async_wait_all();
    }
    __syncthreads();

    for (int c0 = warp * 16; c0 < rows; c0 += NWARP * 16) {
      // S = Q K^T over tokens c0 .. c0+15 (two n-tiles of 8 tokens)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 8; ks += 2) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int r = c0 + nt * 8 + (lane & 7);
          const int ch = ks * 2 + (lane >> 3);        // 16-byte chunk of the 128 dims
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tK) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7), b0, b1, b2, b3);
          mma_bf16(sc[nt], qa[ks], b0, b1);
          mma_bf16(sc[nt], qa[ks + 1], b2, b3);
        }
      }
      // mask, scale to log2 units, online softmax
      float x[2][4];
      float mx0 = neg_inf(), mx1 = neg_inf();
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = c0 + nt * 8 + 2 * (lane & 3) + (e & 1);
          const int slot = r / blk;
          const bool valid = (r < rows) && (r - slot * blk < fs.nvalid[min(slot, nsl - 1)]);
          const float v = valid ? sc[nt][e] * a.scale_log2 : neg_inf();
          x[nt][e] = v;
          if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      const float c0f = (m_run[0] == neg_inf()) ? 0.f : exp2f(m_run[0] - mn0);
      const float c1f = (m_run[1] == neg_inf()) ? 0.f : exp2f(m_run[1] - mn1);
      m_run[0] = mn0;
      m_run[1] = mn1;
      float p[2][4];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mref = (e < 2) ? mn0 : mn1;
          const float pv = (x[nt][e] == neg_inf()) ? 0.f : exp2f(x[nt][e] - mref);
          p[nt][e] = pv;
          if (e < 2) ps0 += pv; else ps1 += pv;
        }
      }
      l_run[0] = l_run[0] * c0f + ps0;
      l_run[1] = l_run[1] * c1f + ps1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        acc[i][0] *= c0f;
        acc[i][1] *= c0f;
        acc[i][2] *= c1f;
        acc[i][3] *= c1f;
      }
      // P as the A operand (rows = heads, k = 16 tokens), split hi + lo
      uint32_t ph[4], pl[4];
      ph[0] = pack_bf16(p[0][0], p[0][1]);
      ph[1] = pack_bf16(p[0][2], p[0][3]);
      ph[2] = pack_bf16(p[1][0], p[1][1]);
      ph[3] = pack_bf16(p[1][2], p[1][3]);
      pl[0] = pack_bf16(p[0][0] - bf16_lo(ph[0]), p[0][1] - bf16_hi(ph[0]));
      pl[1] = pack_bf16(p[0][2] - bf16_lo(ph[1]), p[0][3] - bf16_hi(ph[1]));
      pl[2] = pack_bf16(p[1][0] - bf16_lo(ph[2]), p[1][1] - bf16_hi(ph[2]));
      pl[3] = pack_bf16(p[1][2] - bf16_lo(ph[3]), p[1][3] - bf16_hi(ph[3]));
#pragma unroll
      for (int dt = 0; dt < 16; dt += 2) {
        const int r = c0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = dt + (lane >> 4);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(smem_u32(tV) + (uint32_t)(ch >> 3) * half + swz128(r, ch & 7), v0, v1, v2, v3);
        mma_bf16(acc[dt], ph, v0, v1);
        mma_bf16(acc[dt], pl, v0, v1);
        mma_bf16(acc[dt + 1], ph, v2, v3);
        mma_bf16(acc[dt + 1], pl, v2, v3);
      }
    }
    __syncthreads();   // tiles are reused by the next round
  }

  // ---------------------------------------------------------------- E ------
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
  {
    const int g0 = lane >> 2, g1 = g0 + 8;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      const int d = dt * 8 + 2 * (lane & 3);
      if (g0 < G) {
        float* pp = part + (size_t)(warp * G + g0) * PART_STRIDE + d;
        pp[0] = acc[dt][0];
        pp[1] = acc[dt][1];
      }
      if (g1 < G) {
        float* pp = part + (size_t)(warp * G + g1) * PART_STRIDE + d;
        pp[0] = acc[dt][2];
        pp[1] = acc[dt][3];
      }
    }
    if ((lane & 3) == 0) {
      if (g0 < G) {
        part[(size_t)(warp * G + g0) * PART_STRIDE + HD] = m_run[0];
        part[(size_t)(warp * G + g0) * PART_STRIDE + HD + 1] = l_run[0];
      }
      if (g1 < G) {
        part[(size_t)(warp * G + g1) * PART_STRIDE + HD] = m_run[1];
        part[(size_t)(warp * G + g1) * PART_STRIDE + HD + 1] = l_run[1];
      }
    }
  }
  __syncthreads();
  const int gown = (G + ns - 1) / ns;
  for (int i = tid; i < G * HD; i += NT) {
    const int g = i / HD, d = i % HD;
    float M = neg_inf();
    for (int w = 0; w < NWARP; ++w) M = fmaxf(M, part[(size_t)(w * G + g) * PART_STRIDE + HD]);
    float A = 0.f, L = 0.f;
    for (int w = 0; w < NWARP; ++w) {
      const float* pp = part + (size_t)(w * G + g) * PART_STRIDE;
      const float f = (pp[HD] == neg_inf()) ? 0.f : exp2f(pp[HD] - M);
      A += f * pp[d];
      L += f * pp[HD + 1];
    }
    const int owner = g % ns, gl = g / ns;
    const uint32_t base = smem_u32(recv + ((size_t)rank * gown + gl) * PART_STRIDE);
    st_cluster_f32(mapa(base + 4u * d, owner), A);
    if (d == 0) {
      st_cluster_f32(mapa(base + 4u * HD, owner), M);
      st_cluster_f32(mapa(base + 4u * (HD + 1), owner), L);
    }
  }
  cluster_sync();
  for (int gl = 0; gl < gown; ++gl) {
    const int g = gl * ns + (int)rank;
    if (g >= G) break;
    const int d = tid;
    float M = neg_inf();
    for (int r = 0; r < ns; ++r) M = fmaxf(M, recv[((size_t)r * gown + gl) * PART_STRIDE + HD]);
    float A = 0.f, L = 0.f;
    for (int r = 0; r < ns; ++r) {
      const float* pp = recv + ((size_t)r * gown + gl) * PART_STRIDE;
      const float f = (pp[HD] == neg_inf()) ? 0.f : exp2f(pp[HD] - M);
      A += f * pp[d];
      L += f * pp[HD + 1];
    }
    a.out[((size_t)b * a.Hq + (size_t)hk * G + g) * HD + d] = A / L;
  }
  if (rank == 0 && a.sel_blocks) {
    for (int j = tid; j < a.k2; j += NT) {
      if (j < a.k2e) {
        const int mine = sel[j];
        int pos = 0;
        for (int o = 0; o < a.k2e; ++o) pos += sel[o] < mine;
        a.sel_blocks[(size_t)pair * a.k2 + pos] = mine;
      } else {
        a.sel_blocks[(size_t)pair * a.k2 + j] = -1;
      }
    }
  }
}

}  // namespace

bool hsa_plan(HsaArgs& a) {
  a.nblk = (a.n + a.blk - 1) / a.blk;
  a.k2e = std::min(a.k2, a.nblk);
  int ns = std::min(8, a.k2e);
  if (ns < 1) ns = 1;
  a.ns = ns;
  a.chunk = (a.k2e + ns - 1) / ns;
  a.slots_round = std::max(1, std::min(a.chunk, MAX_ROUND_ROWS / a.blk));
  const int gown = (a.G + ns - 1) / ns;
  auto al = [](uint32_t x, uint32_t q) { return (x + q - 1) / q * q; };
  uint32_t off = FIXED_SMEM;
  a.off_scores = off;
  off = al(off + 4u * (uint32_t)((a.nblk + 3) & ~3), 16);
  a.off_sel = off;
  off = al(off + 4u * (uint32_t)a.k2e, 16);
  a.off_part = off;
  off = al(off + 4u * NWARP * a.G * PART_STRIDE, 16);
  a.off_recv = off;
  off = al(off + 4u * ns * gown * PART_STRIDE, 1024);
  a.off_tiles = off;
  const uint32_t rows16 = al((uint32_t)(a.slots_round * a.blk), 16);
  a.tile_half_bytes = rows16 * 128u;
  off += 4u * a.tile_half_bytes;
  a.smem_bytes = off + 1024u;   // room to align the base to 1024 bytes
  return a.smem_bytes <= 227u * 1024u;
}

cudaError_t hsa_launch(const HsaArgs& a, const CUtensorMap* tmK, const CUtensorMap* tmV, bool mt,
                       cudaStream_t st) {
  static bool attr_done[2] = {false, false};
  auto kern = mt ? hsa_decode_kernel<true> : hsa_decode_kernel<false>;
  if (!attr_done[mt ? 1 : 0]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done[mt ? 1 : 0] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ns, a.Hkv, a.B);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.ns;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, *tmK, *tmV, a);
}

unsigned int hsa_take_device_error() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_hsa_err, sizeof(v)) != cudaSuccess) return ~0u;
  cudaMemcpyToSymbol(g_hsa_err, &z, sizeof(z));
  return v;
}

}  // namespace rkv
