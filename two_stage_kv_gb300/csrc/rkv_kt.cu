// The KT cache of RocketKV's Hybrid Sparse Attention: per block of `blk`
// consecutive (candidate) tokens, the elementwise maximum and minimum of the
// keys, stored channel-major so that the decode step gathers whole rows of
// k1 chosen channels.  Method: "RocketKV: Accelerating Long-Context LLM
// Inference via Two-Stage KV Cache Compression" (papercache digest), section
// 方法细节, HSA step 1 (pages of Kmax/Kmin aligned along the head dimension,
// updated whenever a new key is generated).
#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

constexpr int KT_BLOCKS = 64;     // blocks per CTA
constexpr int KT_NT = 256;

// One CTA per (pair, 64 blocks): warps reduce 8 blocks each over coalesced
// 256-byte key rows, the results are transposed in shared memory and written
// as 128-byte runs along the block axis.  With a mask (the multi-turn reading
// over fixed blocks of the full cache) only candidate rows count: prompt rows
// (< n_prompt) whose bit is set and every later row; a block without one
// stores zeros.
__global__ void __launch_bounds__(KT_NT) kt_build_kernel(const bf16* k, int64_t cap, int64_t n,
                                                         const int32_t* idx, int64_t idx_cap, int blk,
                                                         bf16* kt, int64_t nblk_cap, const uint32_t* mask,
                                                         int64_t mask_ld, int64_t n_prompt) {
  __shared__ bf16 tmax[HD][KT_BLOCKS + 2];
  __shared__ bf16 tmin[HD][KT_BLOCKS + 2];
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblk = (n + blk - 1) / blk;
  const int64_t jb0 = (int64_t)blockIdx.x * KT_BLOCKS;
  const bf16* kp = k + (size_t)pair * cap * HD;
  const int32_t* ip = idx ? idx + (size_t)pair * idx_cap : nullptr;
  const uint32_t* mp = mask ? mask + (size_t)pair * mask_ld : nullptr;
  for (int u = 0; u < KT_BLOCKS / 8; ++u) {
    const int jl = warp * (KT_BLOCKS / 8) + u;
    const int64_t jb = jb0 + jl;
    if (jb >= nblk) break;
    const int64_t t0 = jb * blk, t1 = min(n, t0 + blk);
    float mx[4], mn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mx[i] = neg_inf();
      mn[i] = -neg_inf();
    }
    bool any = false;
    for (int64_t t = t0; t < t1; ++t) {
      if (mp && t < n_prompt && ((__ldg(mp + (t >> 5)) >> (t & 31)) & 1u) == 0) continue;
      any = true;
      const int64_t row = ip ? min(max((int64_t)ip[t], (int64_t)0), cap - 1) : t;
      const uint2 raw = *reinterpret_cast<const uint2*>(kp + row * HD + lane * 4);
      const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
      mx[0] = fmaxf(mx[0], v0); mn[0] = fminf(mn[0], v0);
      mx[1] = fmaxf(mx[1], v1); mn[1] = fminf(mn[1], v1);
      mx[2] = fmaxf(mx[2], v2); mn[2] = fminf(mn[2], v2);
      mx[3] = fmaxf(mx[3], v3); mn[3] = fminf(mn[3], v3);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // values are bf16 already: the conversion back is exact
      tmax[lane * 4 + i][jl] = __float2bfloat16_rn(any ? mx[i] : 0.f);
      tmin[lane * 4 + i][jl] = __float2bfloat16_rn(any ? mn[i] : 0.f);
    }
  }
  __syncthreads();
  const int nb = (int)min((int64_t)KT_BLOCKS, nblk - jb0);
  bf16* base = kt + (size_t)pair * 2 * HD * nblk_cap;
  for (int i = threadIdx.x; i < 2 * HD * KT_BLOCKS; i += KT_NT) {
    const int row = i / KT_BLOCKS, jl = i % KT_BLOCKS;
    if (jl >= nb) continue;
    const int m = row / HD, c = row % HD;
    base[((size_t)m * HD + c) * nblk_cap + jb0 + jl] = m == 0 ? tmax[c][jl] : tmin[c][jl];
  }
}

// One CTA per pair, one thread per channel.
__global__ void __launch_bounds__(HD) append_kernel(const bf16* k_new, const bf16* v_new, bf16* k, bf16* v,
                                                    int64_t cap, int64_t n, int64_t row, int32_t* idx,
                                                    int64_t idx_cap, bf16* kt, int64_t nblk_cap, int blk) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.x, c = threadIdx.x;
  const bf16 kv = k_new[(size_t)pair * HD + c];
  const bf16 vv = v_new[(size_t)pair * HD + c];
  k[((size_t)pair * cap + row) * HD + c] = kv;
  v[((size_t)pair * cap + row) * HD + c] = vv;
  const int64_t jb = n / blk;
  bf16* pmax = kt + ((size_t)pair * 2 * HD + c) * nblk_cap + jb;
  bf16* pmin = kt + ((size_t)pair * 2 * HD + HD + c) * nblk_cap + jb;
  if (n % blk == 0) {
    *pmax = kv;
    *pmin = kv;
  } else {
    const float x = bf2f(kv);
    if (x > bf2f(*pmax)) *pmax = kv;
    if (x < bf2f(*pmin)) *pmin = kv;
  }
  if (idx && c == 0) idx[(size_t)pair * idx_cap + n] = (int32_t)row;
}

// Compaction with the KT cache built on the way: K_c[i] = K[keep[i]],
// V_c[i] = V[keep[i]] for i < B1, and per block of blk compacted rows the
// elementwise Kmax / Kmin of K_c (same values and order as kt_build_kernel).
// One CTA = 16 blocks of one pair; thread (chunk ch, block bl) copies the
// 16-byte chunk ch (8 channels) of every row of block bl and folds it into
// its maxima / minima, so no cross-thread reduction is needed; the KT tile is
// transposed in shared memory and written as 32-byte runs per channel row.
constexpr int CK_BLOCKS = 16;
constexpr int CK_NT = 256;

__global__ void __launch_bounds__(CK_NT) compact_kt_kernel(const bf16* k, const bf16* v, int64_t cap,
                                                           const int32_t* keep, int64_t keep_ld, int64_t B1, int blk,
                                                           bf16* ko, bf16* vo, int64_t out_cap, bf16* kt,
                                                           int64_t nblk_cap, const int32_t* bt, int64_t bt_stride,
                                                           int64_t num_pages, int Hkv) {
  __shared__ __align__(16) bf16 tile[2 * HD][CK_BLOCKS];   // row m*HD + c, column = block in the CTA
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  const int ch = threadIdx.x & 15, bl = threadIdx.x >> 4;
  const int64_t nblk = (B1 + blk - 1) / blk;
  const int64_t jb0 = (int64_t)blockIdx.x * CK_BLOCKS;
  const int64_t jb = jb0 + bl;
  float mx[8], mn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mx[e] = neg_inf();
    mn[e] = -neg_inf();
  }
  if (jb < nblk) {
    const int64_t t0 = jb * blk, t1 = min(B1, t0 + blk);
    const int32_t* kp = keep + (size_t)pair * keep_ld;
    const bf16* ks = k + (size_t)pair * cap * HD + ch * 8;
    const bf16* vs = v + (size_t)pair * cap * HD + ch * 8;
    // output rows: the pair's compacted cache, or (paged) the block's (page, head)
    // slab of blk rows, indexed from the block's first row t0
    size_t obase = (size_t)pair * out_cap * HD;
    int64_t rbase = 0;                       // compacted row of the first output row
    if (bt) {
      const int b = pair / Hkv, h = pair % Hkv;
      const int64_t pg = min(max((int64_t)bt[(size_t)b * bt_stride + jb], (int64_t)0), num_pages - 1);
      obase = (size_t)(pg * Hkv + h) * blk * HD;
      rbase = t0;
    }
    bf16* kd = ko + obase + ch * 8;
    bf16* vd = vo + obase + ch * 8;
    for (int64_t tb = t0; tb < t1; tb += 4) {
      uint4 kr[4], vr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {            // four rows in flight
        if (tb + u < t1) {
          const int64_t src = min(max((int64_t)kp[tb + u], (int64_t)0), cap - 1);
          kr[u] = *reinterpret_cast<const uint4*>(ks + src * HD);
          vr[u] = *reinterpret_cast<const uint4*>(vs + src * HD);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (tb + u < t1) {
          *reinterpret_cast<uint4*>(kd + (tb + u - rbase) * HD) = kr[u];
          *reinterpret_cast<uint4*>(vd + (tb + u - rbase) * HD) = vr[u];
          const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = bf16_lo(w[q]), hi = bf16_hi(w[q]);
            mx[2 * q] = fmaxf(mx[2 * q], lo);
            mn[2 * q] = fminf(mn[2 * q], lo);
            mx[2 * q + 1] = fmaxf(mx[2 * q + 1], hi);
            mn[2 * q + 1] = fminf(mn[2 * q + 1], hi);
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // the values are bf16 already: the conversion back is exact
    tile[ch * 8 + e][bl] = __float2bfloat16_rn(mx[e]);
    tile[HD + ch * 8 + e][bl] = __float2bfloat16_rn(mn[e]);
  }
  __syncthreads();
  const int row = threadIdx.x;                   // KT row m*HD + c
  const int nb = (int)min((int64_t)CK_BLOCKS, nblk - jb0);
  bf16* dst = kt + ((size_t)pair * 2 * HD + row) * nblk_cap + jb0;   // 16-byte aligned: nblk_cap % 8 == 0
  if (nb == CK_BLOCKS) {
    const uint4* srcp = reinterpret_cast<const uint4*>(&tile[row][0]);
    reinterpret_cast<uint4*>(dst)[0] = srcp[0];
    reinterpret_cast<uint4*>(dst)[1] = srcp[1];
  } else {
    for (int i = 0; i < nb; ++i) dst[i] = tile[row][i];
  }
}

// 8 bf16 (one 16-byte chunk) / scale -> 8 e4m3 codes (8 bytes); the codes'
// values are folded into mx / mn.
__device__ __forceinline__ uint2 quantize8(const uint4& r, float scale, float* mx, float* mn) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  uint16_t c[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    c[q] = e4m3x2_from_f32(__fdiv_rn(bf16_lo(w[q]), scale), __fdiv_rn(bf16_hi(w[q]), scale));
    if (mx) {
      const float2 v = e4m3x2_to_f32(c[q]);
      mx[2 * q] = fmaxf(mx[2 * q], v.x);
      mn[2 * q] = fminf(mn[2 * q], v.x);
      mx[2 * q + 1] = fmaxf(mx[2 * q + 1], v.y);
      mn[2 * q + 1] = fminf(mn[2 * q + 1], v.y);
    }
  }
  return make_uint2((uint32_t)c[0] | ((uint32_t)c[1] << 16), (uint32_t)c[2] | ((uint32_t)c[3] << 16));
}

// compact_kt_kernel storing e4m3 codes: K_c[i] = code(K[keep[i]] / k_scale),
// V_c[i] = code(V[keep[i]] / v_scale) (fp32 quotient, nearest even, saturated),
// and the KT cache as the max / min of the key codes' values, stored as codes
// (exact).  Rows are 128 bytes; the KT row stride nblk_cap is a multiple of 16.
__global__ void __launch_bounds__(CK_NT) compact_kt_fp8_kernel(const bf16* k, const bf16* v, int64_t cap,
                                                               const int32_t* keep, int64_t keep_ld, int64_t B1,
                                                               int blk, const float* ksc, const float* vsc,
                                                               uint8_t* ko, uint8_t* vo, int64_t out_cap, uint8_t* kt,
                                                               int64_t nblk_cap) {
  __shared__ __align__(16) uint8_t tile[2 * HD][CK_BLOCKS];
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.y;
  const int ch = threadIdx.x & 15, bl = threadIdx.x >> 4;
  const int64_t nblk = (B1 + blk - 1) / blk;
  const int64_t jb0 = (int64_t)blockIdx.x * CK_BLOCKS;
  const int64_t jb = jb0 + bl;
  const float sk = __ldg(ksc + pair), sv = __ldg(vsc + pair);
  float mx[8], mn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mx[e] = neg_inf();
    mn[e] = -neg_inf();
  }
  if (jb < nblk) {
    const int64_t t0 = jb * blk, t1 = min(B1, t0 + blk);
    const int32_t* kp = keep + (size_t)pair * keep_ld;
    const bf16* ks = k + (size_t)pair * cap * HD + ch * 8;
    const bf16* vs = v + (size_t)pair * cap * HD + ch * 8;
    uint8_t* kd = ko + (size_t)pair * out_cap * HD + ch * 8;
    uint8_t* vd = vo + (size_t)pair * out_cap * HD + ch * 8;
    for (int64_t tb = t0; tb < t1; tb += 4) {
      uint4 kr[4], vr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {            // four rows in flight
        if (tb + u < t1) {
          const int64_t src = min(max((int64_t)kp[tb + u], (int64_t)0), cap - 1);
          kr[u] = *reinterpret_cast<const uint4*>(ks + src * HD);
          vr[u] = *reinterpret_cast<const uint4*>(vs + src * HD);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (tb + u < t1) {
          *reinterpret_cast<uint2*>(kd + (tb + u) * HD) = quantize8(kr[u], sk, mx, mn);
          *reinterpret_cast<uint2*>(vd + (tb + u) * HD) = quantize8(vr[u], sv, nullptr, nullptr);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    // the bounds are code values already: re-encoding them is exact
    const uint16_t hx = e4m3x2_from_f32(mx[e], mx[e + 1]), hn = e4m3x2_from_f32(mn[e], mn[e + 1]);
    tile[ch * 8 + e][bl] = (uint8_t)(hx & 0xFF);
    tile[ch * 8 + e + 1][bl] = (uint8_t)(hx >> 8);
    tile[HD + ch * 8 + e][bl] = (uint8_t)(hn & 0xFF);
    tile[HD + ch * 8 + e + 1][bl] = (uint8_t)(hn >> 8);
  }
  __syncthreads();
  const int row = threadIdx.x;                   // KT row m*HD + c
  const int nb = (int)min((int64_t)CK_BLOCKS, nblk - jb0);
  uint8_t* dst = kt + ((size_t)pair * 2 * HD + row) * nblk_cap + jb0;   // 16-byte aligned: nblk_cap % 16 == 0
  if (nb == CK_BLOCKS) {
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&tile[row][0]);
  } else {
    for (int i = 0; i < nb; ++i) dst[i] = tile[row][i];
  }
}

}  // namespace

cudaError_t kt_build_launch(const void* k, int64_t cap, int64_t n, const int32_t* idx, int64_t idx_cap,
                            int32_t blk, void* kt, int64_t nblk_cap, int32_t pairs, cudaStream_t st,
                            const uint32_t* mask, int64_t mask_ld, int64_t n_prompt) {
  const int64_t nblk = (n + blk - 1) / blk;
  if (nblk == 0 || pairs == 0) return cudaSuccess;
  return launch_pdl(kt_build_kernel, dim3((unsigned)((nblk + KT_BLOCKS - 1) / KT_BLOCKS), pairs), dim3(KT_NT), 0, st,
                    reinterpret_cast<const bf16*>(k), cap, n, idx, idx_cap, (int)blk, reinterpret_cast<bf16*>(kt),
                    nblk_cap, mask, mask_ld, n_prompt);
}

namespace {

// One CTA per pair: clear the prompt's bits, then set the bit of every kept row.
__global__ void __launch_bounds__(256) keep_mask_kernel(const int32_t* keep, int64_t keep_ld, int64_t B1,
                                                        int64_t n_prompt, uint32_t* mask, int64_t mask_ld) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = blockIdx.x;
  uint32_t* m = mask + (size_t)pair * mask_ld;
  const int64_t words = (n_prompt + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += blockDim.x) m[w] = 0u;
  __syncthreads();
  const int32_t* kp = keep + (size_t)pair * keep_ld;
  for (int64_t i = threadIdx.x; i < B1; i += blockDim.x) {
    const int32_t r = kp[i];
    if (r >= 0 && r < n_prompt) atomicOr(m + (r >> 5), 1u << (r & 31));
  }
}

}  // namespace

cudaError_t keep_mask_launch(const int32_t* keep, int64_t keep_ld, int64_t B1, int64_t n_prompt, uint32_t* mask,
                             int64_t mask_ld, int32_t pairs, cudaStream_t st) {
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(keep_mask_kernel, dim3(pairs), dim3(256), 0, st, keep, keep_ld, B1, n_prompt, mask, mask_ld);
}

cudaError_t append_launch(const void* k_new, const void* v_new, void* k, void* v, int64_t cap, int64_t n,
                          int64_t row, int32_t* idx, int64_t idx_cap, void* kt, int64_t nblk_cap, int32_t blk,
                          int32_t pairs, cudaStream_t st) {
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(append_kernel, dim3(pairs), dim3(HD), 0, st, reinterpret_cast<const bf16*>(k_new),
                    reinterpret_cast<const bf16*>(v_new), reinterpret_cast<bf16*>(k), reinterpret_cast<bf16*>(v), cap, n,
                    row, idx, idx_cap, reinterpret_cast<bf16*>(kt), nblk_cap, (int)blk);
}

cudaError_t compact_kt_launch(const void* k, const void* v, int64_t cap, const int32_t* keep, int64_t keep_ld,
                              int64_t B1, int blk, void* ko, void* vo, int64_t out_cap, void* kt, int64_t nblk_cap,
                              int pairs, cudaStream_t st, const int32_t* bt, int64_t bt_stride, int64_t num_pages,
                              int Hkv) {
  const int64_t nblk = (B1 + blk - 1) / blk;
  return launch_pdl(compact_kt_kernel, dim3((unsigned)((nblk + CK_BLOCKS - 1) / CK_BLOCKS), pairs), dim3(CK_NT), 0, st,
                    reinterpret_cast<const bf16*>(k), reinterpret_cast<const bf16*>(v), cap, keep, keep_ld, B1, blk,
                    reinterpret_cast<bf16*>(ko), reinterpret_cast<bf16*>(vo), out_cap, reinterpret_cast<bf16*>(kt),
                    nblk_cap, bt, bt_stride, num_pages, Hkv);
}

cudaError_t compact_kt_fp8_launch(const void* k, const void* v, int64_t cap, const int32_t* keep, int64_t keep_ld,
                                  int64_t B1, int blk, const float* k_scale, const float* v_scale, void* ko, void* vo,
                                  int64_t out_cap, void* kt, int64_t nblk_cap, int pairs, cudaStream_t st) {
  const int64_t nblk = (B1 + blk - 1) / blk;
  return launch_pdl(compact_kt_fp8_kernel, dim3((unsigned)((nblk + CK_BLOCKS - 1) / CK_BLOCKS), pairs), dim3(CK_NT),
                    0, st, reinterpret_cast<const bf16*>(k), reinterpret_cast<const bf16*>(v), cap, keep, keep_ld, B1,
                    blk, k_scale, v_scale, reinterpret_cast<uint8_t*>(ko), reinterpret_cast<uint8_t*>(vo), out_cap,
                    reinterpret_cast<uint8_t*>(kt), nblk_cap);
}

}  // namespace rkv
