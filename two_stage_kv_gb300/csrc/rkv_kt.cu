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
// as 128-byte runs along the block axis.
__global__ void __launch_bounds__(KT_NT) kt_build_kernel(const bf16* k, int64_t cap, int64_t n,
                                                         const int32_t* idx, int64_t idx_cap, int blk,
                                                         bf16* kt, int64_t nblk_cap) {
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
    for (int64_t t = t0; t < t1; ++t) {
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
      tmax[lane * 4 + i][jl] = __float2bfloat16_rn(mx[i]);
      tmin[lane * 4 + i][jl] = __float2bfloat16_rn(mn[i]);
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

}  // namespace

cudaError_t kt_build_launch(const void* k, int64_t cap, int64_t n, const int32_t* idx, int64_t idx_cap,
                            int32_t blk, void* kt, int64_t nblk_cap, int32_t pairs, cudaStream_t st) {
  const int64_t nblk = (n + blk - 1) / blk;
  if (nblk == 0 || pairs == 0) return cudaSuccess;
  return launch_pdl(kt_build_kernel, dim3((unsigned)((nblk + KT_BLOCKS - 1) / KT_BLOCKS), pairs), dim3(KT_NT), 0, st,
                    reinterpret_cast<const bf16*>(k), cap, n, idx, idx_cap, (int)blk, reinterpret_cast<bf16*>(kt),
                    nblk_cap);
}

cudaError_t append_launch(const void* k_new, const void* v_new, void* k, void* v, int64_t cap, int64_t n,
                          int64_t row, int32_t* idx, int64_t idx_cap, void* kt, int64_t nblk_cap, int32_t blk,
                          int32_t pairs, cudaStream_t st) {
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(append_kernel, dim3(pairs), dim3(HD), 0, st, reinterpret_cast<const bf16*>(k_new),
                    reinterpret_cast<const bf16*>(v_new), reinterpret_cast<bf16*>(k), reinterpret_cast<bf16*>(v), cap, n,
                    row, idx, idx_cap, reinterpret_cast<bf16*>(kt), nblk_cap, (int)blk);
}

}  // namespace rkv
