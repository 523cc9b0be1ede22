// pool.cu -- pooled indexer keys (a2').
//
// [P3] "You can offload most of Qwen3.8-Flash-Next's KV cache to RAM ...": the
// indexer runs over a pooled key, indexer_head_dim 128 compressed by ratio 4.
// [P4] "3.14M Context on 3x 3090 ...", "What Needs to Stay in VRAM": pooled
// keys (one per block) stay in HBM.  Reading: the pool is the fp32 mean of the
// block's tokens summed in token order, rounded to bf16.
#include "common.cuh"

namespace skv {
namespace {

// One thread per (block, 8 dims): four 16-byte loads, fp32 sums in token order,
// one 16-byte store.
__global__ __launch_bounds__(256) void pool_keys_kernel(const uint16_t* __restrict__ keys, int B,
                                                        int64_t t_cap, int D, int64_t first_block,
                                                        int64_t n_blocks, uint16_t* __restrict__ pooled) {
  const int lanes = D / 8;
  const int64_t per_req = n_blocks * lanes;
  const int64_t total = per_req * B;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < total;
       it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(it / per_req);
    const int64_t rem = it % per_req;
    const int64_t blk = first_block + rem / lanes;
    const int x8 = static_cast<int>(rem % lanes);
    const uint16_t* src = keys + (static_cast<int64_t>(b) * t_cap + 4 * blk) * D + 8 * x8;
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; u++) v[u] = *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(u) * D);
    uint32_t res[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
      float lo = 0.f, hi = 0.f;
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const uint32_t w = e == 0 ? v[u].x : e == 1 ? v[u].y : e == 2 ? v[u].z : v[u].w;
        lo = (u == 0) ? __uint_as_float(w << 16) : __fadd_rn(lo, __uint_as_float(w << 16));
        hi = (u == 0) ? __uint_as_float(w & 0xffff0000u) : __fadd_rn(hi, __uint_as_float(w & 0xffff0000u));
      }
      lo = __fmul_rn(lo, 0.25f);
      hi = __fmul_rn(hi, 0.25f);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
      res[e] = *reinterpret_cast<uint32_t*>(&h2);
    }
    uint16_t* dst = pooled + (static_cast<int64_t>(b) * (t_cap / 4) + blk) * D + 8 * x8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(res[0], res[1], res[2], res[3]);
  }
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT int skv_pool_keys(const uint16_t* keys, int B, int64_t t_cap, int D, int ratio,
                             int64_t first_block, int64_t n_blocks, uint16_t* pooled, void* stream) {
  if (B < 0 || t_cap < 0 || D <= 0 || D % 8 || ratio != 4 || first_block < 0 || n_blocks < 0)
    return SKV_EINVAL;
  if (4 * (first_block + n_blocks) > t_cap) return SKV_EINVAL;
  if (B == 0 || n_blocks == 0) return SKV_OK;
  if (!keys || !pooled || !aligned16(keys) || !aligned16(pooled)) return SKV_EINVAL;
  const int64_t total = static_cast<int64_t>(B) * n_blocks * (D / 8);
  const int64_t want = (total + 255) / 256;
  const int64_t cap = 8L * sm_count();
  const int grid = static_cast<int>(want < cap ? want : cap);
  pool_keys_kernel<<<grid > 0 ? grid : 1, 256, 0, as_stream(stream)>>>(keys, B, t_cap, D, first_block,
                                                                      n_blocks, pooled);
  return launch_status();
}
