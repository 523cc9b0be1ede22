// score.cu -- indexer score scan (a3): the one read that grows with context.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": each decode
// step scores every token through the rank-64 sketch.  [P4] "3.14M Context on
// 3x 3090 ...", "What Needs to Stay in VRAM": the indexer scores all pooled
// blocks at every step; it is the only read proportional to the context.
//
// The scan is a coalesced streaming pass: consecutive lanes read consecutive
// 16-byte pieces of consecutive rows (a warp-wide 512-byte contiguous load),
// several loads in flight per lane, no L1 allocation.  One order key is
// written per candidate.
#include "common.cuh"

namespace skv {
namespace {

constexpr int kScanThreads = 256;
constexpr int kUnroll = 4;

// int4 sketch x int8 query.  A token row is width/2 bytes, covered by LPT lanes
// holding 16 bytes (32 codes) each.  Codes are two's-complement nibbles; with
// u = code + 8 (flip bit 3 of each nibble) the product sum is
// dot(u, q8) - 8 * sum(q8), and u fits a signed byte, so __dp4a applies.
template <int LPT>
__global__ __launch_bounds__(kScanThreads) void score_int4_kernel(
    const int8_t* __restrict__ q8, const uint8_t* __restrict__ keys, int64_t n_cap,
    const int32_t* __restrict__ lengths, int S, int W, int chunks,
    uint32_t* __restrict__ okeys, int32_t* __restrict__ raw, int32_t* status) {
  constexpr int width = LPT * 32;
  constexpr int row_bytes = width / 2;
  constexpr int TPG = 32 / LPT;  // tokens per warp-wide load
  const int b = blockIdx.y;
  int64_t T = lengths[b];
  if (T > n_cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    T = n_cap;
  }
  const int64_t lo = S, hi = T - W;
  if (hi <= lo) return;
  const int64_t n = hi - lo;
  const int64_t chunk = (n + chunks - 1) / chunks;
  const int64_t t0 = lo + blockIdx.x * chunk;
  const int64_t t1 = t0 + chunk < hi ? t0 + chunk : hi;
  if (t0 >= t1) return;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int p = lane % LPT;       // 16-byte piece of the row
  const int tg = lane / LPT;      // token within a warp-wide load
  // Query codes of this piece: dims [32p, 32p + 32).  Byte b of the piece
  // holds dims 2b (low nibble) and 2b+1 (high nibble).
  const int8_t* qb = q8 + static_cast<int64_t>(b) * width + 32 * p;
  const uint4 qa = *reinterpret_cast<const uint4*>(qb);
  const uint4 qc = *reinterpret_cast<const uint4*>(qb + 16);
  const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
  uint32_t q_even[4], q_odd[4];
  int qsum = 0;
#pragma unroll
  for (int w = 0; w < 4; w++) {
    q_even[w] = prmt(qw[2 * w], qw[2 * w + 1], 0x6420);
    q_odd[w] = prmt(qw[2 * w], qw[2 * w + 1], 0x7531);
    qsum = __dp4a(static_cast<int>(qw[2 * w]), 0x01010101, qsum);
    qsum = __dp4a(static_cast<int>(qw[2 * w + 1]), 0x01010101, qsum);
  }
#pragma unroll
  for (int o = 1; o < LPT; o <<= 1) qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
  const int corr = 8 * qsum;

  const uint8_t* kb = keys + static_cast<int64_t>(b) * n_cap * row_bytes + 16 * p;
  uint32_t* ok = okeys + static_cast<int64_t>(b) * n_cap;
  const int64_t step = static_cast<int64_t>(TPG) * kUnroll * nw;
  for (int64_t base = t0 + static_cast<int64_t>(warp) * TPG * kUnroll; base < t1; base += step) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t t = base + u * TPG + tg;
      v[u] = (t < t1) ? ld_stream16(kb + t * row_bytes) : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      int acc = 0;
#pragma unroll
      for (int w = 0; w < 4; w++) {
        const uint32_t x = w4[w] ^ 0x88888888u;
        acc = __dp4a(static_cast<int>(x & 0x0f0f0f0fu), static_cast<int>(q_even[w]), acc);
        acc = __dp4a(static_cast<int>((x >> 4) & 0x0f0f0f0fu), static_cast<int>(q_odd[w]), acc);
      }
#pragma unroll
      for (int o = 1; o < LPT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const int64_t t = base + u * TPG + tg;
      if (p == 0 && t < t1) {
        const int32_t s = acc - corr;
        ok[t] = order_key_i32(s);
        if (raw) raw[static_cast<int64_t>(b) * n_cap + t] = s;
      }
    }
  }
}

// fp32 sketch x fp32 folded query: one warp per token, lanes stride the row.
__global__ __launch_bounds__(kScanThreads) void score_f32_kernel(
    const float* __restrict__ qp, const float* __restrict__ keys, int64_t n_cap, int width,
    const int32_t* __restrict__ lengths, int S, int W, int chunks, uint32_t* __restrict__ okeys,
    float* __restrict__ raw, int32_t* status) {
  const int b = blockIdx.y;
  int64_t T = lengths[b];
  if (T > n_cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    T = n_cap;
  }
  const int64_t lo = S, hi = T - W;
  if (hi <= lo) return;
  const int64_t n = hi - lo, chunk = (n + chunks - 1) / chunks;
  const int64_t t0 = lo + blockIdx.x * chunk;
  const int64_t t1 = t0 + chunk < hi ? t0 + chunk : hi;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int n4 = width / 4;
  float4 q[8];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const int e = lane + 32 * i;
    q[i] = (e < n4) ? reinterpret_cast<const float4*>(qp + static_cast<int64_t>(b) * width)[e]
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t t = t0 + warp; t < t1; t += nw) {
    const float4* row = reinterpret_cast<const float4*>(keys + (static_cast<int64_t>(b) * n_cap + t) * width);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int e = lane + 32 * i;
      if (e < n4) {
        const float4 k = row[e];
        acc = fmaf(q[i].x, k.x, acc);
        acc = fmaf(q[i].y, k.y, acc);
        acc = fmaf(q[i].z, k.z, acc);
        acc = fmaf(q[i].w, k.w, acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (isnan(acc)) set_status(status, SKV_DEV_NAN);
      okeys[static_cast<int64_t>(b) * n_cap + t] = order_key_f32(acc);
      if (raw) raw[static_cast<int64_t>(b) * n_cap + t] = acc;
    }
  }
}

// bf16 pooled keys (128 dims = 256 bytes per block) x bf16 indexer query:
// 16 lanes per block, 8 dims per lane, fp32 accumulation.
__global__ __launch_bounds__(kScanThreads) void score_pooled_kernel(
    const uint16_t* __restrict__ qidx, const uint16_t* __restrict__ keys, int64_t n_cap,
    const int32_t* __restrict__ lengths, int ratio, int chunks, uint32_t* __restrict__ okeys,
    float* __restrict__ raw, int32_t* status) {
  constexpr int LPT = 16, TPG = 2, width = 128;
  const int b = blockIdx.y;
  int64_t T = lengths[b];
  if (T > n_cap * ratio) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    T = n_cap * ratio;
  }
  const int64_t hi = T / ratio;
  if (hi <= 0) return;
  const int64_t chunk = (hi + chunks - 1) / chunks;
  const int64_t t0 = blockIdx.x * chunk;
  const int64_t t1 = t0 + chunk < hi ? t0 + chunk : hi;
  if (t0 >= t1) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int p = lane % LPT, tg = lane / LPT;
  const uint4 qv = *reinterpret_cast<const uint4*>(qidx + static_cast<int64_t>(b) * width + 8 * p);
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
  float q[8];
#pragma unroll
  for (int e = 0; e < 4; e++) {
    q[2 * e] = __uint_as_float(qw[e] << 16);
    q[2 * e + 1] = __uint_as_float(qw[e] & 0xffff0000u);
  }
  const uint16_t* kb = keys + static_cast<int64_t>(b) * n_cap * width + 8 * p;
  const int64_t step = static_cast<int64_t>(TPG) * kUnroll * nw;
  for (int64_t base = t0 + static_cast<int64_t>(warp) * TPG * kUnroll; base < t1; base += step) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t t = base + u * TPG + tg;
      v[u] = (t < t1) ? ld_stream16(kb + t * width) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; e++) {
        acc = fmaf(q[2 * e], __uint_as_float(w4[e] << 16), acc);
        acc = fmaf(q[2 * e + 1], __uint_as_float(w4[e] & 0xffff0000u), acc);
      }
#pragma unroll
      for (int o = 1; o < LPT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const int64_t t = base + u * TPG + tg;
      if (p == 0 && t < t1) {
        if (isnan(acc)) set_status(status, SKV_DEV_NAN);
        okeys[static_cast<int64_t>(b) * n_cap + t] = order_key_f32(acc);
        if (raw) raw[static_cast<int64_t>(b) * n_cap + t] = acc;
      }
    }
  }
}

template <typename K>
int chunks_for(K kernel, int B) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanThreads, 0) != cudaSuccess ||
      per_sm <= 0)
    per_sm = 1;
  const int total = per_sm * sm_count();
  int c = (total + B - 1) / B;
  return c < 1 ? 1 : (c > 65535 ? 65535 : c);
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT int skv_index_score(int mode, int B, int width, const void* query, const void* keys,
                               int64_t n_cap, const int32_t* lengths, int ratio, int S, int W,
                               uint32_t* order_keys, void* raw_scores, int32_t* dev_status,
                               void* stream) {
  if (B < 0 || B > 65535 || n_cap < 0 || S < 0 || W < 0) return SKV_EINVAL;
  if (B == 0 || n_cap == 0) return SKV_OK;
  if (!query || !keys || !lengths || !order_keys) return SKV_EINVAL;
  if (!aligned16(keys) || !aligned16(query)) return SKV_EINVAL;
  cudaStream_t st = as_stream(stream);
  if (mode == SKV_SCORE_SKETCH_INT4) {
    if (ratio != 1) return SKV_EINVAL;
    if (width == 128) {
      auto k = score_int4_kernel<4>;
      dim3 grid(chunks_for(k, B), B);
      k<<<grid, kScanThreads, 0, st>>>(static_cast<const int8_t*>(query), static_cast<const uint8_t*>(keys),
                                       n_cap, lengths, S, W, grid.x, order_keys,
                                       static_cast<int32_t*>(raw_scores), dev_status);
    } else if (width == 256) {
      auto k = score_int4_kernel<8>;
      dim3 grid(chunks_for(k, B), B);
      k<<<grid, kScanThreads, 0, st>>>(static_cast<const int8_t*>(query), static_cast<const uint8_t*>(keys),
                                       n_cap, lengths, S, W, grid.x, order_keys,
                                       static_cast<int32_t*>(raw_scores), dev_status);
    } else if (width == 512) {
      auto k = score_int4_kernel<16>;
      dim3 grid(chunks_for(k, B), B);
      k<<<grid, kScanThreads, 0, st>>>(static_cast<const int8_t*>(query), static_cast<const uint8_t*>(keys),
                                       n_cap, lengths, S, W, grid.x, order_keys,
                                       static_cast<int32_t*>(raw_scores), dev_status);
    } else {
      return SKV_EUNSUPPORTED;
    }
  } else if (mode == SKV_SCORE_SKETCH_F32) {
    if (ratio != 1 || width <= 0 || width % 4 || width > 1024) return SKV_EINVAL;
    dim3 grid(chunks_for(score_f32_kernel, B), B);
    score_f32_kernel<<<grid, kScanThreads, 0, st>>>(
        static_cast<const float*>(query), static_cast<const float*>(keys), n_cap, width, lengths, S, W,
        grid.x, order_keys, static_cast<float*>(raw_scores), dev_status);
  } else if (mode == SKV_SCORE_POOLED_BF16) {
    if (ratio != 4 || width != 128 || S != 0 || W != 0) return SKV_EINVAL;
    dim3 grid(chunks_for(score_pooled_kernel, B), B);
    score_pooled_kernel<<<grid, kScanThreads, 0, st>>>(
        static_cast<const uint16_t*>(query), static_cast<const uint16_t*>(keys), n_cap, lengths, ratio,
        grid.x, order_keys, static_cast<float*>(raw_scores), dev_status);
  } else {
    return SKV_EINVAL;
  }
  return launch_status();
}
