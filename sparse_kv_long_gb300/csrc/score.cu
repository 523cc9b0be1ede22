// score.cu -- indexer score scan (a3): the one read that grows with context.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": each decode
// step scores every token through the rank-64 sketch.  [P4] "3.14M Context on
// 3x 3090 ...", "What Needs to Stay in VRAM": the indexer scores all pooled
// blocks at every step; it is the only read proportional to the context.
//
// One streaming pass over the candidate rows of every request (loops in
// score_common.cuh); one order key (and optionally the raw score) written per
// candidate.  The grid is one wave, split evenly across the requests.
#include "score_common.cuh"

namespace skv {
namespace {

constexpr int kScanThreads = 256;

// Candidate rows [lo, hi) of this CTA's request and chunk; false if none.
__device__ __forceinline__ bool scan_chunk(int64_t lo, int64_t hi, int chunks, int64_t* t0, int64_t* t1) {
  if (hi <= lo) return false;
  const int64_t n = hi - lo;
  const int64_t chunk = (n + chunks - 1) / chunks;
  *t0 = lo + blockIdx.x * chunk;
  *t1 = *t0 + chunk < hi ? *t0 + chunk : hi;
  return *t0 < *t1;
}

template <int LPT>
__global__ __launch_bounds__(kScanThreads) void score_int4_kernel(
    const int8_t* __restrict__ q8, const uint8_t* __restrict__ keys, int64_t n_cap,
    const int32_t* __restrict__ lengths, int S, int W, int chunks, uint32_t* __restrict__ okeys,
    int32_t* __restrict__ raw, int32_t* status) {
  constexpr int width = LPT * 32;
  const int b = blockIdx.y;
  int64_t T = lengths[b];
  if (T > n_cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    T = n_cap;
  }
  int64_t t0, t1;
  if (!scan_chunk(S, T - W, chunks, &t0, &t1)) return;
  uint32_t* ok = okeys + static_cast<int64_t>(b) * n_cap;
  int32_t* rw = raw ? raw + static_cast<int64_t>(b) * n_cap : nullptr;
  auto emit = [&](int64_t t, int32_t s) {
    ok[t] = order_key_i32(s);
    if (rw) rw[t] = s;
  };
  if (LPT == 8)
    scan_int4_rows128(q8 + static_cast<int64_t>(b) * width, keys + static_cast<int64_t>(b) * n_cap * (width / 2), t0,
                      t1, threadIdx.x >> 5, blockDim.x >> 5, emit);
  else
    scan_int4<LPT>(q8 + static_cast<int64_t>(b) * width, keys + static_cast<int64_t>(b) * n_cap * (width / 2), t0, t1,
                   emit);
}

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
  int64_t t0, t1;
  if (!scan_chunk(S, T - W, chunks, &t0, &t1)) return;
  uint32_t* ok = okeys + static_cast<int64_t>(b) * n_cap;
  float* rw = raw ? raw + static_cast<int64_t>(b) * n_cap : nullptr;
  scan_f32(qp + static_cast<int64_t>(b) * width, keys + static_cast<int64_t>(b) * n_cap * width, width, t0, t1,
           [&](int64_t t, float s) {
             if (isnan(s)) set_status(status, SKV_DEV_NAN);
             ok[t] = order_key_f32(s);
             if (rw) rw[t] = s;
           });
}

__global__ __launch_bounds__(kScanThreads) void score_pooled_kernel(
    const uint16_t* __restrict__ qidx, const uint16_t* __restrict__ keys, int64_t n_cap,
    const int32_t* __restrict__ lengths, int ratio, int chunks, uint32_t* __restrict__ okeys,
    float* __restrict__ raw, int32_t* status) {
  const int b = blockIdx.y;
  int64_t T = lengths[b];
  if (T > n_cap * ratio) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    T = n_cap * ratio;
  }
  int64_t t0, t1;
  if (!scan_chunk(0, T / ratio, chunks, &t0, &t1)) return;
  uint32_t* ok = okeys + static_cast<int64_t>(b) * n_cap;
  float* rw = raw ? raw + static_cast<int64_t>(b) * n_cap : nullptr;
  scan_pooled(qidx + static_cast<int64_t>(b) * 128, keys + static_cast<int64_t>(b) * n_cap * 128, t0, t1,
              [&](int64_t t, float s) {
                if (isnan(s)) set_status(status, SKV_DEV_NAN);
                ok[t] = order_key_f32(s);
                if (rw) rw[t] = s;
              });
}

template <typename K>
int chunks_for(K kernel, int B) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanThreads, 0) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    per_sm = 1;
  }
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
    const int8_t* q8 = static_cast<const int8_t*>(query);
    const uint8_t* kb = static_cast<const uint8_t*>(keys);
    int32_t* raw = static_cast<int32_t*>(raw_scores);
    if (width == 128) {
      dim3 grid(chunks_for(score_int4_kernel<4>, B), B);
      score_int4_kernel<4><<<grid, kScanThreads, 0, st>>>(q8, kb, n_cap, lengths, S, W, grid.x, order_keys, raw,
                                                          dev_status);
    } else if (width == 256) {
      dim3 grid(chunks_for(score_int4_kernel<8>, B), B);
      score_int4_kernel<8><<<grid, kScanThreads, 0, st>>>(q8, kb, n_cap, lengths, S, W, grid.x, order_keys, raw,
                                                          dev_status);
    } else if (width == 512) {
      dim3 grid(chunks_for(score_int4_kernel<16>, B), B);
      score_int4_kernel<16><<<grid, kScanThreads, 0, st>>>(q8, kb, n_cap, lengths, S, W, grid.x, order_keys, raw,
                                                           dev_status);
    } else {
      return SKV_EUNSUPPORTED;
    }
  } else if (mode == SKV_SCORE_SKETCH_F32) {
    if (ratio != 1 || width <= 0 || width % 4 || width > 1024) return SKV_EINVAL;
    dim3 grid(chunks_for(score_f32_kernel, B), B);
    score_f32_kernel<<<grid, kScanThreads, 0, st>>>(
        static_cast<const float*>(query), static_cast<const float*>(keys), n_cap, width, lengths, S, W, grid.x,
        order_keys, static_cast<float*>(raw_scores), dev_status);
  } else if (mode == SKV_SCORE_POOLED_BF16) {
    if (ratio < 1 || ratio > 64 || width != 128 || S != 0 || W != 0) return SKV_EINVAL;
    dim3 grid(chunks_for(score_pooled_kernel, B), B);
    score_pooled_kernel<<<grid, kScanThreads, 0, st>>>(
        static_cast<const uint16_t*>(query), static_cast<const uint16_t*>(keys), n_cap, lengths, ratio, grid.x,
        order_keys, static_cast<float*>(raw_scores), dev_status);
  } else {
    return SKV_EINVAL;
  }
  return launch_status();
}
