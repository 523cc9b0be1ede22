// score_common.cuh -- per-mode indexer score loops shared by the standalone
// score scan and the fused score+select kernel, so that both produce
// bit-identical scores.
//
// A row is split into 16-byte pieces held by consecutive lanes ("LPT" lanes
// per row); each lane reduces its piece, then the row's lanes combine their
// partial sums with xor-shuffles in a fixed order.
#pragma once

#include "common.cuh"

namespace skv {

constexpr int kScoreUnroll = 4;

// ---- int4 sketch x int8 query ---------------------------------------------------
// Codes are two's-complement nibbles; with u = code + 8 (flip bit 3 of each
// nibble) the product sum is dot(u, q8) - 8 * sum(q8), and u fits a signed
// byte, so __dp4a applies to the low and the high nibbles.
template <int LPT>
struct Int4Query {
  uint32_t q_even[4], q_odd[4];
  int corr;
  // Query codes of this lane's piece: dims [32p, 32p + 32) of the row; byte b
  // of the piece holds dims 2b (low nibble) and 2b+1 (high nibble).
  __device__ __forceinline__ void load(const int8_t* q8row, int p) {
    const uint4 qa = *reinterpret_cast<const uint4*>(q8row + 32 * p);
    const uint4 qc = *reinterpret_cast<const uint4*>(q8row + 32 * p + 16);
    const uint32_t qw[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
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
    corr = 8 * qsum;
  }
  // Score of the row whose piece this lane holds (all LPT lanes get it).
  __device__ __forceinline__ int32_t score(const uint4& v) const {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    int acc = 0;
#pragma unroll
    for (int w = 0; w < 4; w++) {
      const uint32_t x = w4[w] ^ 0x88888888u;
      acc = __dp4a(static_cast<int>(x & 0x0f0f0f0fu), static_cast<int>(q_even[w]), acc);
      acc = __dp4a(static_cast<int>((x >> 4) & 0x0f0f0f0fu), static_cast<int>(q_odd[w]), acc);
    }
#pragma unroll
    for (int o = 1; o < LPT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return static_cast<int32_t>(acc - corr);
  }
};

// ---- bf16 pooled keys (128 dims) x bf16 indexer query, fp32 accumulation ----------
struct PooledQuery {
  static constexpr int LPT = 16;
  float q[8];
  __device__ __forceinline__ void load(const uint16_t* qrow, int p) {
    const uint4 qv = *reinterpret_cast<const uint4*>(qrow + 8 * p);
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
      q[2 * e] = __uint_as_float(qw[e] << 16);
      q[2 * e + 1] = __uint_as_float(qw[e] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ float score(const uint4& v) const {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      acc = fmaf(q[2 * e], __uint_as_float(w4[e] << 16), acc);
      acc = fmaf(q[2 * e + 1], __uint_as_float(w4[e] & 0xffff0000u), acc);
    }
#pragma unroll
    for (int o = 1; o < LPT; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
  }
};

// ---- fp32 sketch x fp32 folded query: one warp per row ------------------------------
struct F32Query {
  float4 q[8];
  int n4;
  __device__ __forceinline__ void load(const float* qrow, int width, int lane) {
    n4 = width / 4;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int e = lane + 32 * i;
      q[i] = (e < n4) ? reinterpret_cast<const float4*>(qrow)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // row: the row's first float4 (global or shared memory).
  __device__ __forceinline__ float score(const float4* row, int lane) const {
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
    return acc;
  }
};

// Partial dot product of one 16-byte piece (no cross-lane reduction).
template <int LPT>
__device__ __forceinline__ int int4_piece(const Int4Query<LPT>& q, const uint4& v) {
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  int acc = 0;
#pragma unroll
  for (int w = 0; w < 4; w++) {
    const uint32_t x = w4[w] ^ 0x88888888u;
    acc = __dp4a(static_cast<int>(x & 0x0f0f0f0fu), static_cast<int>(q.q_even[w]), acc);
    acc = __dp4a(static_cast<int>((x >> 4) & 0x0f0f0f0fu), static_cast<int>(q.q_odd[w]), acc);
  }
  return acc;
}

// 128-byte sketch rows (8 lanes x 16 bytes), 32 rows per warp per iteration:
// lane (tg, p) loads piece p of rows base + 4u + tg for u = 0..7 (8 loads in
// flight), and a transposed butterfly over the 8 lanes of the row group (7
// shuffles for 8 rows) leaves lane (tg, p) with the full score of row
// base + 4p + tg.  The exact integer sums equal those of Int4Query::score.
template <typename Emit>
__device__ __forceinline__ void scan_int4_rows128(const int8_t* __restrict__ q8row, const uint8_t* __restrict__ rows,
                                                  int64_t t0, int64_t t1, int warp, int nwarps, Emit&& emit) {
  constexpr int LPT = 8, U = 8;
  const int lane = threadIdx.x & 31;
  const int p = lane & 7, tg = lane >> 3;
  Int4Query<LPT> q;
  q.load(q8row, p);
  const uint8_t* kb = rows + 16 * p;
  for (int64_t base = t0 + static_cast<int64_t>(warp) * 32; base < t1; base += static_cast<int64_t>(nwarps) * 32) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int64_t t = base + 4 * u + tg;
      v[u] = (t < t1) ? ld_stream16(kb + t * 128) : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    }
    int a[U];
#pragma unroll
    for (int u = 0; u < U; u++) a[u] = int4_piece(q, v[u]);
    // butterfly: keep the half named by the lane bit, send the other half
    const bool h4 = p & 4, h2 = p & 2, h1 = p & 1;
    int b4[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int keep = h4 ? a[j + 4] : a[j];
      const int send = h4 ? a[j] : a[j + 4];
      b4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    int b2[2];
#pragma unroll
    for (int j = 0; j < 2; j++) {
      const int keep = h2 ? b4[j + 2] : b4[j];
      const int send = h2 ? b4[j] : b4[j + 2];
      b2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const int keep = h1 ? b2[1] : b2[0];
    const int send = h1 ? b2[0] : b2[1];
    const int sum = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    const int64_t t = base + 4 * p + tg;  // the row whose score this lane now holds
    if (t < t1) emit(t, static_cast<int32_t>(sum - q.corr));
  }
}

// ---- loops over rows in global memory ------------------------------------------------
// Walk rows [t0, t1) of one request with all warps of the CTA; emit(t, score)
// is called once per row from the lane holding the row's first piece.  Loads
// are coalesced (consecutive lanes take consecutive 16-byte pieces of
// consecutive rows), several in flight per lane, without L1 allocation.

template <int LPT, typename Emit>
__device__ __forceinline__ void scan_int4(const int8_t* __restrict__ q8row, const uint8_t* __restrict__ rows,
                                          int64_t t0, int64_t t1, Emit&& emit) {
  constexpr int row_bytes = LPT * 16;
  constexpr int TPG = 32 / LPT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int p = lane % LPT, tg = lane / LPT;
  Int4Query<LPT> q;
  q.load(q8row, p);
  const uint8_t* kb = rows + 16 * p;
  const int64_t step = static_cast<int64_t>(TPG) * kScoreUnroll * nw;
  for (int64_t base = t0 + static_cast<int64_t>(warp) * TPG * kScoreUnroll; base < t1; base += step) {
    uint4 v[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; u++) {
      const int64_t t = base + u * TPG + tg;
      v[u] = (t < t1) ? ld_stream16(kb + t * row_bytes)
                      : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; u++) {
      const int32_t s = q.score(v[u]);
      const int64_t t = base + u * TPG + tg;
      if (p == 0 && t < t1) emit(t, s);
    }
  }
}

template <typename Emit>
__device__ __forceinline__ void scan_pooled(const uint16_t* __restrict__ qrow, const uint16_t* __restrict__ rows,
                                            int64_t t0, int64_t t1, Emit&& emit) {
  constexpr int LPT = 16, TPG = 2, width = 128;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int p = lane % LPT, tg = lane / LPT;
  PooledQuery q;
  q.load(qrow, p);
  const uint16_t* kb = rows + 8 * p;
  const int64_t step = static_cast<int64_t>(TPG) * kScoreUnroll * nw;
  for (int64_t base = t0 + static_cast<int64_t>(warp) * TPG * kScoreUnroll; base < t1; base += step) {
    uint4 v[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; u++) {
      const int64_t t = base + u * TPG + tg;
      v[u] = (t < t1) ? ld_stream16(kb + t * width) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; u++) {
      const float s = q.score(v[u]);
      const int64_t t = base + u * TPG + tg;
      if (p == 0 && t < t1) emit(t, s);
    }
  }
}

template <typename Emit>
__device__ __forceinline__ void scan_f32(const float* __restrict__ qrow, const float* __restrict__ rows, int width,
                                         int64_t t0, int64_t t1, Emit&& emit) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  F32Query q;
  q.load(qrow, width, lane);
  for (int64_t t = t0 + warp; t < t1; t += nw) {
    const float s = q.score(reinterpret_cast<const float4*>(rows + t * width), lane);
    if (lane == 0) emit(t, s);
  }
}

}  // namespace skv
