// fold.cuh -- the per-step preparation arithmetic (a1 for the appended key,
// a2 for the query, int8 encoding of the appended K/V rows), written once so
// that the standalone prepare kernel and the fused prepare + select kernel
// produce the same bits.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": keys are
// projected on a frozen rank-64 basis and stored as int4; one pick per layer
// is shared by the KV heads (read as the sum over heads and over the query
// heads of each group, folded into one int8 query with one scale).
#pragma once

#include "common.cuh"

namespace skv {
namespace fold {

constexpr int kRank = 64;

// Sum of the G query heads of a group at dim x, in head order (the loads of
// eight heads are issued together, the additions stay in order).
__device__ __forceinline__ float group_sum(const uint16_t* qg, int G, int d, int x) {
  float acc = 0.f;
  for (int g0 = 0; g0 < G; g0 += 8) {
    uint16_t v[8];
#pragma unroll
    for (int u = 0; u < 8; u++) v[u] = g0 + u < G ? __ldg(qg + (g0 + u) * d + x) : 0;
#pragma unroll
    for (int u = 0; u < 8; u++)
      if (g0 + u < G) acc = __fadd_rn(acc, bf16_bits_to_f32(v[u]));
  }
  return acc;
}

// Projection on basis column j of nv vectors X + v*xs (fp32, d values),
// restricted to the 32-dim slice `sl` (dims [32 sl, 32 sl + 32) of d): the
// thread loads its slice of the column once (all loads in flight together)
// and, per vector, runs two fused-multiply-add chains (even and odd dims)
// added at the end; result v goes to out[v * out_stride].  combine_slices
// adds the slices of one coordinate in slice order.
constexpr int kSlice = 32;

__device__ __forceinline__ int n_slices(int d) { return (d + kSlice - 1) / kSlice; }

// The thread's slice of basis column j (loads only).
__device__ __forceinline__ void load_slice(const float* __restrict__ basis, int d, int j, int sl,
                                           float (&bcol)[kSlice]) {
  const int x0 = sl * kSlice, n = min(d - x0, kSlice);
#pragma unroll
  for (int i = 0; i < kSlice; i++) bcol[i] = i < n ? __ldg(basis + (x0 + i) * kRank + j) : 0.f;
}

// The dot products of a loaded slice with nv vectors.
__device__ __forceinline__ void dot_slice(const float (&bcol)[kSlice], const float* X, int xs, int nv, int d, int sl,
                                          float* out, int out_stride) {
  const int x0 = sl * kSlice, n = min(d - x0, kSlice);
  for (int v = 0; v < nv; v++) {
    const float* xv = X + v * xs + x0;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < kSlice; i += 2) {
      if (i < n) a0 = fmaf(bcol[i], xv[i], a0);
      if (i + 1 < n) a1 = fmaf(bcol[i + 1], xv[i + 1], a1);
    }
    out[v * out_stride] = a0 + a1;
  }
}

__device__ __forceinline__ void proj_slice(const float* __restrict__ basis, const float* X, int xs, int nv, int d,
                                           int j, int sl, float* out, int out_stride) {
  float bcol[kSlice];
  load_slice(basis, d, j, sl, bcol);
  dot_slice(bcol, X, xs, nv, d, sl, out, out_stride);
}

__device__ __forceinline__ float combine_slices(const float* p, int stride, int ns) {
  float acc = p[0];
  for (int sl = 1; sl < ns; sl++) acc += p[sl * stride];
  return acc;
}

// int4 sketch code of a projected key coordinate (step c_j; zero step: 0).
__device__ __forceinline__ int sketch_code(float s, float cj) {
  return cj != 0.f ? rint_clamp(__fdiv_rn(s, cj), -8, 7) : 0;
}

// One warp encodes a bf16 row of d (<= 512) dims as int8 with one fp16
// scale: load_row_warp reads the row into registers (lane l holds dims
// l + 32 i), encode_row_warp quantises it.
__device__ __forceinline__ void load_row_warp(const uint16_t* src, int d, float (&v)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 16; i++) {
    const int x = lane + 32 * i;
    v[i] = x < d ? bf16_bits_to_f32(__ldg(src + x)) : 0.f;
  }
}

__device__ __forceinline__ void encode_row_warp(const float (&v)[16], int d, int8_t* dst, __half* scale) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const __half sh = __float2half_rn(__fdiv_rn(amax, 127.f));
  const float sf = __half2float(sh);
  const bool ok = (sf != 0.f) && isfinite(sf);
#pragma unroll
  for (int i = 0; i < 16; i++) {
    const int x = lane + 32 * i;
    if (x < d) dst[x] = static_cast<int8_t>(ok ? rint_clamp(__fdiv_rn(v[i], sf), -127, 127) : 0);
  }
  if (lane == 0) *scale = sh;
}

__device__ __forceinline__ void encode_int8_row_warp(const uint16_t* src, int d, int8_t* dst, __half* scale) {
  float v[16];
  load_row_warp(src, d, v);
  encode_row_warp(v, d, dst, scale);
}

// int8 code of a folded query coordinate with the request's scale sigma.
__device__ __forceinline__ int8_t query_code(float qp, float sigma) {
  return static_cast<int8_t>(sigma != 0.f ? rint_clamp(__fdiv_rn(qp, sigma), -127, 127) : 0);
}

}  // namespace fold
}  // namespace skv
