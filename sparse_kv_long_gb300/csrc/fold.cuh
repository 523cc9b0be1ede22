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

// One warp encodes a row of d (a multiple of 64, <= 512) dims held as in
// encode_row_warp (lane l: dims l + 32 i) as an int4 host row: per 64-dim
// group g (values i = 2g, 2g + 1 of every lane) scale = fp16(max|x| / 7),
// code = clamp(rint(x / scale), -8, 7) (zero or non-finite scale: code 0);
// bytes [0, d/2): dim 2j in the low nibble of byte j, 2j + 1 in the high
// nibble; then the d/64 fp16 scales.  dst must be 4-byte aligned.
__device__ __forceinline__ void encode_int4_row_warp(const float (&v)[16], int d, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int g = 0; g < 8; g++) {
    if (64 * g >= d) break;  // the same in every lane
    float m = fmaxf(fabsf(v[2 * g]), fabsf(v[2 * g + 1]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const __half sh = __float2half_rn(__fdiv_rn(m, 7.f));
    const float sf = __half2float(sh);
    const bool ok = (sf != 0.f) && isfinite(sf);
#pragma unroll
    for (int u = 0; u < 2; u++) {
      const int i = 2 * g + u;
      const uint32_t nib = static_cast<uint32_t>(ok ? rint_clamp(__fdiv_rn(v[i], sf), -8, 7) : 0) & 15u;
      // even lanes form the byte of dims (32 i + lane, + 1), lanes 8j the
      // word of dims [32 i + 8 j, + 8)
      const uint32_t byte = nib | (__shfl_down_sync(0xffffffffu, nib, 1) << 4);
      const uint32_t w = byte | (__shfl_down_sync(0xffffffffu, byte, 2) << 8) |
                         (__shfl_down_sync(0xffffffffu, byte, 4) << 16) |
                         (__shfl_down_sync(0xffffffffu, byte, 6) << 24);
      if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(dst + 16 * i + lane / 2) = w;
    }
    if (lane == 0) *reinterpret_cast<__half*>(dst + d / 2 + 2 * g) = sh;
  }
}

// Where the token a decode step appends goes, for request b.  Either explicit
// rows (`rows`: the int8 row, and the sketch row unless `sketch_rows` is
// given), or rows derived from the request's length T = lengths[b] (the
// appended token is T - 1): sketch (and int4 host) row b*n_cap + T - 1, int8
// row b*kv_stride + T - 1, or b*kv_stride + S + (T - 1) mod W when `ring` is
// set (HBM keeps S sinks and a ring of the last W tokens in front of the hot
// slots).  `host4`, when set, receives the token's int4 host row at
// host4 + (b*n_cap + T - 1) * Hkv*2*rb (head h: K at 2h*rb, V at (2h+1)*rb).
struct Append {
  const int64_t* rows;
  const int64_t* sketch_rows;
  const int32_t* lengths;
  int64_t n_cap, kv_stride;
  int S, W, ring;
  uint8_t* host4;
};

// False when the request has no token to append (length <= 0 or beyond the
// capacity): nothing is written for it.
__device__ __forceinline__ bool append_rows(const Append& a, int b, int64_t* kv_row, int64_t* sk_row) {
  if (a.rows) {
    *kv_row = a.rows[b];
    *sk_row = a.sketch_rows ? a.sketch_rows[b] : *kv_row;
    return true;
  }
  const int64_t T = a.lengths[b];
  if (T < 1 || T > a.n_cap) return false;
  *sk_row = static_cast<int64_t>(b) * a.n_cap + (T - 1);
  *kv_row = static_cast<int64_t>(b) * a.kv_stride + (a.ring ? a.S + (T - 1) % a.W : T - 1);
  return true;
}

// int8 code of a folded query coordinate with the request's scale sigma.
__device__ __forceinline__ int8_t query_code(float qp, float sigma) {
  return static_cast<int8_t>(sigma != 0.f ? rint_clamp(__fdiv_rn(qp, sigma), -127, 127) : 0);
}

}  // namespace fold
}  // namespace skv
