// sketch.cu -- key sketch (a1), folded query (a2) and int8 row encoding.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": every
// token is scored through a rank-64 key sketch stored int4, computed on a
// frozen basis; one pick per layer is shared by all KV heads.
#include "common.cuh"
#include "fold.cuh"

namespace skv {
namespace {

constexpr int kRank = 64;
constexpr int kProjThreads = 256;
constexpr int kMaxD = 512;

// One warp per (token, head): lane j computes sketch dims 2j and 2j+1.
__global__ __launch_bounds__(kProjThreads) void sketch_project_kernel(
    const uint16_t* __restrict__ keys, int64_t n_tok, int Hkv, int d,
    const float* __restrict__ basis, const float* __restrict__ c,
    const int64_t* __restrict__ out_rows, uint8_t* __restrict__ out4,
    float* __restrict__ out32) {
  extern __shared__ float smem[];
  float* P = smem;                                   // [d][64]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  float* krow = smem + d * kRank + warp * d;         // [d] per warp
  for (int i = threadIdx.x; i < d * kRank / 4; i += blockDim.x)
    reinterpret_cast<float4*>(P)[i] = reinterpret_cast<const float4*>(basis)[i];
  __syncthreads();
  const int j0 = 2 * lane;
  float c0 = 0.f, c1 = 0.f;
  const int64_t total = n_tok * Hkv;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * nw + warp; item < total;
       item += static_cast<int64_t>(gridDim.x) * nw) {
    const int64_t t = item / Hkv;
    const int h = static_cast<int>(item % Hkv);
    const uint16_t* k = keys + item * d;
    for (int x8 = lane; x8 < d / 8; x8 += 32) {
      uint4 v = *reinterpret_cast<const uint4*>(k + 8 * x8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        krow[8 * x8 + 2 * e] = __uint_as_float(w[e] << 16);
        krow[8 * x8 + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    }
    __syncwarp();
    float s0 = 0.f, s1 = 0.f;
    for (int x = 0; x < d; x++) {
      const float kx = krow[x];
      const float2 p = *reinterpret_cast<const float2*>(P + x * kRank + j0);
      s0 = fmaf(p.x, kx, s0);
      s1 = fmaf(p.y, kx, s1);
    }
    __syncwarp();
    const int64_t row = out_rows ? out_rows[t] : t;
    if (c) {
      c0 = c[h * kRank + j0];
      c1 = c[h * kRank + j0 + 1];
      const int q0 = (c0 != 0.f) ? rint_clamp(__fdiv_rn(s0, c0), -8, 7) : 0;
      const int q1 = (c1 != 0.f) ? rint_clamp(__fdiv_rn(s1, c1), -8, 7) : 0;
      out4[row * (Hkv * kRank / 2) + h * (kRank / 2) + lane] =
          static_cast<uint8_t>((q0 & 15) | ((q1 & 15) << 4));
    } else {
      *reinterpret_cast<float2*>(out32 + (row * Hkv + h) * kRank + j0) = make_float2(s0, s1);
    }
  }
}

constexpr int kQueryThreads = 256;

// One CTA per request.  The group's query heads are summed first (fp32, head
// order), then projected once per KV head: qp[h][j] = c[h][j] * sum_x
// basis[x][j] * Qsum_h[x] -- the same linear map as projecting each head and
// summing, with six times fewer multiply-adds for groups of six.  int8
// quantisation with one scale per request follows.
__global__ __launch_bounds__(kQueryThreads) void sketch_query_kernel(
    const uint16_t* __restrict__ q, int Hq, int Hkv, int d, const float* __restrict__ basis,
    const float* __restrict__ c, int8_t* __restrict__ q8, float* __restrict__ qf32,
    float* __restrict__ sigma_out) {
  extern __shared__ float smem[];
  float* qs = smem;                    // [Hkv][d] group sums
  float* qp = qs + Hkv * d;            // [Hkv][64]
  __shared__ float red[32];
  const int b = blockIdx.x;
  const int G = Hq / Hkv;
  const uint16_t* qb = q + static_cast<int64_t>(b) * Hq * d;
  for (int i = threadIdx.x; i < Hkv * d; i += blockDim.x) {
    const int h = i / d, x = i % d;
    float acc = 0.f;
    for (int gg = 0; gg < G; gg++) acc = __fadd_rn(acc, bf16_bits_to_f32(qb[(h * G + gg) * d + x]));
    qs[i] = acc;
  }
  __syncthreads();
  const int width = Hkv * kRank;
  float amax = 0.f;
  for (int m = threadIdx.x; m < width; m += blockDim.x) {
    const int h = m / kRank, j = m % kRank;
    const float* qh = qs + h * d;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int x = 0;
    for (; x + 3 < d; x += 4) {
      a0 = fmaf(__ldg(basis + x * kRank + j), qh[x], a0);
      a1 = fmaf(__ldg(basis + (x + 1) * kRank + j), qh[x + 1], a1);
      a2 = fmaf(__ldg(basis + (x + 2) * kRank + j), qh[x + 2], a2);
      a3 = fmaf(__ldg(basis + (x + 3) * kRank + j), qh[x + 3], a3);
    }
    for (; x < d; x++) a0 = fmaf(__ldg(basis + x * kRank + j), qh[x], a0);
    float acc = (a0 + a1) + (a2 + a3);
    if (c) acc = __fmul_rn(acc, c[m]);
    qp[m] = acc;
    amax = fmaxf(amax, fabsf(acc));
  }
  if (!c) {
    __syncthreads();
    for (int m = threadIdx.x; m < width; m += blockDim.x)
      qf32[static_cast<int64_t>(b) * width + m] = qp[m];
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float sigma = __fdiv_rn(red[0], 127.f);
  if (threadIdx.x == 0 && sigma_out) sigma_out[b] = sigma;
  for (int m = threadIdx.x; m < width; m += blockDim.x) {
    const int v = (sigma != 0.f) ? rint_clamp(__fdiv_rn(qp[m], sigma), -127, 127) : 0;
    q8[static_cast<int64_t>(b) * width + m] = static_cast<int8_t>(v);
  }
}

// One warp per (row, head).
__global__ __launch_bounds__(256) void quant_int8_kernel(const uint16_t* __restrict__ x,
                                                         int64_t n_items, int d,
                                                         const int64_t* __restrict__ out_rows,
                                                         int Hkv, int8_t* __restrict__ q,
                                                         __half* __restrict__ scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int chunks = d / 8;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * nw + warp; item < n_items;
       item += static_cast<int64_t>(gridDim.x) * nw) {
    const uint16_t* row = x + item * d;
    float amax = 0.f;
    for (int ch = lane; ch < chunks; ch += 32) {
      uint4 v = *reinterpret_cast<const uint4*>(row + 8 * ch);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[e] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[e] & 0xffff0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half sh = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float sf = __half2float(sh);
    const bool ok = (sf != 0.f) && isfinite(sf);
    const int64_t t = item / Hkv;
    const int h = static_cast<int>(item % Hkv);
    const int64_t orow = out_rows ? out_rows[t] : t;
    int8_t* qo = q + (orow * Hkv + h) * d;
    if (lane == 0) scale[orow * Hkv + h] = sh;
    for (int ch = lane; ch < chunks; ch += 32) {
      uint4 v = *reinterpret_cast<const uint4*>(row + 8 * ch);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
        const int a = ok ? rint_clamp(__fdiv_rn(lo, sf), -127, 127) : 0;
        const int bb = ok ? rint_clamp(__fdiv_rn(hi, sf), -127, 127) : 0;
        const uint32_t two = (static_cast<uint32_t>(a) & 0xffu) | ((static_cast<uint32_t>(bb) & 0xffu) << 8);
        packed[e >> 1] |= two << (16 * (e & 1));
      }
      *reinterpret_cast<uint2*>(qo + 8 * ch) = make_uint2(packed[0], packed[1]);
    }
  }
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT int skv_sketch_project(const uint16_t* keys, int64_t n_tok, int Hkv, int d, int r,
                                  const float* basis, const float* c, const int64_t* out_rows,
                                  void* out, void* stream) {
  if (n_tok < 0 || Hkv <= 0 || r != kRank || d <= 0 || d % 8 || d > kMaxD) return SKV_EINVAL;
  if (n_tok == 0) return SKV_OK;
  if (!keys || !basis || !out || !aligned16(keys) || !aligned16(basis)) return SKV_EINVAL;
  const size_t smem = (static_cast<size_t>(d) * kRank + (kProjThreads / 32) * d) * sizeof(float);
  if (cudaFuncSetAttribute(sketch_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SKV_ECUDA;
  const int64_t items = n_tok * Hkv;
  const int64_t want = (items + (kProjThreads / 32) - 1) / (kProjThreads / 32);
  const int grid = static_cast<int>(want < 4L * sm_count() ? want : 4L * sm_count());
  sketch_project_kernel<<<grid > 0 ? grid : 1, kProjThreads, smem, as_stream(stream)>>>(
      keys, n_tok, Hkv, d, basis, c, out_rows, static_cast<uint8_t*>(out), static_cast<float*>(out));
  return launch_status();
}

SKV_EXPORT int skv_sketch_query(const uint16_t* q, int B, int Hq, int Hkv, int d, int r,
                                const float* basis, const float* c, void* out, float* sigma_out,
                                void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || r != kRank || d <= 0 || d > kMaxD ||
      Hkv * kRank > 1024)
    return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (!q || !basis || !out || !aligned16(basis)) return SKV_EINVAL;
  const size_t smem = (static_cast<size_t>(Hkv) * d + Hkv * kRank) * sizeof(float);
  if (smem > 220 * 1024) return SKV_EUNSUPPORTED;
  if (cudaFuncSetAttribute(sketch_query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SKV_ECUDA;
  sketch_query_kernel<<<B, kQueryThreads, smem, as_stream(stream)>>>(
      q, Hq, Hkv, d, basis, c, static_cast<int8_t*>(out), static_cast<float*>(out), sigma_out);
  return launch_status();
}

SKV_EXPORT int skv_quantize_int8_rows(const uint16_t* x, int64_t n_rows, int Hkv, int d,
                                      const int64_t* out_rows, int8_t* q, uint16_t* scale,
                                      void* stream) {
  if (n_rows < 0 || Hkv <= 0 || d <= 0 || d % 8 || d > 1024) return SKV_EINVAL;
  if (n_rows == 0) return SKV_OK;
  if (!x || !q || !scale || !aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7)) return SKV_EINVAL;
  const int64_t items = n_rows * Hkv;
  const int64_t want = (items + 7) / 8;
  const int64_t cap = 16L * sm_count();
  const int grid = static_cast<int>(want < cap ? want : cap);
  quant_int8_kernel<<<grid > 0 ? grid : 1, 256, 0, as_stream(stream)>>>(
      x, items, d, out_rows, Hkv, q, reinterpret_cast<__half*>(scale));
  return launch_status();
}

// ---------------------------------------------------------------------------
// Fused per-layer decode preparation: append the current token (key sketch
// and int8 K/V rows) and fold the query, in one launch.
// ---------------------------------------------------------------------------
namespace skv {
namespace {

constexpr int kPrepThreads = 256;

// CTA (h, b): the sketch of the new key and the folded query of KV head h of
// request b share one pass over the basis (thread t: sketch dim t%64, basis
// rows [64*(t/64), +64)), then warps 0 and 1 encode the new K and V rows of
// head h.  The last CTA of request b (atomic ticket, no waiting) quantises the
// request's folded query with one scale.
__global__ __launch_bounds__(kPrepThreads) void prepare_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ newk, const uint16_t* __restrict__ newv, int Hq,
    int Hkv, int d, const float* __restrict__ basis, const float* __restrict__ c, const fold::Append ap,
    uint8_t* __restrict__ sketch, int8_t* __restrict__ k8,
    __half* __restrict__ ks, int8_t* __restrict__ v8, __half* __restrict__ vs, int8_t* __restrict__ q8,
    float* __restrict__ sigma_out, float* __restrict__ qp_ws, unsigned* __restrict__ tickets) {
  __shared__ float QK[2][kMaxD];                          // folded query, new key (head h)
  __shared__ float part[kMaxD / fold::kSlice][2][kRank];  // per slice: query, key
  __shared__ __align__(16) uint16_t kv_rows[2][kMaxD];    // the new K and V rows of head h
  __shared__ int last;
  __shared__ float red[32];
  const int h = blockIdx.x, b = blockIdx.y;
  const int G = Hq / Hkv;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint16_t* qb = q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(h) * G) * d;
  const uint16_t* kb = newk + (static_cast<int64_t>(b) * Hkv + h) * d;
  // Every load first, so that the first-touch latencies overlap.
  int64_t row = 0, sk_row = 0;
  const bool app = fold::append_rows(ap, b, &row, &sk_row);
  for (int u = t; u < 2 * (d / 8); u += blockDim.x) {
    const int which = u / (d / 8), piece = u - which * (d / 8);
    const uint16_t* src = (which == 0 ? newk : newv) + (static_cast<int64_t>(b) * Hkv + h) * d + 8 * piece;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(&kv_rows[which][8 * piece]))),
                 "l"(src)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  const int ns = fold::n_slices(d);
  constexpr int kTasks = 2;  // slice tasks per thread held in registers (d <= 256)
  float bcol[kTasks][fold::kSlice];
  const bool held = ns * kRank <= kTasks * kPrepThreads;
#pragma unroll
  for (int k = 0; k < kTasks; k++) {
    const int task = t + k * kPrepThreads;
    if (held && task < ns * kRank) fold::load_slice(basis, d, task % kRank, task / kRank, bcol[k]);
  }
  for (int x = t; x < d; x += blockDim.x) {
    QK[0][x] = fold::group_sum(qb, G, d, x);
    QK[1][x] = bf16_bits_to_f32(kb[x]);
  }
  __syncthreads();
  if (held) {
#pragma unroll
    for (int k = 0; k < kTasks; k++) {
      const int task = t + k * kPrepThreads;
      if (task < ns * kRank)
        fold::dot_slice(bcol[k], &QK[0][0], kMaxD, 2, d, task / kRank, &part[task / kRank][0][task % kRank], kRank);
    }
  } else {
    for (int task = t; task < ns * kRank; task += blockDim.x) {
      const int sl = task / kRank, j = task - sl * kRank;
      fold::proj_slice(basis, &QK[0][0], kMaxD, 2, d, j, sl, &part[sl][0][j], kRank);
    }
  }
  __syncthreads();
  if (t < kRank) {
    const float cj = c[h * kRank + t];
    qp_ws[static_cast<int64_t>(b) * Hkv * kRank + h * kRank + t] =
        __fmul_rn(fold::combine_slices(&part[0][0][t], 2 * kRank, ns), cj);
  }
  if (app && t < kRank / 2) {
    const int j0 = 2 * t;
    const int c0 = fold::sketch_code(fold::combine_slices(&part[0][1][j0], 2 * kRank, ns), c[h * kRank + j0]);
    const int c1 = fold::sketch_code(fold::combine_slices(&part[0][1][j0 + 1], 2 * kRank, ns), c[h * kRank + j0 + 1]);
    sketch[sk_row * (Hkv * kRank / 2) + h * (kRank / 2) + t] = static_cast<uint8_t>((c0 & 15) | ((c1 & 15) << 4));
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (app && warp < 2) {  // int8 rows of the new K (warp 0) and V (warp 1) of head h
    float rowv[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const int x = lane + 32 * i;
      rowv[i] = x < d ? bf16_bits_to_f32(kv_rows[warp][x]) : 0.f;
    }
    fold::encode_row_warp(rowv, d, (warp == 0 ? k8 : v8) + (row * Hkv + h) * d, (warp == 0 ? ks : vs) + row * Hkv + h);
    if (ap.host4) {
      const int64_t rb = d / 2 + d / 32;
      fold::encode_int4_row_warp(rowv, d, ap.host4 + (sk_row * Hkv * 2 + 2 * h + warp) * rb);
    }
  }
  // Folded query: the request's last CTA quantises all heads with one scale.
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(&tickets[b], 1u) == static_cast<unsigned>(Hkv - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int width = Hkv * kRank;
  const float* qpb = qp_ws + static_cast<int64_t>(b) * width;
  float amax = 0.f;
  for (int m = t; m < width; m += blockDim.x) amax = fmaxf(amax, fabsf(__ldcg(qpb + m)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (t < 32) {
    float v = t < (blockDim.x >> 5) ? red[t] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (t == 0) red[0] = v;
  }
  __syncthreads();
  const float sigma = __fdiv_rn(red[0], 127.f);
  if (t == 0) {
    if (sigma_out) sigma_out[b] = sigma;
    tickets[b] = 0u;
  }
  for (int m = t; m < width; m += blockDim.x) {
    q8[static_cast<int64_t>(b) * width + m] = fold::query_code(__ldcg(qpb + m), sigma);
  }
}

// One CTA per request, the same arithmetic as prepare_kernel: the group sums
// of every KV head and every appended key share one pass over the basis
// (each thread holds the basis slices it projects), so the request's scale
// and int8 query are formed in the same CTA -- no ticket, no round trip
// through global memory -- and the warps then encode the appended K and V
// rows.  Dynamic shared memory: X [2 Hkv][d] floats (group sums, then new
// keys), part [ns][2 Hkv][64] floats, qp [Hkv*64] floats, rows [2 Hkv][d] bf16.
size_t prepare_req_smem(int Hkv, int d) {
  const size_t nv = 2 * static_cast<size_t>(Hkv), ns = (static_cast<size_t>(d) + fold::kSlice - 1) / fold::kSlice;
  return nv * d * 4 + ns * nv * kRank * 4 + static_cast<size_t>(Hkv) * kRank * 4 + nv * d * 2;
}

constexpr int kReqThreads = 1024;

__global__ __launch_bounds__(kReqThreads, 1) void prepare_req_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ newk, const uint16_t* __restrict__ newv, int Hq,
    int Hkv, int d, const float* __restrict__ basis, const float* __restrict__ c, const fold::Append ap,
    uint8_t* __restrict__ sketch, int8_t* __restrict__ k8,
    __half* __restrict__ ks, int8_t* __restrict__ v8, __half* __restrict__ vs, int8_t* __restrict__ q8,
    float* __restrict__ sigma_out) {
  extern __shared__ __align__(16) float dsm[];
  __shared__ float red[32];
  const int b = blockIdx.x, G = Hq / Hkv, nv = 2 * Hkv, ns = fold::n_slices(d);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float* X = dsm;                                                  // [nv][d]
  float* part = X + nv * d;                                        // [ns][nv][64]
  float* qp = part + ns * nv * kRank;                              // [Hkv*64]
  uint16_t* rows = reinterpret_cast<uint16_t*>(qp + Hkv * kRank);  // [nv][d]: K rows, then V rows
  int64_t row = 0, sk_row = 0;
  // One warp encodes appended row r: int8 (K of head r, then V of head
  // r - Hkv), and with the host tier the token's int4 host row.
  auto encode_appended = [&](int r) {
    float rowv[16];
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const int x = lane + 32 * i;
      rowv[i] = x < d ? bf16_bits_to_f32(rows[r * d + x]) : 0.f;
    }
    const int h = r % Hkv;
    fold::encode_row_warp(rowv, d, (r < Hkv ? k8 : v8) + (row * Hkv + h) * d, (r < Hkv ? ks : vs) + row * Hkv + h);
    if (ap.host4) {  // the token's int4 host row: head h, K then V
      const int64_t rb = d / 2 + d / 32;
      fold::encode_int4_row_warp(rowv, d, ap.host4 + (sk_row * Hkv * 2 + 2 * h + (r < Hkv ? 0 : 1)) * rb);
    }
  };
  // Every load first, so that the first-touch latencies overlap.
  const bool app = fold::append_rows(ap, b, &row, &sk_row);
  // When there are enough warps, warp enc_w0 + r copies and later encodes
  // appended row r while the warps before it combine the folded query.
  const int enc_w0 = (Hkv * kRank + 31) / 32;
  const bool overlap = enc_w0 + nv <= static_cast<int>(blockDim.x >> 5);
  const bool encoder = overlap && warp >= enc_w0 && warp < enc_w0 + nv;
  const int u0 = overlap ? (encoder ? (warp - enc_w0) * (d / 8) + lane : nv * (d / 8)) : t;
  const int u1 = overlap ? (encoder ? (warp - enc_w0 + 1) * (d / 8) : 0) : nv * (d / 8);
  const int ustep = overlap ? 32 : static_cast<int>(blockDim.x);
  for (int u = u0; u < u1; u += ustep) {
    const int r = u / (d / 8), piece = u - r * (d / 8);
    const uint16_t* src = (r < Hkv ? newk : newv) + (static_cast<int64_t>(b) * Hkv + r % Hkv) * d + 8 * piece;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(rows + r * d + 8 * piece))),
                 "l"(src)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  // Thread t: basis column t % 64 of slice (t / 64) % ns, projected on the
  // group sums (first half of the threads) or on the new keys (second half).
  const int half = kReqThreads / 2;
  const bool held = ns * kRank <= half;
  const int task = t % half, vh = t / half;
  float bcol[fold::kSlice];
  if (held && task < ns * kRank) fold::load_slice(basis, d, task % kRank, task / kRank, bcol);
  for (int x = t; x < Hkv * d; x += blockDim.x) {
    const int h = x / d, xi = x - h * d;
    X[h * d + xi] = fold::group_sum(q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(h) * G) * d, G, d, xi);
    X[(Hkv + h) * d + xi] = bf16_bits_to_f32(newk[(static_cast<int64_t>(b) * Hkv + h) * d + xi]);
  }
  __syncthreads();
  if (held) {
    if (task < ns * kRank)
      fold::dot_slice(bcol, X + vh * Hkv * d, d, Hkv, d, task / kRank,
                      part + (task / kRank) * nv * kRank + vh * Hkv * kRank + task % kRank, kRank);
  } else {
    for (int task = t; task < ns * kRank; task += blockDim.x) {
      const int sl = task / kRank, j = task - sl * kRank;
      fold::proj_slice(basis, X, d, nv, d, j, sl, part + sl * nv * kRank + j, kRank);
    }
  }
  __syncthreads();
  float amax = 0.f;
  if (encoder) {  // int8 row r (K of head r, then V of head r - Hkv), beside the query's combination
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
    if (app) encode_appended(warp - enc_w0);
  }
  for (int m = t; m < Hkv * kRank; m += blockDim.x) {  // folded query of head m/64, dim m%64
    const float v = __fmul_rn(fold::combine_slices(part + m, nv * kRank, ns), c[m]);
    qp[m] = v;
    amax = fmaxf(amax, fabsf(v));
  }
  for (int m = t; app && m < Hkv * kRank / 2; m += blockDim.x) {  // sketch codes of the new keys, two per byte
    const int h = m / (kRank / 2), j0 = 2 * (m % (kRank / 2));
    const float* pk = part + (Hkv + h) * kRank;
    const int c0 = fold::sketch_code(fold::combine_slices(pk + j0, nv * kRank, ns), c[h * kRank + j0]);
    const int c1 = fold::sketch_code(fold::combine_slices(pk + j0 + 1, nv * kRank, ns), c[h * kRank + j0 + 1]);
    sketch[sk_row * (Hkv * kRank / 2) + m] = static_cast<uint8_t>((c0 & 15) | ((c1 & 15) << 4));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (t < 32) {
    float v = t < (blockDim.x >> 5) ? red[t] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (t == 0) red[0] = v;
  }
  for (int r = warp; !overlap && app && r < nv; r += blockDim.x >> 5) encode_appended(r);
  __syncthreads();
  const float sigma = __fdiv_rn(red[0], 127.f);
  if (t == 0 && sigma_out) sigma_out[b] = sigma;
  for (int m = t; m < Hkv * kRank; m += blockDim.x)
    q8[static_cast<int64_t>(b) * Hkv * kRank + m] = fold::query_code(qp[m], sigma);
}

}  // namespace
}  // namespace skv

SKV_EXPORT size_t skv_decode_prepare_workspace_size(int B, int Hkv, int r) {
  if (B <= 0 || Hkv <= 0 || r != kRank) return 0;
  return (static_cast<size_t>(B) * Hkv * kRank * sizeof(float) + 255) / 256 * 256 + (B * sizeof(unsigned) + 255) / 256 * 256;
}

namespace skv {

// Launches the per-step preparation (a1 + a2 + the int8 / int4 append) with
// the appended rows given by `ap`; used by skv_decode_prepare and by the
// chained layer step.
int launch_prepare(const uint16_t* q, const uint16_t* new_k, const uint16_t* new_v, int B, int Hq, int Hkv, int d,
                   const float* basis, const float* c, const fold::Append& ap, uint8_t* sketch, int8_t* k8,
                   uint16_t* k_scale, int8_t* v8, uint16_t* v_scale, int8_t* q8, float* sigma, void* workspace,
                   cudaStream_t st) {
  float* qp_ws = static_cast<float*>(workspace);
  unsigned* tickets = reinterpret_cast<unsigned*>(
      static_cast<char*>(workspace) + (static_cast<size_t>(B) * Hkv * kRank * sizeof(float) + 255) / 256 * 256);
  const size_t smem = prepare_req_smem(Hkv, d);
  if (smem <= 48 * 1024) {  // one CTA per request
    prepare_req_kernel<<<B, kReqThreads, smem, st>>>(q, new_k, new_v, Hq, Hkv, d, basis, c, ap, sketch, k8,
                                                     reinterpret_cast<__half*>(k_scale), v8,
                                                     reinterpret_cast<__half*>(v_scale), q8, sigma);
    return launch_status();
  }
  dim3 grid(Hkv, B);
  prepare_kernel<<<grid, kPrepThreads, 0, st>>>(q, new_k, new_v, Hq, Hkv, d, basis, c, ap, sketch, k8,
                                                reinterpret_cast<__half*>(k_scale), v8,
                                                reinterpret_cast<__half*>(v_scale), q8, sigma, qp_ws, tickets);
  return launch_status();
}

}  // namespace skv

SKV_EXPORT int skv_decode_prepare(const uint16_t* q, const uint16_t* new_k, const uint16_t* new_v, int B, int Hq,
                                  int Hkv, int d, int r, const float* basis, const float* c,
                                  const int64_t* new_rows, uint8_t* sketch, int8_t* k8, uint16_t* k_scale,
                                  int8_t* v8, uint16_t* v_scale, int8_t* q8, float* sigma, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || r != kRank || d <= 0 || d % 8 || d > kMaxD || Hkv > 65535)
    return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (!q || !new_k || !new_v || !basis || !c || !new_rows || !sketch || !k8 || !k_scale || !v8 || !v_scale || !q8 ||
      !workspace)
    return SKV_EINVAL;
  if (workspace_bytes < skv_decode_prepare_workspace_size(B, Hkv, r)) return SKV_ENOMEM;
  fold::Append ap{};
  ap.rows = new_rows;
  return launch_prepare(q, new_k, new_v, B, Hq, Hkv, d, basis, c, ap, sketch, k8, k_scale, v8, v_scale, q8, sigma,
                        workspace, as_stream(stream));
}
