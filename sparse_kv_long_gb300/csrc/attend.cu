// attend.cu -- exact attention over the selected rows (a6), split-K decode.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": exact int8
// attention on the top 2048 tokens, 64 sinks and the last 1024.  [P4] "3.14M
// Context on 3x 3090 ...", "No Need to Rewrite the Kernel": a row is found by
// adding (token*n_kv_heads + kv_head)*head_dim to the base, so the pool may be
// HBM or host memory mapped for the GPU.
//
// Design.  A CTA owns one (request, KV head, group of up to 8 query heads,
// split of the selected rows); its 4 warps take 16-row tiles in turn.  Per
// tile a warp computes S = Q K^T with m16n8k16 tensor-core MMAs (the query
// heads are the M rows, padded to 16; two n8 tiles cover the 16 rows), runs
// the online softmax on the accumulator registers, and accumulates O^T += V^T
// P^T with the probabilities reused straight from the S accumulators as the B
// operand.  The head dimension is permuted consistently on Q and K so that
// each lane loads contiguous 16-byte pieces of a row; the V dimension is
// permuted so that a lane loads 32 contiguous dims of 4 rows.  int8 codes are
// converted to fp16 exactly (magic-number trick), and the per-row scales are
// applied in fp32: the K scale to the logits, the V scale folded into P.
// bf16 rows keep bf16 operands, with P split into two bf16 terms.
// Partials (m, l, O) of the 4 warps are merged in shared memory, each CTA
// writes one partial, and the last CTA of a (request, head group) merges all
// splits in split order (deterministic) and writes the output.
#include "common.cuh"

namespace skv {
namespace {

constexpr int D = 256;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kPart = 16 + 8 * D;  // m[8], l[8], O[8][D] floats per partial

struct AttendArgs {
  const uint16_t* q;
  const uint8_t* kpool;
  const uint8_t* vpool;
  const uint16_t* kscale;
  const uint16_t* vscale;
  int64_t req_row_stride;
  int64_t n_pool_rows;
  const int32_t* rows;
  int max_rows;
  const int32_t* count;
  int B, Hq, Hkv, G, hgroups, nsplit, rows_per_split;
  float scale_log2;
  float* part;
  unsigned* tickets;
  float* out;
  int32_t* status;
};

__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two int8 codes held as offset-binary bytes (code + 128) in bytes sel of u,
// to an exact fp16 pair: 0x64xx is 1024 + xx, minus 1152 = 1024 + 128.
__device__ __forceinline__ uint32_t u8pair_to_h2(uint32_t u, uint32_t sel) {
  const uint32_t m = prmt(u, 0x64646464u, sel);
  uint32_t r;
  asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(0x64806480u));
  return r;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float exp2_fast(float x) { return exp2f(x); }

template <int KV>
__global__ __launch_bounds__(kThreads) void attend_kernel(AttendArgs a) {
  constexpr int ES = KV == SKV_KV_INT8 ? 1 : 2;  // bytes per element
  __shared__ float sm_m[kWarps][8], sm_l[kWarps][8];
  __shared__ float sm_o[kWarps][8][D];
  __shared__ float fin_m[8], fin_l[8];
  __shared__ int is_last;

  const int b = blockIdx.z, hy = blockIdx.y, split = blockIdx.x;
  const int h = hy / a.hgroups, hg = hy % a.hgroups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int head_local = hg * 8 + g;
  const bool head_ok = head_local < a.G;
  const int qh = h * a.G + head_local;

  int n = a.count[b];
  n = n < 0 ? 0 : (n > a.max_rows ? a.max_rows : n);
  const int r0 = split * a.rows_per_split;
  const int r1 = r0 + a.rows_per_split < n ? r0 + a.rows_per_split : n;

  // ---- query fragments (A operand of S = Q K^T), permuted head dim ----------
  uint32_t qa[16][2];
  {
    const uint16_t* qrow = a.q + (static_cast<int64_t>(b) * a.Hq + (head_ok ? qh : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < 16; ks++) {
      const int base = KV == SKV_KV_INT8 ? 16 * (c + 4 * (ks >> 2)) + 4 * (ks & 3)
                                         : 8 * (c + 4 * (ks >> 1)) + 4 * (ks & 1);
      uint2 v = head_ok ? *reinterpret_cast<const uint2*>(qrow + base) : make_uint2(0u, 0u);
      if (KV == SKV_KV_INT8) {
        qa[ks][0] = pack_h2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
        qa[ks][1] = pack_h2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
      } else {
        qa[ks][0] = v.x;
        qa[ks][1] = v.y;
      }
    }
  }

  float o[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; mt++) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run = -INFINITY, l_part = 0.f;

  const int64_t pitch = static_cast<int64_t>(a.Hkv) * D * ES;  // bytes per pool row
  const uint8_t* kbase = a.kpool + static_cast<int64_t>(h) * D * ES;
  const uint8_t* vbase = a.vpool + static_cast<int64_t>(h) * D * ES;
  const int32_t* rows = a.rows + static_cast<int64_t>(b) * a.max_rows;

  for (int tile = r0 + warp * 16; tile < r1; tile += 16 * kWarps) {
    // Physical row of tile row `lane` (lanes 0..15), -1 when absent.
    int64_t prow = -1;
    if (lane < 16 && tile + lane < r1) {
      const int32_t rid = rows[tile + lane];
      const int64_t p = static_cast<int64_t>(b) * a.req_row_stride + rid;
      if (rid >= 0 && p >= 0 && p < a.n_pool_rows) {
        prow = p;
      } else {
        set_status(a.status, SKV_DEV_RANGE);
      }
    }
    const int64_t pk0 = __shfl_sync(0xffffffffu, prow, g);
    const int64_t pk1 = __shfl_sync(0xffffffffu, prow, g + 8);
    int64_t pv[4];
    pv[0] = __shfl_sync(0xffffffffu, prow, 2 * c);
    pv[1] = __shfl_sync(0xffffffffu, prow, 2 * c + 1);
    pv[2] = __shfl_sync(0xffffffffu, prow, 2 * c + 8);
    pv[3] = __shfl_sync(0xffffffffu, prow, 2 * c + 9);

    // ---- S = Q K^T ----------------------------------------------------------
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    if (KV == SKV_KV_INT8) {
      uint4 k0[4], k1[4];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        k0[i] = pk0 >= 0 ? ld_nc16(kbase + pk0 * pitch + 16 * (c + 4 * i)) : make_uint4(0u, 0u, 0u, 0u);
        k1[i] = pk1 >= 0 ? ld_nc16(kbase + pk1 * pitch + 16 * (c + 4 * i)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 16; ks++) {
        const int i = ks >> 2, wsel = ks & 3;
        const uint32_t w0 = (wsel == 0 ? k0[i].x : wsel == 1 ? k0[i].y : wsel == 2 ? k0[i].z : k0[i].w) ^ 0x80808080u;
        const uint32_t w1 = (wsel == 0 ? k1[i].x : wsel == 1 ? k1[i].y : wsel == 2 ? k1[i].z : k1[i].w) ^ 0x80808080u;
        mma_f16(s0, qa[ks][0], 0u, qa[ks][1], 0u, u8pair_to_h2(w0, 0x4140), u8pair_to_h2(w0, 0x4342));
        mma_f16(s1, qa[ks][0], 0u, qa[ks][1], 0u, u8pair_to_h2(w1, 0x4140), u8pair_to_h2(w1, 0x4342));
      }
    } else {
      uint4 k0[8], k1[8];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        k0[i] = pk0 >= 0 ? ld_nc16(kbase + pk0 * pitch + 16 * (c + 4 * i)) : make_uint4(0u, 0u, 0u, 0u);
        k1[i] = pk1 >= 0 ? ld_nc16(kbase + pk1 * pitch + 16 * (c + 4 * i)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int ks = 0; ks < 16; ks++) {
        const int i = ks >> 1;
        const uint32_t b0a = (ks & 1) ? k0[i].z : k0[i].x, b1a = (ks & 1) ? k0[i].w : k0[i].y;
        const uint32_t b0b = (ks & 1) ? k1[i].z : k1[i].x, b1b = (ks & 1) ? k1[i].w : k1[i].y;
        mma_bf16(s0, qa[ks][0], 0u, qa[ks][1], 0u, b0a, b1a);
        mma_bf16(s1, qa[ks][0], 0u, qa[ks][1], 0u, b0b, b1b);
      }
    }

    // ---- online softmax on S[head g][rows 2c, 2c+1, 2c+8, 2c+9] -------------
    float x[4] = {s0[0], s0[1], s1[0], s1[1]};
    float vsc[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      if (pv[i] >= 0) {
        float f = a.scale_log2;
        vsc[i] = 1.f;
        if (KV == SKV_KV_INT8) {
          f *= __half2float(__ushort_as_half(a.kscale[pv[i] * a.Hkv + h]));
          vsc[i] = __half2float(__ushort_as_half(a.vscale[pv[i] * a.Hkv + h]));
        }
        x[i] *= f;
      } else {
        x[i] = -INFINITY;
        vsc[i] = 0.f;
      }
    }
    float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m_run, tmax);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2_fast(m_run - m_use);
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; i++) p[i] = exp2_fast(x[i] - m_use);
    l_part = l_part * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
    m_run = m_new;
    const float a_e = __shfl_sync(0xffffffffu, alpha, 8 * c);
    const float a_o = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
    for (int mt = 0; mt < 16; mt++) {
      o[mt][0] *= a_e;
      o[mt][1] *= a_o;
      o[mt][2] *= a_e;
      o[mt][3] *= a_o;
    }

    // ---- O^T += V^T P^T -----------------------------------------------------
    if (KV == SKV_KV_INT8) {
      const uint32_t bp0 = pack_h2(p[0] * vsc[0], p[1] * vsc[1]);
      const uint32_t bp1 = pack_h2(p[2] * vsc[2], p[3] * vsc[3]);
      uint4 v[4][2];
#pragma unroll
      for (int r = 0; r < 4; r++) {
#pragma unroll
        for (int hh = 0; hh < 2; hh++)
          v[r][hh] = pv[r] >= 0 ? ld_nc16(vbase + pv[r] * pitch + 32 * g + 16 * hh)
                                : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int qq = 0; qq < 8; qq++) {
        const int hh = qq >> 2, ws = qq & 3;
        uint32_t w[4];
#pragma unroll
        for (int r = 0; r < 4; r++)
          w[r] = ws == 0 ? v[r][hh].x : ws == 1 ? v[r][hh].y : ws == 2 ? v[r][hh].z : v[r][hh].w;
        const uint32_t t01 = prmt(w[0], w[1], 0x5140) ^ 0x80808080u;  // rows 2c,2c+1: dims 4qq, 4qq+1
        const uint32_t t23 = prmt(w[0], w[1], 0x7362) ^ 0x80808080u;  // dims 4qq+2, 4qq+3
        const uint32_t u01 = prmt(w[2], w[3], 0x5140) ^ 0x80808080u;  // rows 2c+8, 2c+9
        const uint32_t u23 = prmt(w[2], w[3], 0x7362) ^ 0x80808080u;
        mma_f16(o[2 * qq], u8pair_to_h2(t01, 0x4140), u8pair_to_h2(t01, 0x4342), u8pair_to_h2(u01, 0x4140),
                u8pair_to_h2(u01, 0x4342), bp0, bp1);
        mma_f16(o[2 * qq + 1], u8pair_to_h2(t23, 0x4140), u8pair_to_h2(t23, 0x4342),
                u8pair_to_h2(u23, 0x4140), u8pair_to_h2(u23, 0x4342), bp0, bp1);
      }
    } else {
      const uint32_t ph0 = pack_bf2(p[0], p[1]), ph1 = pack_bf2(p[2], p[3]);
      const float r0f = p[0] - __uint_as_float(ph0 << 16), r1f = p[1] - __uint_as_float(ph0 & 0xffff0000u);
      const float r2f = p[2] - __uint_as_float(ph1 << 16), r3f = p[3] - __uint_as_float(ph1 & 0xffff0000u);
      const uint32_t pl0 = pack_bf2(r0f, r1f), pl1 = pack_bf2(r2f, r3f);
#pragma unroll
      for (int hh = 0; hh < 4; hh++) {  // 16-byte piece hh: dims 32g + 8hh .. +7
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; r++)
          v[r] = pv[r] >= 0 ? ld_nc16(vbase + pv[r] * pitch + 64 * g + 16 * hh) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int ws = 0; ws < 4; ws++) {
          const int mt = 4 * hh + ws;  // dims 32g + 2mt, 32g + 2mt + 1
          uint32_t w[4];
#pragma unroll
          for (int r = 0; r < 4; r++) w[r] = ws == 0 ? v[r].x : ws == 1 ? v[r].y : ws == 2 ? v[r].z : v[r].w;
          const uint32_t a0 = prmt(w[0], w[1], 0x5410), a1 = prmt(w[0], w[1], 0x7632);
          const uint32_t a2 = prmt(w[2], w[3], 0x5410), a3 = prmt(w[2], w[3], 0x7632);
          mma_bf16(o[mt], a0, a1, a2, a3, ph0, ph1);
          mma_bf16(o[mt], a0, a1, a2, a3, pl0, pl1);
        }
      }
    }
  }

  // ---- merge the 4 warps ---------------------------------------------------
  float l_grp = l_part;
  l_grp += __shfl_xor_sync(0xffffffffu, l_grp, 1);
  l_grp += __shfl_xor_sync(0xffffffffu, l_grp, 2);
  if (c == 0) {
    sm_m[warp][g] = m_run;
    sm_l[warp][g] = l_grp;
  }
#pragma unroll
  for (int mt = 0; mt < 16; mt++) {
    const int d0 = 32 * g + 2 * mt;
    sm_o[warp][2 * c][d0] = o[mt][0];
    sm_o[warp][2 * c + 1][d0] = o[mt][1];
    sm_o[warp][2 * c][d0 + 1] = o[mt][2];
    sm_o[warp][2 * c + 1][d0 + 1] = o[mt][3];
  }
  __syncthreads();
  const int gy = gridDim.y;
  float* mypart = a.part + ((static_cast<int64_t>(b) * gy + hy) * a.nsplit + split) * kPart;
  if (threadIdx.x < 8) {
    const int hd = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; w++) M = fmaxf(M, sm_m[w][hd]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kWarps; w++) L += exp2_fast(sm_m[w][hd] - M) * sm_l[w][hd];
    fin_m[hd] = M;
    mypart[hd] = M;
    mypart[8 + hd] = L;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 8 * D; e += blockDim.x) {
    const int hd = e / D, dd = e % D;
    const float M = fin_m[hd];
    float acc = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kWarps; w++) acc += exp2_fast(sm_m[w][hd] - M) * sm_o[w][hd][dd];
    mypart[16 + e] = acc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    is_last = atomicAdd(&a.tickets[b * gy + hy], 1u) == static_cast<unsigned>(a.nsplit - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- last CTA: merge the splits in split order ----------------------------
  const float* parts = a.part + (static_cast<int64_t>(b) * gy + hy) * a.nsplit * kPart;
  if (threadIdx.x < 8) {
    const int hd = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; s++) M = fmaxf(M, __ldcg(parts + s * kPart + hd));
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < a.nsplit; s++)
        L += exp2_fast(__ldcg(parts + s * kPart + hd) - M) * __ldcg(parts + s * kPart + 8 + hd);
    fin_m[hd] = M;
    fin_l[hd] = L;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 8 * D; e += blockDim.x) {
    const int hd = e / D, dd = e % D;
    const int hl = hg * 8 + hd;
    if (hl >= a.G) continue;
    const float M = fin_m[hd], L = fin_l[hd];
    float acc = 0.f;
    if (M != -INFINITY && L > 0.f) {
      for (int s = 0; s < a.nsplit; s++)
        acc += exp2_fast(__ldcg(parts + s * kPart + hd) - M) * __ldcg(parts + s * kPart + 16 + e);
      acc = acc / L;
    }
    a.out[(static_cast<int64_t>(b) * a.Hq + h * a.G + hl) * D + dd] = acc;
  }
  if (threadIdx.x == 0) a.tickets[b * gy + hy] = 0;
}

struct Plan {
  int hgroups, gy, nsplit, rows_per_split;
  size_t part_bytes, ticket_bytes;
};

Plan make_plan(int B, int Hq, int Hkv, int max_rows) {
  Plan p;
  const int G = Hq / Hkv;
  p.hgroups = (G + 7) / 8;
  p.gy = Hkv * p.hgroups;
  const int pairs = B * p.gy;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<SKV_KV_INT8>, kThreads, 0) !=
          cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int target = per_sm * (sm_count() > 0 ? sm_count() : 1);
  int ns = target / pairs;  // at most one wave
  const int max_ns = (max_rows + 63) / 64;
  ns = ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  if (ns < 1) ns = 1;
  int rps = (max_rows + ns - 1) / ns;
  rps = (rps + 15) / 16 * 16;
  ns = (max_rows + rps - 1) / rps;
  if (ns < 1) ns = 1;
  p.nsplit = ns;
  p.rows_per_split = rps;
  p.part_bytes = static_cast<size_t>(B) * p.gy * ns * kPart * sizeof(float);
  p.ticket_bytes = (static_cast<size_t>(B) * p.gy * sizeof(unsigned) + 255) / 256 * 256;
  return p;
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_attend_workspace_size(int B, int Hq, int Hkv, int d, int max_rows) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d != D || max_rows < 1) return 0;
  Plan p = make_plan(B, Hq, Hkv, max_rows);
  return p.ticket_bytes + p.part_bytes;
}

SKV_EXPORT int skv_sparse_attend_decode(int kv_kind, int B, int Hq, int Hkv, int d, const uint16_t* q,
                                        const void* k_pool, const void* v_pool, const uint16_t* k_scale,
                                        const uint16_t* v_scale, int64_t req_row_stride,
                                        int64_t n_pool_rows, const int32_t* rows, int max_rows,
                                        const int32_t* count, float softmax_scale, float* out,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                        void* stream) {
  if (B < 0 || B > 65535 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_rows < 1 || n_pool_rows < 0)
    return SKV_EINVAL;
  if (d != D) return SKV_EUNSUPPORTED;
  if (kv_kind != SKV_KV_BF16 && kv_kind != SKV_KV_INT8) return SKV_EUNSUPPORTED;
  if (B == 0) return SKV_OK;
  if (!q || !k_pool || !v_pool || !rows || !count || !out || !workspace) return SKV_EINVAL;
  if (kv_kind == SKV_KV_INT8 && (!k_scale || !v_scale)) return SKV_EINVAL;
  if (!aligned16(k_pool) || !aligned16(v_pool) || (reinterpret_cast<uintptr_t>(q) & 7)) return SKV_EINVAL;
  Plan p = make_plan(B, Hq, Hkv, max_rows);
  if (workspace_bytes < p.ticket_bytes + p.part_bytes) return SKV_ENOMEM;
  if (p.gy > 65535) return SKV_EUNSUPPORTED;
  AttendArgs a;
  a.q = q;
  a.kpool = static_cast<const uint8_t*>(k_pool);
  a.vpool = static_cast<const uint8_t*>(v_pool);
  a.kscale = k_scale;
  a.vscale = v_scale;
  a.req_row_stride = req_row_stride;
  a.n_pool_rows = n_pool_rows;
  a.rows = rows;
  a.max_rows = max_rows;
  a.count = count;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.hgroups = p.hgroups;
  a.nsplit = p.nsplit;
  a.rows_per_split = p.rows_per_split;
  a.scale_log2 = softmax_scale * kLog2e;
  a.tickets = static_cast<unsigned*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.ticket_bytes);
  a.out = out;
  a.status = dev_status;
  dim3 grid(p.nsplit, p.gy, B);
  if (kv_kind == SKV_KV_INT8)
    attend_kernel<SKV_KV_INT8><<<grid, kThreads, 0, as_stream(stream)>>>(a);
  else
    attend_kernel<SKV_KV_BF16><<<grid, kThreads, 0, as_stream(stream)>>>(a);
  return launch_status();
}
