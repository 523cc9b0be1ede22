// prefill.cu -- chunked sparse prefill: per-query indexer scores and the
// loop-swapped attention over a host-resident history.
//
// [P4] "3.14M Context on 3x 3090 ...", "The Downside to Keep in Mind": during
// prefill every token picks its own top blocks, and together the picks of a
// prompt chunk touch almost the whole history, so reading each query's rows
// from host memory would move the history across the host link once per
// query.  The loops are swapped instead: the outer loop copies one chunk of
// the history into a small HBM working buffer once, the inner loop lets every
// query attend to its picks inside that chunk, and the partial softmax
// results of the chunks are merged.
//
// Scores.  The queries of a prefill chunk share one request's pooled keys, so
// their scores are one dense product Q_idx [nq x 128] . P^T [128 x n_blocks]:
// bf16 tensor-core tiles (mma.sync m16n8k16, fp32 accumulate), 64 queries x
// 128 blocks per CTA step.  A warp keeps its 16 queries' A fragments in
// registers for the whole sweep; key tiles are double-buffered in shared
// memory with cp.async and read with ldmatrix.  The CTAs of one block range
// are consecutive in launch order, so a key tile comes from DRAM once and
// from L2 for the other query tiles.  The epilogue writes order keys, which
// skv_topk_select turns into each query's causal selection.
//
// Attention.  One CTA per (query, KV head); warp w handles query heads
// w, w + 8, ... of the group; a lane holds 8 of the 256 dims.  The query's
// picks inside the staged chunk are a contiguous run of its ascending index
// list (two binary searches); rows are taken eight at a time, all sixteen
// 16-byte K/V loads of a lane in flight before the first use.  The chunk's
// partial (m, l, acc) is merged into the running state in global memory.
#include "common.cuh"

namespace skv {
namespace {

constexpr int kIdx = 128;          // indexer dimension
constexpr int kQT = 64;            // queries per score tile
constexpr int kBT = 128;           // blocks per score tile
constexpr int kPitch = kIdx + 8;   // bf16 per shared-memory row (272 B: conflict-free ldmatrix)
constexpr int kScoreThreads = 256;
constexpr int kTilesPerCta = 16;   // block tiles swept by one CTA

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy key tile `tile` (kBT blocks x 256 B) into shared memory; blocks past
// the end are zero-filled so every fragment read is defined.
__device__ __forceinline__ void load_key_tile(uint16_t* dst, const uint16_t* __restrict__ pooled, int64_t n_blocks,
                                              int64_t tile) {
  constexpr int kPieces = kBT * kIdx / 8;  // 16-byte pieces
  for (int p = threadIdx.x; p < kPieces; p += kScoreThreads) {
    const int r = p / (kIdx / 8), c = p % (kIdx / 8);
    const int64_t blk = tile * kBT + r;
    uint16_t* d = dst + r * kPitch + 8 * c;
    if (blk < n_blocks)
      cp16(d, pooled + blk * kIdx + 8 * c);
    else
      *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
  }
}

__global__ __launch_bounds__(kScoreThreads, 2) void prefill_scores_kernel(const uint16_t* __restrict__ q_idx, int nq,
                                                                          const uint16_t* __restrict__ pooled,
                                                                          int64_t n_blocks, uint32_t* __restrict__ out,
                                                                          int64_t stride, int32_t* status) {
  extern __shared__ __align__(16) uint16_t sm[];
  uint16_t* sq = sm;                    // [kQT][kPitch]
  uint16_t* sk = sm + kQT * kPitch;     // [2][kBT][kPitch]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kQT;
  const int64_t n_tiles = (n_blocks + kBT - 1) / kBT;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kTilesPerCta;
  const int64_t t1 = t0 + kTilesPerCta < n_tiles ? t0 + kTilesPerCta : n_tiles;
  if (t0 >= t1) return;
  // query tile (rows past nq zero) and the first key tile
  for (int p = threadIdx.x; p < kQT * kIdx / 8; p += kScoreThreads) {
    const int r = p / (kIdx / 8), c = p % (kIdx / 8);
    uint16_t* d = sq + r * kPitch + 8 * c;
    if (q0 + r < nq)
      cp16(d, q_idx + static_cast<int64_t>(q0 + r) * kIdx + 8 * c);
    else
      *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
  }
  load_key_tile(sk, pooled, n_blocks, t0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  // warp tile: 16 queries (m-tile warp & 3) x 64 blocks (half warp >> 2)
  const int mq = 16 * (warp & 3), nh = 64 * (warp >> 2);
  const int mi = lane >> 3, rr = lane & 7;
  uint32_t a[kIdx / 16][4];
  for (int64_t t = t0; t < t1; t++) {
    const int buf = static_cast<int>((t - t0) & 1);
    if (t + 1 < t1) load_key_tile(sk + (buf ^ 1) * kBT * kPitch, pooled, n_blocks, t + 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    if (t == t0) {
#pragma unroll
      for (int ks = 0; ks < kIdx / 16; ks++)  // A: rows mq + (mi&1)*8 + rr, k 16ks + (mi>>1)*8
        ldsm_x4(sq + (mq + (mi & 1) * 8 + rr) * kPitch + 16 * ks + (mi >> 1) * 8, a[ks][0], a[ks][1], a[ks][2],
                a[ks][3]);
    }
    const uint16_t* kt = sk + buf * kBT * kPitch;
    float c[8][4];
#pragma unroll
    for (int j = 0; j < 8; j++) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kIdx / 16; ks++) {
#pragma unroll
      for (int jp = 0; jp < 4; jp++) {  // n-tiles 2jp, 2jp+1: rows nh + 16jp + (mi>>1)*8 + rr, k 16ks + (mi&1)*8
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + (nh + 16 * jp + (mi >> 1) * 8 + rr) * kPitch + 16 * ks + (mi & 1) * 8, b0, b1, b2, b3);
        mma_bf16_16816(c[2 * jp], a[ks], b0, b1);
        mma_bf16_16816(c[2 * jp + 1], a[ks], b2, b3);
      }
    }
    // epilogue: c[j] = (query g, blocks 2cc, 2cc+1) and (query g + 8, ...)
    const int g = lane >> 2, cc = lane & 3;
#pragma unroll
    for (int j = 0; j < 8; j++) {
      const int64_t blk = t * kBT + nh + 8 * j + 2 * cc;
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int qi = q0 + mq + g + 8 * h;
        const float s0 = c[j][2 * h], s1 = c[j][2 * h + 1];
        if (isnan(s0) || isnan(s1)) set_status(status, SKV_DEV_NAN);
        if (qi < nq && blk < n_blocks) {
          uint32_t* o = out + static_cast<int64_t>(qi) * stride + blk;
          if (blk + 1 < n_blocks)
            *reinterpret_cast<uint2*>(o) = make_uint2(order_key_f32(s0), order_key_f32(s1));
          else
            o[0] = order_key_f32(s0);
        }
      }
    }
    __syncthreads();  // the buffer just read is refilled by the next step's prefetch
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---- attention over one staged history chunk --------------------------------------
constexpr int kD = 256;
constexpr int kAttThreads = 256;  // 8 warps
constexpr int kRowBatch = 8;      // rows whose K/V loads are in flight together
constexpr int kStatePitch = kD + 4;  // floats per query head: acc, m, l, pad (16-byte rows for float4)

struct ChunkArgs {
  int nq, Hq, Hkv, G;
  const uint16_t* q;        // [nq][Hq][kD]
  const uint16_t* k_stage;  // [chunk][Hkv][kD], row t - c0
  const uint16_t* v_stage;
  int64_t c0, c1, n_tokens;
  const int32_t* idx;  // [nq][max_rows] ascending
  int max_rows;
  const int32_t* count;
  float scale_log2;  // softmax scale * log2(e)
  float* state;      // [nq][Hq][kStatePitch]: acc[kD], m (log2 units), l, 2 pad
  int first;         // the first chunk: the state has no contents yet
  int32_t* status;
};

// First index in idx[0, n) whose value is >= v (idx ascending).
__device__ __forceinline__ int lower_bound(const int32_t* idx, int n, int64_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(__ldg(idx + mid)) < v)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ __launch_bounds__(kAttThreads) void prefill_chunk_kernel(ChunkArgs a) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_range[2];
  const int cnt = min(max(a.count[i], 0), a.max_rows);
  const int32_t* row = a.idx + static_cast<int64_t>(i) * a.max_rows;
  if (threadIdx.x == 0) {
    s_range[0] = lower_bound(row, cnt, a.c0);
    s_range[1] = lower_bound(row, cnt, a.c1);
    // picks below 0 precede the first chunk; picks at or past n_tokens follow the last
    if ((a.c0 == 0 && s_range[0] > 0) || (a.c1 == a.n_tokens && s_range[1] < cnt))
      set_status(a.status, SKV_DEV_RANGE);
  }
  __syncthreads();
  const int j0 = s_range[0], j1 = s_range[1];
  if (j0 == j1 && !a.first) return;  // no pick of this query in the chunk: the state stays
  for (int gi = warp; gi < a.G; gi += kAttThreads / 32) {
    const int g = h * a.G + gi;
    float qv[8], acc[8];
    {
      const uint4 qq = *reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(i) * a.Hq + g) * kD + 8 * lane);
      unpack8(qq, qv);
    }
#pragma unroll
    for (int u = 0; u < 8; u++) acc[u] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int jb = j0; jb < j1; jb += kRowBatch) {
      uint4 kr[kRowBatch], vr[kRowBatch];
      bool ok[kRowBatch];
#pragma unroll
      for (int r = 0; r < kRowBatch; r++) {
        const int j = jb + r;
        const int64_t t = j < j1 ? static_cast<int64_t>(__ldg(row + j)) : a.c0;
        ok[r] = j < j1 && t >= a.c0 && t < a.c1;  // false only for a list that is not ascending
        const int64_t off = ((ok[r] ? t - a.c0 : 0) * a.Hkv + h) * kD + 8 * lane;
        kr[r] = ok[r] ? ld_nc16(a.k_stage + off) : make_uint4(0u, 0u, 0u, 0u);
        vr[r] = ok[r] ? ld_nc16(a.v_stage + off) : make_uint4(0u, 0u, 0u, 0u);
        if (j < j1 && !ok[r] && lane == 0) set_status(a.status, SKV_DEV_RANGE);
      }
      float s[kRowBatch];
#pragma unroll
      for (int r = 0; r < kRowBatch; r++) {
        float kf[8];
        unpack8(kr[r], kf);
        float p = 0.f;
#pragma unroll
        for (int u = 0; u < 8; u++) p = fmaf(qv[u], kf[u], p);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
        s[r] = ok[r] ? p * a.scale_log2 : -INFINITY;
      }
      float mb = m;
#pragma unroll
      for (int r = 0; r < kRowBatch; r++) mb = fmaxf(mb, s[r]);
      if (mb == -INFINITY) continue;  // nothing valid yet
      const float alpha = exp2f(m - mb);  // m == -inf: 0
      l *= alpha;
#pragma unroll
      for (int u = 0; u < 8; u++) acc[u] *= alpha;
#pragma unroll
      for (int r = 0; r < kRowBatch; r++) {
        const float p = exp2f(s[r] - mb);  // invalid rows: exp2(-inf) = 0
        l += p;
        float vf[8];
        unpack8(vr[r], vf);
#pragma unroll
        for (int u = 0; u < 8; u++) acc[u] = fmaf(p, vf[u], acc[u]);
      }
      m = mb;
    }
    // merge with the running state
    float* st = a.state + (static_cast<int64_t>(i) * a.Hq + g) * kStatePitch;
    float M = -INFINITY, L = 0.f;
    float A[8];
#pragma unroll
    for (int u = 0; u < 8; u++) A[u] = 0.f;
    if (!a.first) {
      M = st[kD];
      L = st[kD + 1];
      const float4 x0 = *reinterpret_cast<const float4*>(st + 8 * lane);
      const float4 x1 = *reinterpret_cast<const float4*>(st + 8 * lane + 4);
      A[0] = x0.x; A[1] = x0.y; A[2] = x0.z; A[3] = x0.w;
      A[4] = x1.x; A[5] = x1.y; A[6] = x1.z; A[7] = x1.w;
    }
    const float Mn = fmaxf(M, m);
    if (Mn != -INFINITY) {
      const float wa = exp2f(M - Mn), wb = exp2f(m - Mn);
      L = L * wa + l * wb;
#pragma unroll
      for (int u = 0; u < 8; u++) A[u] = A[u] * wa + acc[u] * wb;
      M = Mn;
    }
    *reinterpret_cast<float4*>(st + 8 * lane) = make_float4(A[0], A[1], A[2], A[3]);
    *reinterpret_cast<float4*>(st + 8 * lane + 4) = make_float4(A[4], A[5], A[6], A[7]);
    if (lane == 0) {
      st[kD] = M;
      st[kD + 1] = L;
    }
  }
}

// out = acc / l (zeros for a query head that attended to nothing).
__global__ __launch_bounds__(kAttThreads) void prefill_finish_kernel(const float* __restrict__ state, int64_t n_heads,
                                                                     float* __restrict__ out) {
  const int64_t gh = static_cast<int64_t>(blockIdx.x) * (kAttThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gh >= n_heads) return;
  const float* st = state + gh * kStatePitch;
  const float L = st[kD + 1];
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float* o = out + gh * kD + 8 * lane;
  const float4 x0 = *reinterpret_cast<const float4*>(st + 8 * lane);
  const float4 x1 = *reinterpret_cast<const float4*>(st + 8 * lane + 4);
  *reinterpret_cast<float4*>(o) = make_float4(x0.x * inv, x0.y * inv, x0.z * inv, x0.w * inv);
  *reinterpret_cast<float4*>(o + 4) = make_float4(x1.x * inv, x1.y * inv, x1.z * inv, x1.w * inv);
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT int skv_prefill_index_scores(int nq, const uint16_t* q_idx, const uint16_t* pooled, int64_t n_blocks,
                                        uint32_t* order_keys, int64_t key_stride, int32_t* dev_status,
                                        void* stream) {
  if (nq < 0 || n_blocks < 0 || key_stride < n_blocks || key_stride % 2) return SKV_EINVAL;
  if (nq == 0 || n_blocks == 0) return SKV_OK;
  if (!q_idx || !pooled || !order_keys || !aligned16(q_idx) || !aligned16(pooled) ||
      (reinterpret_cast<uintptr_t>(order_keys) & 7u))
    return SKV_EINVAL;
  const int64_t n_tiles = (n_blocks + kBT - 1) / kBT;
  const int64_t gy = (n_tiles + kTilesPerCta - 1) / kTilesPerCta;
  const int64_t gx = (nq + kQT - 1) / kQT;
  if (gy > 65535 || gx > 2147483647) return SKV_EUNSUPPORTED;
  constexpr size_t smem = (static_cast<size_t>(kQT) + 2 * kBT) * kPitch * sizeof(uint16_t);
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(prefill_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess) {
      cudaGetLastError();
      return SKV_ECUDA;
    }
    configured = true;
  }
  prefill_scores_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kScoreThreads, smem,
                          as_stream(stream)>>>(q_idx, nq, pooled, n_blocks, order_keys, key_stride, dev_status);
  return launch_status();
}

SKV_EXPORT int skv_prefill_attend(int nq, int Hq, int Hkv, int d, const uint16_t* q, const uint16_t* k_src,
                                  const uint16_t* v_src, int64_t n_tokens, uint16_t* k_stage, uint16_t* v_stage,
                                  int64_t chunk_tokens, const int32_t* idx, int max_rows, const int32_t* count,
                                  float softmax_scale, float* state, float* out, int32_t* dev_status,
                                  void* stream) {
  if (nq < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > 32 || d != kD || n_tokens < 0 || chunk_tokens < 1 ||
      max_rows < 1)
    return SKV_EINVAL;
  if (nq == 0) return SKV_OK;
  if (nq > 2147483647 / Hq || Hkv > 65535) return SKV_EUNSUPPORTED;
  if (!q || !idx || !count || !state || !out || !aligned16(q) || !aligned16(state) || !aligned16(out))
    return SKV_EINVAL;
  if (n_tokens > 0 && (!k_src || !v_src || !k_stage || !v_stage || !aligned16(k_stage) || !aligned16(v_stage)))
    return SKV_EINVAL;
  cudaStream_t st = as_stream(stream);
  const size_t row_bytes = static_cast<size_t>(Hkv) * kD * sizeof(uint16_t);
  ChunkArgs a{nq, Hq, Hkv, Hq / Hkv, q, k_stage, v_stage, 0, 0, n_tokens, idx, max_rows, count,
              softmax_scale * kLog2e, state, 1, dev_status};
  // Chunk 0 also initialises the state, so one chunk pass runs even when
  // n_tokens == 0 (every query then attends to nothing).
  for (int64_t c0 = 0; c0 == 0 || c0 < n_tokens; c0 += chunk_tokens) {
    const int64_t c1 = c0 + chunk_tokens < n_tokens ? c0 + chunk_tokens : n_tokens;
    if (c1 > c0) {
      const size_t bytes = static_cast<size_t>(c1 - c0) * row_bytes;
      if (cudaMemcpyAsync(k_stage, k_src + c0 * Hkv * kD, bytes, cudaMemcpyDefault, st) != cudaSuccess ||
          cudaMemcpyAsync(v_stage, v_src + c0 * Hkv * kD, bytes, cudaMemcpyDefault, st) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ECUDA;
      }
    }
    a.c0 = c0;
    a.c1 = c1;
    a.first = c0 == 0;
    prefill_chunk_kernel<<<dim3(static_cast<unsigned>(nq), static_cast<unsigned>(Hkv)), kAttThreads, 0, st>>>(a);
    const int rc = launch_status();
    if (rc != SKV_OK) return rc;
  }
  const int64_t n_heads = static_cast<int64_t>(nq) * Hq;
  prefill_finish_kernel<<<static_cast<unsigned>((n_heads + 7) / 8), kAttThreads, 0, st>>>(state, n_heads, out);
  return launch_status();
}
