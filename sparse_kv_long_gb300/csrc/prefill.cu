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
// list, starting where the previous chunk's run ended (a cursor kept in the
// state; one binary search in the first chunk); rows are taken eight at a time, all sixteen
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
constexpr int kStatePitch = kD + 4;  // floats per query head: acc, m, l, cursor, pad (16-byte rows)

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
  float* state;      // [nq][Hq][kStatePitch]: acc[kD], m (log2 units), l, cursor, pad
  int first;         // the first chunk: the state has no contents yet
  int32_t* status;
  // Staging of the next chunk by the first CTAs of the same launch (blockIdx.x
  // < ncx; they start first): next_rows rows of K and V from device-readable
  // sources into the other half of the buffers.
  const uint16_t* k_next_src;
  const uint16_t* v_next_src;
  uint16_t* k_next;
  uint16_t* v_next;
  int64_t next_rows;
  int ncx;     // copy columns of the grid (0: no staging in this launch)
  int n_copy;  // copy CTAs = ncx * gridDim.y
};

// Copy CTA `cid` of n_copy: its share of the next chunk's K and V bytes, 16-byte
// pieces, several loads in flight per thread.
__device__ __forceinline__ void stage_next(const ChunkArgs& a, int cid) {
  const int64_t n16 = a.next_rows * a.Hkv * kD / 8;  // pieces per tensor
  const int64_t per = (n16 + a.n_copy - 1) / a.n_copy;
  const int64_t p0 = cid * per, p1 = p0 + per < n16 ? p0 + per : n16;
  const uint4* ks = reinterpret_cast<const uint4*>(a.k_next_src);
  const uint4* vs = reinterpret_cast<const uint4*>(a.v_next_src);
  uint4* kd = reinterpret_cast<uint4*>(a.k_next);
  uint4* vd = reinterpret_cast<uint4*>(a.v_next);
  constexpr int kU = 4;
  for (int64_t i0 = p0 + threadIdx.x; i0 < p1; i0 += static_cast<int64_t>(blockDim.x) * kU) {
    uint4 kv[kU], vv[kU];
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int64_t i = i0 + u * blockDim.x;
      if (i < p1) {
        kv[u] = ld_nc16(ks + i);
        vv[u] = ld_nc16(vs + i);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int64_t i = i0 + u * blockDim.x;
      if (i < p1) {
        kd[i] = kv[u];
        vd[i] = vv[u];
      }
    }
  }
}

// First index in idx[0, n) whose value is >= v (idx ascending).  Only the
// first chunk searches; later chunks start where the previous one stopped.
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
  if (static_cast<int>(blockIdx.x) < a.ncx) {
    stage_next(a, blockIdx.x * gridDim.y + blockIdx.y);
    return;
  }
  const int i = blockIdx.x - a.ncx, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int s_j0;
  const int cnt = min(max(a.count[i], 0), a.max_rows);
  const int32_t* row = a.idx + static_cast<int64_t>(i) * a.max_rows;
  // The query's picks are ascending, so the chunks take consecutive runs of
  // them: each (query, KV head) keeps the index where its next chunk starts in
  // the pad word after l of its group's first head.
  float* cur = a.state + (static_cast<int64_t>(i) * a.Hq + h * a.G) * kStatePitch + kD + 2;
  if (threadIdx.x == 0) {
    int j0;
    if (a.first) {
      j0 = lower_bound(row, cnt, a.c0);
      if (j0 > 0) set_status(a.status, SKV_DEV_RANGE);  // picks below 0 precede the first chunk
    } else {
      j0 = __float_as_int(*cur);
    }
    s_j0 = j0;
  }
  __syncthreads();
  const int j0 = s_j0;
  if (!a.first && (j0 >= cnt || __ldg(row + j0) >= a.c1)) {
    if (a.c1 == a.n_tokens && j0 < cnt && threadIdx.x == 0) set_status(a.status, SKV_DEV_RANGE);
    return;  // no pick of this query in the chunk: the state stays
  }
  int j1 = j0;  // end of the run inside [c0, c1), found by the row loop
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
    bool more = true;
    for (int jb = j0; more && jb < cnt; jb += kRowBatch) {
      uint4 kr[kRowBatch], vr[kRowBatch];
      bool ok[kRowBatch];
#pragma unroll
      for (int r = 0; r < kRowBatch; r++) {
        const int j = jb + r;
        const int64_t t = j < cnt ? static_cast<int64_t>(__ldg(row + j)) : a.c1;
        more = more && t < a.c1;  // ascending: the run stops at the first pick past the chunk
        ok[r] = more;
        if (more) j1 = j + 1;
        if (ok[r] && t < a.c0) {  // a list that is not ascending
          ok[r] = false;
          if (lane == 0) set_status(a.status, SKV_DEV_RANGE);
        }
        const int64_t off = ((ok[r] ? t - a.c0 : 0) * a.Hkv + h) * kD + 8 * lane;
        kr[r] = ok[r] ? ld_nc16(a.k_stage + off) : make_uint4(0u, 0u, 0u, 0u);
        vr[r] = ok[r] ? ld_nc16(a.v_stage + off) : make_uint4(0u, 0u, 0u, 0u);
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
  __syncthreads();  // every warp has read the cursor (s_j0) and found the same run
  if (threadIdx.x == 0) {
    *cur = __int_as_float(j1);
    if (a.c1 == a.n_tokens && j1 < cnt) set_status(a.status, SKV_DEV_RANGE);  // picks past the history
  }
}

// ---- the same on tensor cores (query groups of at most 8 heads) ---------------------
// One warp per (query, KV head).  A 16-row tile of the query's run:
//   S = Q . K^T   (m16n8k16, M = the group's heads padded to 16, N = rows,
//                  K = dims): lane (g, c) holds the 8-byte groups at dims
//                  64c + 4ks of row g -- one permutation of the 256 dims used
//                  for Q and K alike, so a lane reads a contiguous 128 B of a
//                  K row;
//   O^T += V^T . P^T  (M = dims, N = heads, K = rows): lane g owns dims
//                  [32g, 32g + 32) of the output; the probabilities come from
//                  the S accumulators (their layout is the B operand's), split
//                  into bf16 hi + lo parts so that they keep ~16 bits.
constexpr int kTcMaxG = 8;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__global__ __launch_bounds__(32) void prefill_chunk_tc_kernel(ChunkArgs a) {
  if (static_cast<int>(blockIdx.x) < a.ncx) {
    stage_next(a, blockIdx.x * gridDim.y + blockIdx.y);
    return;
  }
  const int i = blockIdx.x - a.ncx, h = blockIdx.y, lane = threadIdx.x;
  const int g = lane >> 2, c = lane & 3;
  const int cnt = min(max(a.count[i], 0), a.max_rows);
  const int32_t* row = a.idx + static_cast<int64_t>(i) * a.max_rows;
  float* cur = a.state + (static_cast<int64_t>(i) * a.Hq + h * a.G) * kStatePitch + kD + 2;
  int j0;
  if (a.first) {
    j0 = lower_bound(row, cnt, a.c0);
    if (j0 > 0 && lane == 0) set_status(a.status, SKV_DEV_RANGE);  // picks below 0 precede the first chunk
  } else {
    j0 = __float_as_int(*cur);
    if (j0 >= cnt || __ldg(row + j0) >= a.c1) {
      if (a.c1 == a.n_tokens && j0 < cnt && lane == 0) set_status(a.status, SKV_DEV_RANGE);
      return;  // no pick of this query in the chunk: the state stays
    }
  }
  // Q fragments (a0, a2) of head g, k-step ks: dims 64c + 4ks .. +3; padded heads are zero
  uint32_t qa[16][2];
  {
    const bool live = g < a.G;
    const uint16_t* qg = a.q + (static_cast<int64_t>(i) * a.Hq + h * a.G + (live ? g : 0)) * kD + 64 * c;
#pragma unroll
    for (int p = 0; p < 8; p++) {
      const uint4 v = live ? *reinterpret_cast<const uint4*>(qg + 8 * p) : make_uint4(0u, 0u, 0u, 0u);
      qa[2 * p][0] = v.x;
      qa[2 * p][1] = v.y;
      qa[2 * p + 1][0] = v.z;
      qa[2 * p + 1][1] = v.w;
    }
  }
  float o[16][4];  // O^T tile mt: (dim 32g + 2mt, heads 2c, 2c+1), (dim 32g + 2mt + 1, ...)
#pragma unroll
  for (int mt = 0; mt < 16; mt++) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m = -INFINITY, l = 0.f;  // running max (log2 units) and sum of head g
  int j1 = j0;
  bool more = true;
  for (int jt = j0; more && jt < cnt; jt += 16) {
    // the tile's token ids: lane r < 16 loads row jt + r; a row counts while the run is ascending in the chunk
    const int jr = jt + (lane & 15);
    const int64_t tr = jr < cnt ? static_cast<int64_t>(__ldg(row + jr)) : a.c1;
    const bool in_chunk = tr < a.c1;
    const unsigned inb = __ballot_sync(0xffffffffu, in_chunk) & 0xffffu;
    const int nvalid = __popc(~inb & 0xffffu) ? __ffs(~inb & 0xffffu) - 1 : 16;  // leading rows in the chunk
    if (nvalid < 16) more = false;
    j1 = jt + nvalid;
    const bool low = in_chunk && tr < a.c0 && (lane & 15) < nvalid;  // a list that is not ascending
    if (__any_sync(0xffffffffu, low) && lane == 0) set_status(a.status, SKV_DEV_RANGE);
    auto tok = [&](int r) -> int64_t { return __shfl_sync(0xffffffffu, tr, r); };
    auto valid = [&](int r, int64_t t) { return r < nvalid && t >= a.c0; };
    // S = Q K^T for rows g (n-tile 0) and 8 + g (n-tile 1)
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
      const int r = 8 * nt + g;
      const int64_t t = tok(r);
      const bool ok = valid(r, t);
      const uint16_t* kp = a.k_stage + ((ok ? t - a.c0 : 0) * a.Hkv + h) * kD + 64 * c;
      uint4 kv[8];
#pragma unroll
      for (int p = 0; p < 8; p++) kv[p] = ok ? ld_nc16(kp + 8 * p) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int p = 0; p < 8; p++) {
        const uint32_t a0[4] = {qa[2 * p][0], 0u, qa[2 * p][1], 0u};
        const uint32_t a1[4] = {qa[2 * p + 1][0], 0u, qa[2 * p + 1][1], 0u};
        mma_bf16_16816(sacc[nt], a0, kv[p].x, kv[p].y);
        mma_bf16_16816(sacc[nt], a1, kv[p].z, kv[p].w);
      }
    }
    // online softmax of head g over the tile's rows 2c, 2c+1 (n-tile 0) and 8 + 2c, 9 + 2c (n-tile 1)
    float sv[4];
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
      for (int e = 0; e < 2; e++) {
        const int r = 8 * nt + 2 * c + e;
        const int64_t t = tok(r);  // every lane shuffles: the source lane varies with c
        const bool ok = r < nvalid && t >= a.c0;
        sv[2 * nt + e] = ok ? sacc[nt][e] * a.scale_log2 : -INFINITY;
      }
    float tmax = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float mn = fmaxf(m, tmax);
    const float alpha = mn == -INFINITY ? 1.f : exp2f(m - mn);
    float pv[4], psum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; e++) {
      pv[e] = mn == -INFINITY ? 0.f : exp2f(sv[e] - mn);
      psum += pv[e];
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    l = l * alpha + psum;
    m = mn;
    // rescale O: lane (g, c) holds heads 2c, 2c+1, whose alpha lives in lanes 4(2c), 4(2c+1)
    const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * c), al1 = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
    for (int mt = 0; mt < 16; mt++) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
    // P^T as the B operand (rows 2c, 2c+1 | 8 + 2c, 9 + 2c; head g), hi and lo bf16 parts
    const uint32_t bh0 = pack_bf16x2(pv[0], pv[1]), bh1 = pack_bf16x2(pv[2], pv[3]);
    float h0, h1, h2, h3;
    bf16x2_to_f32(bh0, h0, h1);
    bf16x2_to_f32(bh1, h2, h3);
    const uint32_t bl0 = pack_bf16x2(pv[0] - h0, pv[1] - h1), bl1 = pack_bf16x2(pv[2] - h2, pv[3] - h3);
    // V rows 2c, 2c+1, 8 + 2c, 9 + 2c; dims [32g, 32g + 32) in four 16-byte pieces
    const uint16_t* vp[4];
    bool vok[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int r = (e & 1) + 2 * c + 8 * (e >> 1);
      const int64_t t = tok(r);
      vok[e] = valid(r, t);
      vp[e] = a.v_stage + ((vok[e] ? t - a.c0 : 0) * a.Hkv + h) * kD + 32 * g;
    }
#pragma unroll
    for (int q = 0; q < 4; q++) {
      uint4 vv[4];
#pragma unroll
      for (int e = 0; e < 4; e++) vv[e] = vok[e] ? ld_nc16(vp[e] + 8 * q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int w = 0; w < 4; w++) {  // m-tile 4q + w: dims 32g + 8q + 2w (a0, a2) and + 1 (a1, a3)
        const uint32_t r0 = (&vv[0].x)[w], r1 = (&vv[1].x)[w], r2 = (&vv[2].x)[w], r3 = (&vv[3].x)[w];
        const uint32_t av[4] = {__byte_perm(r0, r1, 0x5410), __byte_perm(r0, r1, 0x7632),
                                __byte_perm(r2, r3, 0x5410), __byte_perm(r2, r3, 0x7632)};
        mma_bf16_16816(o[4 * q + w], av, bh0, bh1);
        mma_bf16_16816(o[4 * q + w], av, bl0, bl1);
      }
    }
  }
  // merge into the running state: heads 2c, 2c+1 (when < G), dims [32g, 32g + 32)
  const float mh0 = __shfl_sync(0xffffffffu, m, 8 * c), mh1 = __shfl_sync(0xffffffffu, m, 8 * c + 4);
  const float lh0 = __shfl_sync(0xffffffffu, l, 8 * c), lh1 = __shfl_sync(0xffffffffu, l, 8 * c + 4);
#pragma unroll
  for (int e = 0; e < 2; e++) {
    const int hd = 2 * c + e;
    if (hd >= a.G) continue;
    float* st = a.state + (static_cast<int64_t>(i) * a.Hq + h * a.G + hd) * kStatePitch;
    const float mp = e ? mh1 : mh0, lp = e ? lh1 : lh0;
    const float M = a.first ? -INFINITY : st[kD], L = a.first ? 0.f : st[kD + 1];
    const float Mn = fmaxf(M, mp);
    const float wa = Mn == -INFINITY ? 0.f : exp2f(M - Mn), wb = Mn == -INFINITY ? 0.f : exp2f(mp - Mn);
#pragma unroll
    for (int mt = 0; mt < 16; mt++) {
      float2* sp = reinterpret_cast<float2*>(st + 32 * g + 2 * mt);
      const float2 old = a.first ? make_float2(0.f, 0.f) : *sp;
      *sp = make_float2(old.x * wa + o[mt][e] * wb, old.y * wa + o[mt][2 + e] * wb);
    }
    if (g == 0) {
      st[kD] = Mn;
      st[kD + 1] = L * wa + lp * wb;
    }
  }
  __syncwarp();
  if (lane == 0) {
    *cur = __int_as_float(j1);
    if (a.c1 == a.n_tokens && j1 < cnt) set_status(a.status, SKV_DEV_RANGE);  // picks past the history
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

// A device-readable view of a source pointer: device or managed memory as
// is, a registered host buffer through its device alias; false for anything
// else (pageable host memory is copied with cudaMemcpyAsync only).
bool device_view(const void* p, const uint16_t** out) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged && at.type != cudaMemoryTypeHost) ||
      !at.devicePointer)
    return false;
  *out = static_cast<const uint16_t*>(at.devicePointer);
  return true;
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
  static std::atomic<int> configured[kMaxDevices];
  if (smem_limit_once(configured, prefill_scores_kernel, smem) != SKV_OK) return SKV_ECUDA;
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
  const int64_t row_elems = static_cast<int64_t>(Hkv) * kD;
  // With device-readable sources (device memory, or a registered host buffer
  // through its alias) the launch that attends chunk j also stages chunk j + 1
  // into the other half of the buffers, so the copies overlap the attention.
  const uint16_t* kd = nullptr;
  const uint16_t* vd = nullptr;
  const bool overlap = chunk_tokens >= 2 && n_tokens > chunk_tokens / 2 && device_view(k_src, &kd) &&
                       device_view(v_src, &vd) && aligned16(kd) && aligned16(vd);
  const int64_t chunk = overlap ? chunk_tokens / 2 : chunk_tokens;
  const bool tc = Hq / Hkv <= kTcMaxG;
  const int ncx = overlap ? ((tc ? 4 : 1) * (sm_count() > 0 ? sm_count() : 1) + Hkv - 1) / Hkv : 0;
  ChunkArgs a{nq, Hq, Hkv, Hq / Hkv, q, k_stage, v_stage, 0, 0, n_tokens, idx, max_rows, count,
              softmax_scale * kLog2e, state, 1, dev_status, nullptr, nullptr, nullptr, nullptr, 0, 0, 0};
  // Chunk 0 also initialises the state, so one chunk pass runs even when
  // n_tokens == 0 (every query then attends to nothing).
  int buf = 0;
  for (int64_t c0 = 0; c0 == 0 || c0 < n_tokens; c0 += chunk) {
    const int64_t c1 = c0 + chunk < n_tokens ? c0 + chunk : n_tokens;
    uint16_t* kb = k_stage + buf * chunk * row_elems;
    uint16_t* vb = v_stage + buf * chunk * row_elems;
    if (c1 > c0 && (!overlap || c0 == 0)) {  // staged by the previous launch otherwise
      const size_t bytes = static_cast<size_t>(c1 - c0) * row_bytes;
      if (cudaMemcpyAsync(kb, k_src + c0 * row_elems, bytes, cudaMemcpyDefault, st) != cudaSuccess ||
          cudaMemcpyAsync(vb, v_src + c0 * row_elems, bytes, cudaMemcpyDefault, st) != cudaSuccess) {
        cudaGetLastError();
        return SKV_ECUDA;
      }
    }
    a.k_stage = kb;
    a.v_stage = vb;
    a.c0 = c0;
    a.c1 = c1;
    a.first = c0 == 0;
    const int64_t n1 = c1 + chunk < n_tokens ? c1 + chunk : n_tokens;
    a.ncx = overlap && n1 > c1 ? ncx : 0;
    a.n_copy = a.ncx * Hkv;
    a.next_rows = n1 - c1;
    a.k_next_src = kd ? kd + c1 * row_elems : nullptr;
    a.v_next_src = vd ? vd + c1 * row_elems : nullptr;
    a.k_next = k_stage + (buf ^ 1) * chunk * row_elems;
    a.v_next = v_stage + (buf ^ 1) * chunk * row_elems;
    const dim3 grid(static_cast<unsigned>(nq + a.ncx), static_cast<unsigned>(Hkv));
    if (tc)
      prefill_chunk_tc_kernel<<<grid, 32, 0, st>>>(a);
    else
      prefill_chunk_kernel<<<grid, kAttThreads, 0, st>>>(a);
    const int rc = launch_status();
    if (rc != SKV_OK) return rc;
    if (overlap) buf ^= 1;
  }
  const int64_t n_heads = static_cast<int64_t>(nq) * Hq;
  prefill_finish_kernel<<<static_cast<unsigned>((n_heads + 7) / 8), kAttThreads, 0, st>>>(state, n_heads, out);
  return launch_status();
}
