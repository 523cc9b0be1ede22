// attend.cu -- exact attention over the selected rows (a6), split-K decode.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": exact int8
// attention on the top 2048 tokens, 64 sinks and the last 1024.  [P4] "3.14M
// Context on 3x 3090 ...", "No Need to Rewrite the Kernel": a row is found by
// adding (token*n_kv_heads + kv_head)*head_dim to the base, layout
// [token][kv_head][dim].
//
// Design.  A CTA owns one (request, KV head, group of up to 8 query heads,
// split of the selected rows) and runs three warp pairs.  Each pair takes
// 16-row tiles in turn through its own 3-stage shared-memory ring: the pair's
// 64 threads copy a tile's K and V rows of the KV head with 16-byte cp.async
// (gathering scattered 256-byte rows this way runs well above the rate of one
// bulk copy per row) and arrive on the stage's mbarrier when their copies
// land, so two tiles are in flight while one is computed.  The first tiles go
// out as soon as their row numbers are read; the split's row numbers, the
// int8 scales and the query heads are then staged in shared memory.  Rows
// land at pitches chosen so that the fragment loads below are free of
// shared-memory bank conflicts.
//
// The two warps of a pair split the head dimension: warp e owns dims
// [128e, 128e + 128) for both products.  Per tile each computes the partial
// logits of its half with m16n8k16 tensor-core MMAs (query heads are the M
// rows, padded to 16; two n8 tiles cover the 16 rows); the halves are
// exchanged through shared memory and added in a fixed order, so both warps
// run the same online softmax on bit-identical logits (its reference max
// moves only when a tile's logits pass it by more than 2^4 in probability,
// so most tiles rescale nothing; the rows' factors are read before the
// tile's copies land); each then accumulates
// its half of O^T += V^T P^T with the probabilities reused from the
// accumulators as the B operand.  The head dimension is permuted consistently
// on Q and K so that a lane reads contiguous 16-byte pieces of a row; the V
// dimension is permuted so that a lane reads 16 contiguous dims of 4 rows.
// int8 codes convert to fp16 exactly (0x6400 magic); the K scale multiplies
// the logits in fp32 and the V scale is folded into P.  bf16 rows keep bf16
// operands with P split into two bf16 terms.  The pairs' partials (m, l, O)
// merge in shared memory, each CTA writes one partial, and the last CTA of a
// (request, head group) merges the splits in split order (deterministic) and
// writes the output.
#include "common.cuh"

namespace skv {

// The rows every selection holds besides its picks (known-rows mode of the
// attention): request b's first S tokens and last W tokens, with k picks in
// between (all T = lengths[b] tokens when T <= S + W + k), as skv_score_select
// writes them; physical row b*req_row_stride + token.
struct KnownRows {
  const int32_t* lengths;
  int S, W, k;
};

namespace {

constexpr int D = 256;
constexpr int DH = D / 2;          // dims per warp of a pair
constexpr int kPairs = 3;
constexpr int kWarps = 2 * kPairs;
constexpr int kThreads = 32 * kWarps;
constexpr int kPart = 16 + 8 * D;  // m[8], l[8], O[8][D] floats per partial
constexpr int kMaxSplit = 64;
constexpr int kMaxRowsPerSplit = 512;
constexpr int kStages = 3;
constexpr int kTileRows = 16;
constexpr long kWaitLimit = 1L << 20;  // bounded mbarrier polls (~1 s with backoff)
// Lazy softmax rescaling: probabilities of a tile may reach 2^kLazy before
// the reference max moves (int8 rows fold the V scale into them in fp16, so
// this bounds p * v_scale by 16 * v_scale).
constexpr float kLazy = 4.f;
// Pair partials in shared memory: float (head, dim) at head*kMH + (dim/32)*33 +
// dim%32, so the fragment-order stores of a warp hit 32 different banks.
constexpr int kMH = 8 * 33 + 4;
constexpr int kMW = 8 * kMH;  // floats per pair
__device__ __forceinline__ int mix(int head, int dim) { return head * kMH + (dim >> 5) * 33 + (dim & 31); }

template <int KV>
struct Geo {
  static constexpr int ES = KV == SKV_KV_INT8 ? 1 : 2;
  static constexpr int RB = D * ES;       // bytes of one row of one head
  static constexpr int KP = RB + 64;      // K row pitch: 16-byte units = 4 (mod 8)
  static constexpr int VP = RB + 16;      // V row pitch: 16-byte units = 1 (mod 8)
  static constexpr int STAGE = kTileRows * (KP + VP);
  static constexpr int PAIR_BYTES = kStages * STAGE;
};

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
  // known-rows mode (lengths != NULL): the selection of request b holds its
  // first kS tokens and last kW tokens besides kK picks (all T tokens when
  // T <= kS + kW + kK); split s takes known_per_split of the former and
  // picks_per_split of the picks
  const int32_t* lengths;
  int kS, kW, kK, known_per_split, picks_per_split;
  float scale_log2;
  float* part;
  unsigned* tickets;
  float* out;
  int32_t* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase `parity` of `bar`; false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long i = 0; i < kWaitLimit; i++) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 16) __nanosleep(256);
  }
  return false;
}

// 16-byte asynchronous global -> shared copy (L2 only), and an arrive on `bar`
// once all of this thread's earlier copies have landed.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

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

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Barrier of the 64 threads of warp pair `pair` (named barriers 1..4).
__device__ __forceinline__ void pair_sync(int pair) {
  switch (pair) {
    case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
    case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
    case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
    default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
  }
}

// Pair barrier that also ANDs a predicate across the 64 threads, so both warps
// of the pair take the same branch afterwards.
__device__ __forceinline__ bool pair_all(int pair, bool v) {
  uint32_t r;
#define SKV_PAIR_ALL(ID)                                                                              \
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, " #ID             \
               ", 64, p;\n selp.u32 %0, 1, 0, q;\n}"                                                   \
               : "=r"(r)                                                                              \
               : "r"(static_cast<uint32_t>(v))                                                        \
               : "memory")
  switch (pair) {
    case 0: SKV_PAIR_ALL(1); break;
    case 1: SKV_PAIR_ALL(2); break;
    case 2: SKV_PAIR_ALL(3); break;
    default: SKV_PAIR_ALL(4); break;
  }
#undef SKV_PAIR_ALL
  return r != 0;
}

template <int KV>
__host__ __device__ constexpr size_t dyn_smem() {
  return static_cast<size_t>(kPairs) * Geo<KV>::PAIR_BYTES > static_cast<size_t>(kPairs) * kMW * sizeof(float)
             ? static_cast<size_t>(kPairs) * Geo<KV>::PAIR_BYTES
             : static_cast<size_t>(kPairs) * kMW * sizeof(float);
}

template <int KV>
__global__ __launch_bounds__(kThreads, 2) void attend_kernel(AttendArgs a) {
  using Gm = Geo<KV>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bars[kPairs][kStages];
  __shared__ int64_t s_prow[kMaxRowsPerSplit];
  __shared__ float s_ks[KV == SKV_KV_INT8 ? kMaxRowsPerSplit : 1], s_vs[KV == SKV_KV_INT8 ? kMaxRowsPerSplit : 1];
  __shared__ __align__(16) uint16_t s_q[8][D];
  __shared__ __align__(16) float s_x[kPairs][2][32][4];  // partial logits of each warp of a pair
  __shared__ float sm_m[kPairs][8], sm_l[kPairs][8];
  __shared__ float fin_m[8];
  __shared__ float wts[8][kMaxSplit];
  __shared__ int is_last;

  const int b = blockIdx.z, hy = blockIdx.y, split = blockIdx.x;
  const int h = hy / a.hgroups, hg = hy % a.hgroups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp >> 1, e = warp & 1;  // e: which half of the head dimension
  const int g = lane >> 2, c = lane & 3;

  // Rows of the split.  In known-rows mode (a.lengths set) the split takes a
  // slice of the rows every selection contains -- the sinks and the recent
  // tail, found from the request's length -- and a slice of the picks; the
  // first are staged and their first tiles copied before waiting for the
  // kernel that writes the selection (a programmatic dependency), the picks
  // after; then every tile is attended in turn.  s_prow[i]:
  // physical row of split row i (-1: none); known rows take [0, npad), picks
  // start at npad (a whole number of tiles).
  if (threadIdx.x < kPairs * kStages) mbar_init(&bars[threadIdx.x / kStages][threadIdx.x % kStages], 64);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

  const int64_t pitch = static_cast<int64_t>(a.Hkv) * Gm::RB;  // bytes per pool row
  const uint8_t* kbase = a.kpool + static_cast<int64_t>(h) * Gm::RB;
  const uint8_t* vbase = a.vpool + static_cast<int64_t>(h) * Gm::RB;

  unsigned char* pbuf = smem + pair * Gm::PAIR_BYTES;
  // The 64 threads of the pair copy tile `it` (16 K rows and 16 V rows) into
  // stage it % kStages in 16-byte pieces: thread u of the pair takes piece
  // u % (RB/16) of rows u / (RB/16) + 64/(RB/16) * i.  Rows without a
  // physical row read pool row 0 (masked later).  Each thread then arrives on
  // the stage's barrier when its copies have landed.
  constexpr int kPieces = Gm::RB / 16;                 // 16-byte pieces per row
  constexpr int kRowsPerRound = 64 / kPieces;          // rows covered by one round of the pair
  const int u = 32 * e + lane;
  int nr = 0;  // split rows whose physical rows are staged so far
  auto copy_tile = [&](int it) {
    const int stage = it % kStages;
    const int tb = (pair + kPairs * it) * kTileRows;
    unsigned char* kst = pbuf + stage * Gm::STAGE;
    unsigned char* vst = kst + kTileRows * Gm::KP;
    const int piece = u % kPieces;
#pragma unroll
    for (int i = 0; i < kTileRows / kRowsPerRound; i++) {
      const int row = u / kPieces + kRowsPerRound * i;
      int64_t prow = tb + row < nr ? s_prow[tb + row] : int64_t(-1);
      if (prow < 0) prow = 0;
      cp_async16(kst + row * Gm::KP + 16 * piece, kbase + prow * pitch + 16 * piece);
      cp_async16(vst + row * Gm::VP + 16 * piece, vbase + prow * pitch + 16 * piece);
    }
    cp_async_arrive(&bars[pair][stage]);
  };
  // Physical row of split row i from a token / row id p (-1: none).
  auto stage_row = [&](int i, int64_t p) {
    const bool ok = p >= 0 && p < a.n_pool_rows;
    if (!ok) set_status(a.status, SKV_DEV_RANGE);
    s_prow[i] = ok ? p : -1;
  };
  // The int8 scales of split rows [i0, i1), every load in flight before any
  // is stored (called once the rows' tiles are on their way).
  constexpr int kRowsPerThread = (kMaxRowsPerSplit + kThreads - 1) / kThreads;
  auto stage_scales = [&](int i0, int i1) {
    if (KV != SKV_KV_INT8) return;
    uint16_t ksv[kRowsPerThread], vsv[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; j++) {
      const int i = i0 + threadIdx.x + j * kThreads;
      const int64_t p = i < i1 ? s_prow[i] : int64_t(-1);
      ksv[j] = p >= 0 ? a.kscale[p * a.Hkv + h] : 0;
      vsv[j] = p >= 0 ? a.vscale[p * a.Hkv + h] : 0;
    }
#pragma unroll
    for (int j = 0; j < kRowsPerThread; j++) {
      const int i = i0 + threadIdx.x + j * kThreads;
      if (i < i1) {
        s_ks[i] = __half2float(__ushort_as_half(ksv[j]));
        s_vs[i] = __half2float(__ushort_as_half(vsv[j]));
      }
    }
  };

  int64_t T = 0;
  int head = 0, tailn = 0, npick = 0, kk0 = 0, nk = 0;
  if (a.lengths) {  // sinks [0, head) and the tail [T - tailn, T) of every selection
    T = a.lengths[b];
    if (T < 0) T = 0;
    if (a.req_row_stride > 0 && T > a.req_row_stride) {  // the selection clamps it the same way
      if (split == 0 && threadIdx.x == 0) set_status(a.status, SKV_DEV_RANGE);
      T = a.req_row_stride;
    }
    const bool dense = T <= static_cast<int64_t>(a.kS) + a.kW + a.kK;
    head = static_cast<int>(T < a.kS ? T : a.kS);
    tailn = static_cast<int>(T - head < a.kW ? T - head : a.kW);
    const int64_t npos = dense ? T : static_cast<int64_t>(a.kS) + a.kK + a.kW;
    npick = static_cast<int>(npos - head - tailn);
    kk0 = split * a.known_per_split;
    const int kk1 = kk0 + a.known_per_split < head + tailn ? kk0 + a.known_per_split : head + tailn;
    nk = kk1 > kk0 ? kk1 - kk0 : 0;
  }
  const int npad = (nk + kTileRows - 1) / kTileRows * kTileRows;
  for (int i = threadIdx.x; i < npad; i += blockDim.x) {
    if (i < nk) {
      const int pos = kk0 + i;
      const int64_t tok = pos < head ? pos : T - tailn + (pos - head);
      stage_row(i, static_cast<int64_t>(b) * a.req_row_stride + tok);
    } else {
      s_prow[i] = -1;
    }
  }
  constexpr int kQPerThread = (8 * D / 8 + kThreads - 1) / kThreads;
  uint4 qv[kQPerThread];
#pragma unroll
  for (int j = 0; j < kQPerThread; j++) {  // 16-byte pieces of 8 query heads
    const int i = threadIdx.x + j * kThreads;
    const int hd = i / (D / 8), x8 = i % (D / 8);
    const int hl = hg * 8 + hd;
    qv[j] = make_uint4(0u, 0u, 0u, 0u);
    if (i < 8 * D / 8 && hl < a.G)
      qv[j] = *reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.Hq + h * a.G + hl) * D + 8 * x8);
  }
  __syncthreads();
  nr = npad;
  const int ntk = npad / kTileRows;  // tiles of known rows
  int my_known = 0;
  for (int t = pair; t < ntk; t += kPairs) my_known++;
  int issued = 0;
  while (issued < my_known && issued < kStages) copy_tile(issued++);  // the pair's first known tiles go out at once
  stage_scales(0, npad);
#pragma unroll
  for (int j = 0; j < kQPerThread; j++) {
    const int i = threadIdx.x + j * kThreads;
    if (i < 8 * D / 8) *reinterpret_cast<uint4*>(&s_q[i / (D / 8)][8 * (i % (D / 8))]) = qv[j];
  }
  __syncthreads();

  // ---- query fragments of this warp's half (A operand of S = Q K^T) -----------
  // k-step ks covers 4 dims of the half: base(ks) below; slots 2c,2c+1 <- +0,+1
  // and 2c+8,2c+9 <- +2,+3, the same permutation as the K fragments.
  uint32_t qa[8][2];
#pragma unroll
  for (int ks = 0; ks < 8; ks++) {
    const int base = KV == SKV_KV_INT8 ? DH * e + 16 * (c + 4 * (ks >> 2)) + 4 * (ks & 3)
                                       : DH * e + 8 * (c + 4 * (ks >> 1)) + 4 * (ks & 1);
    const uint2 v = *reinterpret_cast<const uint2*>(&s_q[g][base]);
    if (KV == SKV_KV_INT8) {
      qa[ks][0] = pack_h2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
      qa[ks][1] = pack_h2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    } else {
      qa[ks][0] = v.x;
      qa[ks][1] = v.y;
    }
  }

  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; mt++) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m_run = -INFINITY, l_part = 0.f;

  int completed = 0;  // tiles whose copies have landed and were attended
  // Attends tile `it` of the pair (its copies were issued); false when the
  // wait for its copies gave up.
  auto attend_tile = [&](int it) -> bool {
    const int stage = it % kStages;
    const uint32_t parity = (it / kStages) & 1;
    const int tbase = (pair + kPairs * it) * kTileRows;  // index of the tile's first row in the split
    // This lane's rows' logit factors and V scales (0: no row), read while
    // the tile's copies are still landing.
    const int rr[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
    float fx[4], vsc[4];
    bool okr[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int idx = tbase + rr[i];
      okr[i] = idx < nr && s_prow[idx] >= 0;
      fx[i] = okr[i] ? (KV == SKV_KV_INT8 ? a.scale_log2 * s_ks[idx] : a.scale_log2) : 0.f;
      vsc[i] = okr[i] ? (KV == SKV_KV_INT8 ? s_vs[idx] : 1.f) : 0.f;
    }
    // Both warps of the pair must agree, or one would wait for the other at
    // the pair barriers below.
    if (!pair_all(pair, mbar_wait(&bars[pair][stage], parity))) {
      set_status(a.status, SKV_DEV_TIMEOUT);
      return false;
    }
    completed = it + 1;
    const unsigned char* kst = pbuf + stage * Gm::STAGE;
    const unsigned char* vst = kst + kTileRows * Gm::KP;

    // ---- partial S = Q K^T over this warp's half of the dims -------------------
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};  // second chains (odd k-steps)
    if (KV == SKV_KV_INT8) {
#pragma unroll
      for (int i = 0; i < 2; i++) {
        const uint4 ka = lds128(kst + g * Gm::KP + DH * e + 16 * (c + 4 * i));
        const uint4 kb = lds128(kst + (g + 8) * Gm::KP + DH * e + 16 * (c + 4 * i));
#pragma unroll
        for (int ws = 0; ws < 4; ws++) {
          const int ks = 4 * i + ws;
          const uint32_t w0 = word(ka, ws) ^ 0x80808080u;
          const uint32_t w1 = word(kb, ws) ^ 0x80808080u;
          float* d0 = (ks & 1) ? t0 : s0;
          float* d1 = (ks & 1) ? t1 : s1;
          mma_f16(d0, qa[ks][0], 0u, qa[ks][1], 0u, u8pair_to_h2(w0, 0x4140), u8pair_to_h2(w0, 0x4342));
          mma_f16(d1, qa[ks][0], 0u, qa[ks][1], 0u, u8pair_to_h2(w1, 0x4140), u8pair_to_h2(w1, 0x4342));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const uint4 ka = lds128(kst + g * Gm::KP + 2 * DH * e + 16 * (c + 4 * i));
        const uint4 kb = lds128(kst + (g + 8) * Gm::KP + 2 * DH * e + 16 * (c + 4 * i));
        mma_bf16(s0, qa[2 * i][0], 0u, qa[2 * i][1], 0u, ka.x, ka.y);
        mma_bf16(s1, qa[2 * i][0], 0u, qa[2 * i][1], 0u, kb.x, kb.y);
        mma_bf16(t0, qa[2 * i + 1][0], 0u, qa[2 * i + 1][1], 0u, ka.z, ka.w);
        mma_bf16(t1, qa[2 * i + 1][0], 0u, qa[2 * i + 1][1], 0u, kb.z, kb.w);
      }
    }
    // ---- exchange halves: full logits = half 0 + half 1 in both warps -------
    {
      float4 mine = make_float4(s0[0] + t0[0], s0[1] + t0[1], s1[0] + t1[0], s1[1] + t1[1]);
      *reinterpret_cast<float4*>(s_x[pair][e][lane]) = mine;
      pair_sync(pair);
      const float4 other = *reinterpret_cast<const float4*>(s_x[pair][1 - e][lane]);
      const float4 h0 = e == 0 ? mine : other, h1 = e == 0 ? other : mine;
      s0[0] = h0.x + h1.x;
      s0[1] = h0.y + h1.y;
      s1[0] = h0.z + h1.z;
      s1[1] = h0.w + h1.w;
    }

    // ---- online softmax on S[head g][rows 2c, 2c+1, 2c+8, 2c+9] ---------------
    // The reference max m_run of a head moves only when a tile's logits pass
    // it by more than kLazy (log2 units); then every head takes its exact
    // running max and the accumulators are rescaled.  Otherwise the tile's
    // probabilities are exp2(x - m_run) <= 2^kLazy and nothing is rescaled.
    // Both warps of the pair see bit-identical logits, so they decide alike.
    float x[4] = {s0[0], s0[1], s1[0], s1[1]};
#pragma unroll
    for (int i = 0; i < 4; i++) x[i] = okr[i] ? x[i] * fx[i] : -INFINITY;
    const float lmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    if (__any_sync(0xffffffffu, lmax > m_run + kLazy)) {
      float tmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float m_new = fmaxf(m_run, tmax);
      const float alpha = exp2f(m_run - (m_new == -INFINITY ? 0.f : m_new));
      l_part *= alpha;
      m_run = m_new;
      const float a_e = __shfl_sync(0xffffffffu, alpha, 8 * c);
      const float a_o = __shfl_sync(0xffffffffu, alpha, 8 * c + 4);
#pragma unroll
      for (int mt = 0; mt < 8; mt++) {
        o[mt][0] *= a_e;
        o[mt][1] *= a_o;
        o[mt][2] *= a_e;
        o[mt][3] *= a_o;
      }
    }
    const float m_use = m_run == -INFINITY ? 0.f : m_run;
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; i++) p[i] = exp2f(x[i] - m_use);
    l_part += (p[0] + p[1]) + (p[2] + p[3]);

    // ---- this half of O^T += V^T P^T -----------------------------------------
    // M-tile mt, slot g <-> dim 128e + 16g + 2mt, slot g+8 <-> the next dim.
    if (KV == SKV_KV_INT8) {
      const uint32_t bp0 = pack_h2(p[0] * vsc[0], p[1] * vsc[1]);
      const uint32_t bp1 = pack_h2(p[2] * vsc[2], p[3] * vsc[3]);
      uint4 v[4];
#pragma unroll
      for (int r = 0; r < 4; r++) v[r] = lds128(vst + rr[r] * Gm::VP + DH * e + 16 * g);
#pragma unroll
      for (int ws = 0; ws < 4; ws++) {  // dims 16g + 4ws .. +3 of the half
        const uint32_t t01 = prmt(word(v[0], ws), word(v[1], ws), 0x5140) ^ 0x80808080u;
        const uint32_t t23 = prmt(word(v[0], ws), word(v[1], ws), 0x7362) ^ 0x80808080u;
        const uint32_t u01 = prmt(word(v[2], ws), word(v[3], ws), 0x5140) ^ 0x80808080u;
        const uint32_t u23 = prmt(word(v[2], ws), word(v[3], ws), 0x7362) ^ 0x80808080u;
        mma_f16(o[2 * ws], u8pair_to_h2(t01, 0x4140), u8pair_to_h2(t01, 0x4342), u8pair_to_h2(u01, 0x4140),
                u8pair_to_h2(u01, 0x4342), bp0, bp1);
        mma_f16(o[2 * ws + 1], u8pair_to_h2(t23, 0x4140), u8pair_to_h2(t23, 0x4342), u8pair_to_h2(u23, 0x4140),
                u8pair_to_h2(u23, 0x4342), bp0, bp1);
      }
    } else {
      const uint32_t ph0 = pack_bf2(p[0], p[1]), ph1 = pack_bf2(p[2], p[3]);
      const float e0 = p[0] - __uint_as_float(ph0 << 16), e1 = p[1] - __uint_as_float(ph0 & 0xffff0000u);
      const float e2 = p[2] - __uint_as_float(ph1 << 16), e3 = p[3] - __uint_as_float(ph1 & 0xffff0000u);
      const uint32_t pl0 = pack_bf2(e0, e1), pl1 = pack_bf2(e2, e3);
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {  // 16-byte piece hh: dims 16g + 8hh .. +7 of the half
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; r++) v[r] = lds128(vst + rr[r] * Gm::VP + 2 * DH * e + 32 * g + 16 * hh);
#pragma unroll
        for (int ws = 0; ws < 4; ws++) {
          const int mt = 4 * hh + ws;  // dims 16g + 2mt, 16g + 2mt + 1 of the half
          const uint32_t a0 = prmt(word(v[0], ws), word(v[1], ws), 0x5410);
          const uint32_t a1 = prmt(word(v[0], ws), word(v[1], ws), 0x7632);
          const uint32_t a2 = prmt(word(v[2], ws), word(v[3], ws), 0x5410);
          const uint32_t a3 = prmt(word(v[2], ws), word(v[3], ws), 0x7632);
          mma_bf16(o[mt], a0, a1, a2, a3, ph0, ph1);
          mma_bf16(o[mt], a0, a1, a2, a3, pl0, pl1);
        }
      }
    }
    pair_sync(pair);  // both warps are done with this stage (and with s_x)
    return true;
  };
  bool live = true;
  // ---- the picks: after the kernel that wrote the selection -------------------------
  // The known rows' first tiles are already on their way; the picks are
  // staged before any tile is attended, so that their tiles follow the known
  // ones through the ring without a drain between the two.
  grid_dependency_wait();
  int np = 0, pos0 = 0;
  if (a.lengths) {
    const int pp0 = split * a.picks_per_split;
    const int pp1 = pp0 + a.picks_per_split < npick ? pp0 + a.picks_per_split : npick;
    np = pp1 > pp0 ? pp1 - pp0 : 0;
    pos0 = head + pp0;
  } else {
    int n = a.count[b];
    n = n < 0 ? 0 : (n > a.max_rows ? a.max_rows : n);
    const int r0 = split * a.rows_per_split;
    const int r1 = r0 + a.rows_per_split < n ? r0 + a.rows_per_split : n;
    np = r1 > r0 ? r1 - r0 : 0;
    pos0 = r0;
  }
  {  // every row id load in flight before any is used
    int32_t rid[kRowsPerThread];
#pragma unroll
    for (int j = 0; j < kRowsPerThread; j++) {
      const int i = threadIdx.x + j * kThreads;
      rid[j] = i < np ? a.rows[static_cast<int64_t>(b) * a.max_rows + pos0 + i] : -1;
    }
#pragma unroll
    for (int j = 0; j < kRowsPerThread; j++) {
      const int i = threadIdx.x + j * kThreads;
      if (i < np) stage_row(npad + i, rid[j] >= 0 ? static_cast<int64_t>(b) * a.req_row_stride + rid[j] : -1);
    }
  }
  __syncthreads();
  nr = npad + np;
  const int ntiles = (nr + kTileRows - 1) / kTileRows;
  int my_tiles = 0;
  for (int t = pair; t < ntiles; t += kPairs) my_tiles++;
  while (issued < my_tiles && issued < kStages) copy_tile(issued++);
  stage_scales(npad, nr);
  __syncthreads();
  // ---- every tile of the pair: the known rows', then the picks' ----------------------
  for (int it = 0; live && it < my_tiles; it++) {
    live = attend_tile(it);
    if (live && issued < my_tiles && issued < it + 1 + kStages) copy_tile(issued++);
  }
  // After a timeout, give the copies still in flight a bounded chance to land
  // before the buffers are reused for the merge.
  for (int it = completed; it < issued; it++) mbar_wait(&bars[pair][it % kStages], (it / kStages) & 1);

  // ---- merge the 2 pairs (partials staged in the ring buffers) --------------------
  __syncthreads();
  float* sm_o = reinterpret_cast<float*>(smem);  // [kPairs][kMW], see mix()
  if (e == 0) {
    float l_grp = l_part;
    l_grp += __shfl_xor_sync(0xffffffffu, l_grp, 1);
    l_grp += __shfl_xor_sync(0xffffffffu, l_grp, 2);
    if (c == 0) {
      sm_m[pair][g] = m_run;
      sm_l[pair][g] = l_grp;
    }
  }
#pragma unroll
  for (int mt = 0; mt < 8; mt++) {
    const int d0 = DH * e + 16 * g + 2 * mt;
    float* ow = sm_o + pair * kMW;
    ow[mix(2 * c, d0)] = o[mt][0];
    ow[mix(2 * c + 1, d0)] = o[mt][1];
    ow[mix(2 * c, d0 + 1)] = o[mt][2];
    ow[mix(2 * c + 1, d0 + 1)] = o[mt][3];
  }
  __syncthreads();
  const int gy = gridDim.y;
  float* mypart = a.part + ((static_cast<int64_t>(b) * gy + hy) * a.nsplit + split) * kPart;
  if (threadIdx.x < 8) {
    const int hd = threadIdx.x;
    float M = -INFINITY;
    for (int w = 0; w < kPairs; w++) M = fmaxf(M, sm_m[w][hd]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < kPairs; w++) L += exp2f(sm_m[w][hd] - M) * sm_l[w][hd];
    fin_m[hd] = M;
    mypart[hd] = M;
    mypart[8 + hd] = L;
  }
  __syncthreads();
  for (int e4 = threadIdx.x; e4 < 8 * D / 4; e4 += blockDim.x) {
    const int el = 4 * e4;
    const int hd = el / D, dd = el % D;
    const float M = fin_m[hd];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY)
      for (int w = 0; w < kPairs; w++) {
        const float wgt = exp2f(sm_m[w][hd] - M);
        const float* ow = sm_o + w * kMW;
        acc.x += wgt * ow[mix(hd, dd)];
        acc.y += wgt * ow[mix(hd, dd + 1)];
        acc.z += wgt * ow[mix(hd, dd + 2)];
        acc.w += wgt * ow[mix(hd, dd + 3)];
      }
    *reinterpret_cast<float4*>(mypart + 16 + el) = acc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    is_last = atomicAdd(&a.tickets[b * gy + hy], 1u) == static_cast<unsigned>(a.nsplit - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // ---- last CTA: merge the splits in split order ----------------------------------
  // When they fit in shared memory (the ring is free now), all the splits'
  // partials are copied in at once with 16-byte cp.async (one round of
  // latency); otherwise they are read from global memory (L2) in place.
  // Weights w[h][s] = exp2(m_s - M) / L are formed once per head.
  const float* parts = a.part + (static_cast<int64_t>(b) * gy + hy) * a.nsplit * kPart;
  if (static_cast<size_t>(a.nsplit) * kPart * sizeof(float) <= dyn_smem<KV>()) {
    float* sp = reinterpret_cast<float*>(smem);
    for (int i = threadIdx.x; i < a.nsplit * kPart / 4; i += blockDim.x) cp_async16(sp + 4 * i, parts + 4 * i);
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    parts = sp;
  }
  // One warp per head (heads hd = warp, warp + kWarps, ...; only the group's
  // real heads): the splits' maxima and weighted sums reduce across lanes in
  // a fixed order, and the weights go to shared memory once.
  for (int hd = warp; hd < 8; hd += kWarps) {
    if (hg * 8 + hd >= a.G) continue;  // padding head: no output
    float mx = -INFINITY;
    for (int s2 = lane; s2 < a.nsplit; s2 += 32) mx = fmaxf(mx, parts[s2 * kPart + hd]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float L = 0.f;
    for (int s2 = lane; s2 < a.nsplit; s2 += 32) {
      const float w = mx == -INFINITY ? 0.f : exp2f(parts[s2 * kPart + hd] - mx);
      wts[hd][s2] = w;
      L += w * parts[s2 * kPart + 8 + hd];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    for (int s2 = lane; s2 < a.nsplit; s2 += 32) wts[hd][s2] = L > 0.f ? wts[hd][s2] / L : 0.f;
  }
  __syncthreads();
  for (int e4 = threadIdx.x; e4 < 8 * D / 4; e4 += blockDim.x) {
    const int el = 4 * e4;
    const int hd = el / D, dd = el % D;
    const int hl = hg * 8 + hd;
    if (hl >= a.G) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s2 = 0; s2 < a.nsplit; s2++) {
      const float4 v = *reinterpret_cast<const float4*>(parts + s2 * kPart + 16 + el);
      const float wgt = wts[hd][s2];
      acc.x += wgt * v.x;
      acc.y += wgt * v.y;
      acc.z += wgt * v.z;
      acc.w += wgt * v.w;
    }
    *reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * a.Hq + h * a.G + hl) * D + dd) = acc;
  }
  if (threadIdx.x == 0) a.tickets[b * gy + hy] = 0;
}


// CTAs per SM on the current device; also raises the kernel's dynamic
// shared-memory limit there (once per device).
template <int KV>
int occupancy() {
  static std::atomic<int> cached[kMaxDevices];
  return once_per_device(cached, []() -> int {
    int per_sm = 0;
    if (cudaFuncSetAttribute(attend_kernel<KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(dyn_smem<KV>())) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<KV>, kThreads, dyn_smem<KV>()) !=
            cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      return -1;
    }
    return per_sm;
  });
}

struct Plan {
  int hgroups, gy, nsplit, rows_per_split, known_per_split, picks_per_split;
  size_t part_bytes, ticket_bytes;
};

Plan make_plan(int kv_kind, int B, int Hq, int Hkv, int max_rows, const KnownRows* known) {
  Plan p;
  const int G = Hq / Hkv;
  p.hgroups = (G + 7) / 8;
  p.gy = Hkv * p.hgroups;
  const int pairs = B * p.gy;
  const int per_sm = kv_kind == SKV_KV_INT8 ? occupancy<SKV_KV_INT8>() : occupancy<SKV_KV_BF16>();
  const int target = (per_sm > 0 ? per_sm : 1) * (sm_count() > 0 ? sm_count() : 1);
  int ns = target / pairs;  // at most one wave ...
  const int min_ns = (max_rows + kMaxRowsPerSplit - 1) / kMaxRowsPerSplit;  // ... unless splits get long
  const int max_ns = (max_rows + 63) / 64;
  if (ns > max_ns) ns = max_ns;
  if (ns > kMaxSplit) ns = kMaxSplit;
  if (ns < min_ns) ns = min_ns;
  if (ns < 1) ns = 1;
  int rps = (max_rows + ns - 1) / ns;
  rps = (rps + 15) / 16 * 16;
  if (rps > kMaxRowsPerSplit) rps = kMaxRowsPerSplit;
  ns = (max_rows + rps - 1) / rps;
  p.known_per_split = p.picks_per_split = 0;
  if (known) {  // a slice of the sinks + tail and a slice of the picks per split, each whole tiles
    const int nknown = known->S + known->W, npicks = max_rows - nknown;
    for (;; ns++) {
      p.known_per_split = ((nknown + ns - 1) / ns + 15) / 16 * 16;
      p.picks_per_split = ((npicks + ns - 1) / ns + 15) / 16 * 16;
      if (p.known_per_split + p.picks_per_split <= kMaxRowsPerSplit || ns >= kMaxSplit) break;
    }
    rps = p.known_per_split + p.picks_per_split;
  }
  p.nsplit = ns;
  p.rows_per_split = rps;
  p.part_bytes = static_cast<size_t>(B) * p.gy * ns * kPart * sizeof(float);
  p.ticket_bytes = (static_cast<size_t>(B) * p.gy * sizeof(unsigned) + 255) / 256 * 256;
  return p;
}

}  // namespace

size_t attend_workspace_bytes(int kv_kind, int B, int Hq, int Hkv, int max_rows, const KnownRows* known) {
  const Plan p = make_plan(kv_kind, B, Hq, Hkv, max_rows, known);
  return p.ticket_bytes + p.part_bytes;
}

int launch_attend(int kv_kind, int B, int Hq, int Hkv, const uint16_t* q, const void* k_pool, const void* v_pool,
                  const uint16_t* k_scale, const uint16_t* v_scale, int64_t req_row_stride, int64_t n_pool_rows,
                  const int32_t* rows, int max_rows, const int32_t* count, float softmax_scale, float* out,
                  void* workspace, size_t workspace_bytes, int32_t* dev_status, const KnownRows* known,
                  cudaStream_t st) {
  Plan p = make_plan(kv_kind, B, Hq, Hkv, max_rows, known);
  if (workspace_bytes < p.ticket_bytes + p.part_bytes) return SKV_ENOMEM;
  if (p.gy > 65535) return SKV_EUNSUPPORTED;
  if (known && p.known_per_split + p.picks_per_split > kMaxRowsPerSplit) return SKV_EUNSUPPORTED;
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
  a.lengths = known ? known->lengths : nullptr;
  a.kS = known ? known->S : 0;
  a.kW = known ? known->W : 0;
  a.kK = known ? known->k : 0;
  a.known_per_split = p.known_per_split;
  a.picks_per_split = p.picks_per_split;
  a.scale_log2 = softmax_scale * kLog2e;
  a.tickets = static_cast<unsigned*>(workspace);
  a.part = reinterpret_cast<float*>(static_cast<char*>(workspace) + p.ticket_bytes);
  a.out = out;
  a.status = dev_status;
  // Launched with programmatic stream serialization: the CTAs may start (and
  // set up, and in known-rows mode attend the sinks and the tail) while the
  // selection that produces `rows` is still finishing.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, p.gy, B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kv_kind == SKV_KV_INT8 ? dyn_smem<SKV_KV_INT8>() : dyn_smem<SKV_KV_BF16>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = kv_kind == SKV_KV_INT8 ? cudaLaunchKernelEx(&cfg, attend_kernel<SKV_KV_INT8>, a)
                                               : cudaLaunchKernelEx(&cfg, attend_kernel<SKV_KV_BF16>, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  return SKV_OK;
}

}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_attend_workspace_size(int B, int Hq, int Hkv, int d, int max_rows) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d != D || max_rows < 1 ||
      max_rows > kMaxSplit * kMaxRowsPerSplit)
    return 0;
  // Sized for the larger of the two row encodings' plans.
  const size_t s8 = attend_workspace_bytes(SKV_KV_INT8, B, Hq, Hkv, max_rows, nullptr);
  const size_t s16 = attend_workspace_bytes(SKV_KV_BF16, B, Hq, Hkv, max_rows, nullptr);
  return s8 > s16 ? s8 : s16;
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
  if (max_rows > kMaxSplit * kMaxRowsPerSplit) return SKV_EUNSUPPORTED;
  if (B == 0) return SKV_OK;
  if (n_pool_rows < 1) return SKV_EINVAL;
  if (!q || !k_pool || !v_pool || !rows || !count || !out || !workspace) return SKV_EINVAL;
  if (kv_kind == SKV_KV_INT8 && (!k_scale || !v_scale)) return SKV_EINVAL;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(q) & 7))
    return SKV_EINVAL;
  return launch_attend(kv_kind, B, Hq, Hkv, q, k_pool, v_pool, k_scale, v_scale, req_row_stride, n_pool_rows, rows,
                       max_rows, count, softmax_scale, out, workspace, workspace_bytes, dev_status, nullptr,
                       as_stream(stream));
}
