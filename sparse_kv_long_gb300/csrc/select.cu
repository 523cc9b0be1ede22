// select.cu -- fused indexer score scan + deterministic top-k (a3 + a4).
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": every token
// is scored through the sketch each step, the top 2048 are picked by a
// deterministic radix select, one pick per layer, and unioned with 64 sinks
// and the last 1024 tokens.  [P4] "3.14M Context on 3x 3090 ...", "Why": with
// pooled keys the top blocks are expanded to tokens once the context exceeds
// 4*block_topk + 3.
//
// One cooperative launch per layer-step.  The CTAs of a request split its
// candidate rows into contiguous chunks.  Each CTA
//   1. streams its chunk of indexer rows (the same loops, hence the same
//      scores, as skv_index_score: coalesced 16-byte loads, eight in flight
//      per lane) and keeps the order keys in shared memory;
//   2. works on rel = key - base: int32 sketch scores are bounded
//      (|s| < 2^20), so rel fits 21 bits above a fixed base; fp32 order keys
//      take all 32 bits;
//   3. radix passes over rel, top digits first: each non-final pass (<= 13
//      bits) histograms the keys still matching the prefix, adds the bins to
//      the request's global histogram, and after a request-wide barrier every
//      CTA derives the same digit (the first pass reads back only windows of
//      bins below the highest occupied one, the first of them guessed from
//      the CTA's own top bin and read in the same round trip as the
//      request's);
//   4. the final pass (8 bits) adds its bins to a request-wide histogram and
//      publishes per-CTA suffix counts (keys above the prefix plus keys in
//      bins >= d, for every d); once every CTA has arrived -- the poll reads
//      the request's bins with the arrival count, and they are complete when
//      they sum to the keys matching the prefix -- every CTA knows the exact
//      k-th key K*, how many keys equal to K* are taken, and -- from two
//      counts per earlier chunk -- where its own picks go; it writes them in
//      ascending index order (equal keys: lowest index first).
// int32 scores need one barrier and the final poll, fp32 scores two barriers
// and the poll.  A barrier is a monotonic arrival counter (release add,
// acquire poll); the last CTA to leave resets it.  Polls are bounded: a wait
// that runs out sets SKV_DEV_TIMEOUT and the kernel goes on.  The
// cooperative launch guarantees that all CTAs are resident together.
#include "fold.cuh"
#include "score_common.cuh"

namespace skv {
namespace {

constexpr int kWarpsF = 16;
constexpr int kThreads = 32 * kWarpsF;
constexpr int kMaxDigit = 13;                    // bits of a non-final pass
constexpr int kBins = 1 << kMaxDigit;
constexpr int kLastBits = 8;                     // bits of the final pass
constexpr int kLastBins = 1 << kLastBits;
constexpr int kFin = 4 + kLastBins;              // per-CTA final record: kLastBins + 1 suffix counts, pad
constexpr int kCMax = 512;                       // CTAs per request
constexpr long kSpinLimit = 1L << 21;            // bounded barrier polls (well under a second)
constexpr size_t kKeyBudget = 96 * 1024;         // shared memory for the chunk's order keys
constexpr uint32_t kInt4Base = 0x80000000u - (1u << 20);  // order key of score -2^20
constexpr int kWin = 1024;                                 // bins read back per window (int4 first pass)
constexpr int kAhead = 256;                                // first window: bins above the CTA's own top
constexpr uint32_t kUnknown = 0xffffffffu;                 // keys matching the prefix: not counted

// Scratch of one request, at a fixed stride whatever B is, so that one
// zero-filled workspace serves calls with any number of requests: the words
// that must start at zero (barrier counters, the range word, histograms) are
// returned to zero by the request's CTAs before the launch ends, the epoch
// only grows (its tag never takes the value 0 of a fresh workspace), and a
// per-CTA record word is read only once it carries this launch's tag.
//   bar   [2]              arrivals (monotonic within a launch), exits
//   rng   [2]              highest occupied first-pass bin + 1, launch epoch
//   hist  [2][kBins]       non-final passes
//   fhist [kLastBins]      final pass, request-wide bins
//   fin   [kCMax][kFin]    final pass, per-CTA suffix counts, each word tagged
//                          with the launch epoch (high 16 bits)
constexpr size_t kReqWords = 4 + 2ull * kBins + kLastBins + static_cast<size_t>(kCMax) * kFin;
static_assert(kReqWords % 4 == 0, "request blocks stay 16-byte aligned");
static_assert(kKeyBudget / 4 < 65536, "a CTA's counts fit the 16 low bits of a tagged record word");

struct Ws {
  unsigned* base;
  __device__ __forceinline__ unsigned* req(int b) const { return base + static_cast<size_t>(b) * kReqWords; }
  __device__ __forceinline__ unsigned* bar(int b) const { return req(b); }
  __device__ __forceinline__ unsigned* rng(int b) const { return req(b) + 2; }
  __device__ __forceinline__ unsigned* hist(int pass, int b) const { return req(b) + 4 + static_cast<size_t>(pass) * kBins; }
  __device__ __forceinline__ unsigned* fhist(int b) const { return req(b) + 4 + 2 * kBins; }
  __device__ __forceinline__ int* fin(int b, int c) const {
    return reinterpret_cast<int*>(req(b) + 4 + 2 * kBins + kLastBins) + static_cast<size_t>(c) * kFin;
  }
};

size_t ws_bytes(int B) { return (kReqWords * 4 * static_cast<size_t>(B) + 255) / 256 * 256; }

Ws ws_carve(void* base, int) { return Ws{static_cast<unsigned*>(base)}; }

// Optional per-step preparation done inside the launch (skv_decode_select):
// every CTA folds its request's query into int8 itself (same arithmetic as
// skv_decode_prepare, so the same q8 in every CTA), and CTA h < Hkv of each
// request appends head h of the current token (sketch codes, int8 K and V
// rows).  The appended token is in the recent tail, so no CTA scores it.
struct Prep {
  const uint16_t* q;  // bf16 [B][Hq][d]; NULL: q8 is read from Args::query
  const uint16_t* newk;
  const uint16_t* newv;
  const float* basis;  // [d][64]
  const float* c;      // [Hkv][64]
  const int64_t* new_rows;
  uint8_t* sketch;  // [rows][Hkv*32]
  int8_t* k8;
  __half* ks;
  int8_t* v8;
  __half* vs;
  int8_t* q8_out;  // optional copy of the folded query
  int Hq, Hkv, d;
};

struct Args {
  int mode, width;
  const void* query;
  const void* keys;
  int64_t n_cap;
  const int32_t* lengths;
  int ratio, k, S, W;
  int32_t* idx;
  int max_rows;
  int32_t* count;
  uint32_t* okeys;  // optional copy of the order keys
  int32_t* status;
  int B;
  Prep prep;
};

// The preparation step inside every CTA of a request: the group sums of the
// query heads (Hkv vectors) and, in CTA h < Hkv, the appended key of head h
// share one pass over the basis (one 32-dim slice of one basis column per
// thread, the arithmetic of skv_decode_prepare); every CTA then derives the
// request's scale and int8 query itself (the same bits everywhere, no
// waiting), and CTA h writes head h's sketch codes and int8 K and V rows.
// `scratch` holds (Hkv + 2)*d + (Hkv + 1)*64*ceil(d/32) + Hkv*64 floats.
__device__ __noinline__ void prepare_in_cta(const Prep& p, int b, int c, int64_t n_cap, int64_t T, int S, int W,
                                            float* scratch, int8_t* s_q8, float* red, int32_t* status) {
  using fold::kRank;
  const int Hkv = p.Hkv, d = p.d, G = p.Hq / Hkv, ns = fold::n_slices(d), width = Hkv * kRank;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const bool app = c < Hkv;  // this CTA appends head c
  const int nv = Hkv + (app ? 1 : 0);
  float* X = scratch;                   // [Hkv + 1][d]: group sums, appended key of head c
  float* part = X + (Hkv + 1) * d;      // [ns][Hkv + 1][64]
  float* qp = part + ns * (Hkv + 1) * kRank;  // [width]
  uint16_t* kv_rows = reinterpret_cast<uint16_t*>(qp + width);  // [2][d] bf16 rows to encode
  int64_t row = 0;
  if (app) {
    row = p.new_rows[b];
    for (int u = tid; u < 2 * (d / 8); u += nt) {
      const int which = u / (d / 8), piece = u - which * (d / 8);
      const uint16_t* src = (which == 0 ? p.newk : p.newv) + (static_cast<int64_t>(b) * Hkv + c) * d + 8 * piece;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                       __cvta_generic_to_shared(kv_rows + which * d + 8 * piece))),
                   "l"(src)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const bool one_task = ns * kRank <= nt;
  float bcol[fold::kSlice];
  if (one_task && tid < ns * kRank) fold::load_slice(p.basis, d, tid % kRank, tid / kRank, bcol);
  for (int i = tid; i < Hkv * d; i += nt) {
    const int h = i / d, x = i - h * d;
    X[i] = fold::group_sum(p.q + (static_cast<int64_t>(b) * p.Hq + static_cast<int64_t>(h) * G) * d, G, d, x);
  }
  if (app)
    for (int x = tid; x < d; x += nt) X[Hkv * d + x] = bf16_bits_to_f32(p.newk[(static_cast<int64_t>(b) * Hkv + c) * d + x]);
  __syncthreads();
  if (one_task) {
    if (tid < ns * kRank) {
      const int sl = tid / kRank, j = tid - sl * kRank;
      fold::dot_slice(bcol, X, d, nv, d, sl, part + sl * (Hkv + 1) * kRank + j, kRank);
    }
  } else {
    for (int task = tid; task < ns * kRank; task += nt) {
      const int sl = task / kRank, j = task - sl * kRank;
      fold::proj_slice(p.basis, X, d, nv, d, j, sl, part + sl * (Hkv + 1) * kRank + j, kRank);
    }
  }
  __syncthreads();
  float amax = 0.f;
  for (int m = tid; m < width; m += nt) {
    const float v = __fmul_rn(fold::combine_slices(part + m, (Hkv + 1) * kRank, ns), p.c[m]);
    qp[m] = v;
    amax = fmaxf(amax, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = 0.f;
  for (int v = 0; v < (nt >> 5); v++) amax = fmaxf(amax, red[v]);
  const float sigma = __fdiv_rn(amax, 127.f);
  for (int m = tid; m < width; m += nt) {
    const int8_t qc = fold::query_code(qp[m], sigma);
    s_q8[m] = qc;
    if (c == 0 && p.q8_out) p.q8_out[static_cast<int64_t>(b) * width + m] = qc;
  }
  if (app) {
    const float* pk = part + Hkv * kRank;  // the appended key's slices
    if (tid < kRank / 2) {
      const int j0 = 2 * tid;
      const int stride = (Hkv + 1) * kRank;
      const int c0 = fold::sketch_code(fold::combine_slices(pk + j0, stride, ns), p.c[c * kRank + j0]);
      const int c1 = fold::sketch_code(fold::combine_slices(pk + j0 + 1, stride, ns), p.c[c * kRank + j0 + 1]);
      p.sketch[row * (Hkv * kRank / 2) + c * (kRank / 2) + tid] = static_cast<uint8_t>((c0 & 15) | ((c1 & 15) << 4));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (warp < 2) {
      float rowv[16];
#pragma unroll
      for (int i = 0; i < 16; i++) {
        const int x = lane + 32 * i;
        rowv[i] = x < d ? bf16_bits_to_f32(kv_rows[warp * d + x]) : 0.f;
      }
      fold::encode_row_warp(rowv, d, (warp == 0 ? p.k8 : p.v8) + (row * Hkv + c) * d,
                            (warp == 0 ? p.ks : p.vs) + row * Hkv + c);
    }
    const int64_t t = row - static_cast<int64_t>(b) * n_cap;
    if (tid == 0 && c == 0 && t >= S && t < T - W) set_status(status, SKV_DEV_RANGE);  // would race the scan
  }
  __syncthreads();
}

// Request-wide barrier: the n-th barrier of a launch waits until the
// request's arrival counter reaches n * C.
__device__ void req_barrier(unsigned* arrive, unsigned target, int32_t* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(arrive) : "memory");
    bool ok = false;
    for (long i = 0; i < kSpinLimit; i++) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(arrive) : "memory");
      if (v >= target) {
        ok = true;
        break;
      }
      if (i > 64) __nanosleep(32);
    }
    if (!ok) set_status(status, SKV_DEV_TIMEOUT);
  }
  __syncthreads();
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const unsigned* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// rel >> sh, with a shift of 32 giving 0.
__device__ __forceinline__ uint32_t top_bits(uint32_t rel, int sh) { return sh >= 32 ? 0u : rel >> sh; }

// Find the digit holding the need-th largest key from bins h[0..nb) and the
// number of keys in the bins above it.  Position r = 0, 1, ... counts bins
// from the top (bin nb-1-r).  Warp v sums positions [v*span, (v+1)*span) with
// lane-strided (bank-conflict-free) reads; the warp whose range holds the
// need-th key then scans it 32 positions at a time.
__device__ void find_digit(const uint32_t* h, int nb, uint32_t need, uint32_t* digit, uint32_t* above_out,
                           int32_t* status) {
  __shared__ unsigned wsum[kWarpsF];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int span = ((nb + kWarpsF - 1) / kWarpsF + 31) / 32 * 32;
  const int r0 = warp * span;
  unsigned sum = 0;
  for (int r = r0 + lane; r < r0 + span && r < nb; r += 32) sum += h[nb - 1 - r];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) wsum[warp] = sum;
  __syncthreads();
  unsigned before = 0, total = 0;
  for (int v = 0; v < kWarpsF; v++) {
    if (v < warp) before += wsum[v];
    total += wsum[v];
  }
  if (threadIdx.x == 0 && total < need) set_status(status, SKV_DEV_COUNT);
  if (before < need && before + wsum[warp] >= need) {  // warp-uniform
    unsigned run = before;
    for (int r = r0; r < r0 + span && r < nb; r += 32) {
      const int rr = r + lane;
      const unsigned cnt = rr < nb && rr < r0 + span ? h[nb - 1 - rr] : 0u;
      unsigned incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (run + incl - cnt < need && run + incl >= need) {
        *digit = static_cast<uint32_t>(nb - 1 - rr);
        *above_out = run + incl - cnt;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      if (run >= need) break;
    }
  }
  __syncthreads();
}

template <int MODE, int LPT>
__global__ __launch_bounds__(kThreads, 2) void score_select_kernel(Args a, Ws w) {
  extern __shared__ __align__(16) uint32_t skey[];
  __shared__ __align__(16) uint32_t hist[kBins];
  __shared__ int wgt[kWarpsF], weq[kWarpsF];
  __shared__ unsigned red_a[kWarpsF];
  __shared__ uint32_t s_digit, s_above, s_top;
  __shared__ int s_before[2];
  __shared__ int s_ok;

  __shared__ __align__(16) int8_t s_q8[512];
  __shared__ float s_red[kWarpsF];
  allow_dependent_launch();  // the attention that follows may set up meanwhile
  const int b = blockIdx.y, c = blockIdx.x, C = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool pooled = MODE == SKV_SCORE_POOLED_BF16;
  const int ratio = pooled ? a.ratio : 1;
  int64_t T = a.lengths[b];
  const int64_t cap = pooled ? a.n_cap * ratio : a.n_cap;
  if (T > cap) {
    if (threadIdx.x == 0 && c == 0) set_status(a.status, SKV_DEV_RANGE);
    T = cap;
  }
  if (T < 0) T = 0;
  int32_t* out = a.idx + static_cast<int64_t>(b) * a.max_rows;
  const bool prepared = MODE == SKV_SCORE_SKETCH_INT4 && a.prep.q != nullptr;
  unsigned* arrive = w.bar(b);
  unsigned nbar = 0;
  if (prepared)  // before the dense shortcut: the append and q8 happen either way
    prepare_in_cta(a.prep, b, c, a.n_cap, T, a.S, a.W, reinterpret_cast<float*>(hist), s_q8, s_red, a.status);
  const bool dense = pooled ? T <= static_cast<int64_t>(ratio) * a.k + ratio - 1
                            : T <= static_cast<int64_t>(a.S) + a.W + a.k;
  if (dense) {  // every token; the same decision in every CTA of the request
    for (int64_t i = static_cast<int64_t>(c) * blockDim.x + threadIdx.x; i < T;
         i += static_cast<int64_t>(C) * blockDim.x)
      out[i] = static_cast<int32_t>(i);
    if (c == 0 && threadIdx.x == 0) a.count[b] = static_cast<int32_t>(T);
    return;
  }
  // The request's launch epoch: bumped by the last CTA of each launch, so
  // every CTA of this launch reads the same value.  Its tag marks the words
  // of this launch's final records.
  const unsigned epoch = __ldcg(w.rng(b) + 1);
  const unsigned tag = (epoch % 65535u + 1u) << 16;
  const int64_t lo = pooled ? 0 : a.S;
  const int64_t hi = pooled ? T / ratio : T - a.W;
  const int64_t chunk = (hi - lo + C - 1) / C;
  int64_t c0 = lo + c * chunk;
  if (c0 > hi) c0 = hi;
  const int64_t c1 = c0 + chunk < hi ? c0 + chunk : hi;
  const int len = static_cast<int>(c1 - c0);

  // ---- 1. scores of the chunk into shared memory -----------------------------------
  // rel = key - base fits `bits` bits: int32 sketch scores are bounded
  // (|s| < 2^20), so 21 bits above a fixed base; fp32 order keys take all 32.
  // int32 keys: the first radix pass (the top kMaxDigit bits) is counted
  // during the scan.  (fp32 keys crowd into a few bins of that pass, and the
  // contended atomics would slow the scan; they are counted after it.)
  const uint32_t base = MODE == SKV_SCORE_SKETCH_INT4 ? kInt4Base : 0u;
  const int bits = MODE == SKV_SCORE_SKETCH_INT4 ? 21 : 32;
  constexpr bool count0 = MODE == SKV_SCORE_SKETCH_INT4;
  const int shift0 = bits - kMaxDigit;  // bits - kLastBits >= kMaxDigit in every mode
  for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0u;
  if (threadIdx.x == 0) s_top = 0u;
  __syncthreads();
  uint32_t* gk = a.okeys ? a.okeys + static_cast<int64_t>(b) * a.n_cap : nullptr;
  auto keep = [&](int64_t t, uint32_t key) {
    skey[t - c0] = key;
    if (gk) gk[t] = key;
    if (count0) atomicAdd(&hist[(key - base) >> shift0], 1u);
  };
  if (MODE == SKV_SCORE_SKETCH_INT4) {
    constexpr int width = LPT * 32;
    const int8_t* q8 = prepared ? s_q8 : static_cast<const int8_t*>(a.query) + static_cast<int64_t>(b) * width;
    const uint8_t* rows = static_cast<const uint8_t*>(a.keys) + static_cast<int64_t>(b) * a.n_cap * (width / 2);
    auto emit = [&](int64_t t, int32_t sc) { keep(t, order_key_i32(sc)); };
    if (LPT == 8)
      scan_int4_rows128(q8, rows, c0, c1, warp, kWarpsF, emit);
    else
      scan_int4<LPT>(q8, rows, c0, c1, emit);
  } else if (MODE == SKV_SCORE_POOLED_BF16) {
    scan_pooled(static_cast<const uint16_t*>(a.query) + static_cast<int64_t>(b) * 128,
                static_cast<const uint16_t*>(a.keys) + static_cast<int64_t>(b) * a.n_cap * 128, c0, c1,
                [&](int64_t t, float sc) {
                  if (isnan(sc)) set_status(a.status, SKV_DEV_NAN);
                  keep(t, order_key_f32(sc));
                });
  } else {
    scan_f32(static_cast<const float*>(a.query) + static_cast<int64_t>(b) * a.width,
             static_cast<const float*>(a.keys) + static_cast<int64_t>(b) * a.n_cap * a.width, a.width, c0, c1,
             [&](int64_t t, float sc) {
               if (isnan(sc)) set_status(a.status, SKV_DEV_NAN);
               keep(t, order_key_f32(sc));
             });
  }
  __syncthreads();

  // ---- 2. non-final radix passes ---------------------------------------------------
  // int32 keys: one (13 bits, windowed); fp32 keys: two (13 windowed, 11).
  uint32_t need = static_cast<uint32_t>(a.k);
  uint32_t P = 0;         // rel >> rem of the keys still in play
  uint32_t n_match = kUnknown;  // the request's keys matching P
  int rem = bits;
  const int wlast = bits < kLastBits ? bits : kLastBits;
  int pass = 0;
  while (rem > wlast) {
    const int wb = rem - wlast < kMaxDigit ? rem - wlast : kMaxDigit;
    const int shift = rem - wb;
    const int nb = 1 << wb;
    if (pass > 0 || !count0) {
      if (pass > 0) {
        for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
      }
      for (int i = threadIdx.x; i < len; i += blockDim.x) {
        const uint32_t rel = skey[i] - base;
        if (top_bits(rel, rem) == P) atomicAdd(&hist[(rel >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
      }
      __syncthreads();
    }
    unsigned* gh = w.hist(pass, b);
    // First pass: the request's highest occupied bin is published too, so that
    // only a window of bins below it has to be read back.
    const bool windowed = pass == 0;
    unsigned top_local = 0u;
    for (int i = threadIdx.x; i < nb; i += blockDim.x)
      if (hist[i]) {
        atomicAdd(&gh[i], hist[i]);
        top_local = max(top_local, static_cast<unsigned>(i) + 1u);
      }
    if (windowed) {  // one global atomic per CTA
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) top_local = max(top_local, __shfl_xor_sync(0xffffffffu, top_local, o));
      if (lane == 0 && top_local) atomicMax(&s_top, top_local);
      __syncthreads();
      if (threadIdx.x == 0 && s_top) atomicMax(w.rng(b), s_top);  // bin + 1 (0: none)
    }
    // The request's highest bin is rarely far above this CTA's own: the first
    // window is read around the local top, in the same round trip as the
    // request's top, and kept when it covers that top and `need` keys.
    const int guess_hi = windowed && s_top ? min(nb - 1, static_cast<int>(s_top) - 1 + kAhead) : -1;
    req_barrier(arrive, ++nbar * C, a.status);
    if (windowed) {
      unsigned need_rem = need, above_acc = 0u;
      uint32_t dig = 0u, abv = 0u;
      bool found = false;
      const int g_lo = guess_hi >= kWin - 1 ? guess_hi - (kWin - 1) : 0;
      const int g_n = guess_hi - g_lo + 1;  // 0 without a guess
      const unsigned gtop = __ldcg(w.rng(b));
      {
        unsigned v[kWin / kThreads];
#pragma unroll
        for (int j = 0; j < kWin / kThreads; j++) {
          const int i = threadIdx.x + j * kThreads;
          v[j] = i < g_n ? __ldcg(&gh[g_lo + i]) : 0u;
        }
        unsigned part = 0u;
#pragma unroll
        for (int j = 0; j < kWin / kThreads; j++) {
          const int i = threadIdx.x + j * kThreads;
          if (i < g_n) hist[i] = v[j];
          part += v[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red_a[warp] = part;
        __syncthreads();
        unsigned total = 0u;
        for (int v2 = 0; v2 < kWarpsF; v2++) total += red_a[v2];
        if (g_n > 0 && static_cast<int>(gtop) - 1 <= guess_hi && total >= need_rem) {  // the same in every thread
          find_digit(hist, g_n, need_rem, &s_digit, &s_above, a.status);
          dig = s_digit + static_cast<uint32_t>(g_lo);
          abv = s_above;
          n_match = hist[s_digit];
          found = true;
        }
        __syncthreads();  // hist and red_a are rewritten below
      }
      // Otherwise windows of kWin bins from the request's top down until
      // `need` keys are covered.
      int hi = found ? -1 : static_cast<int>(gtop) - 1;  // highest occupied bin
      while (hi >= 0) {
        const int lo_bin = hi >= kWin - 1 ? hi - (kWin - 1) : 0;
        const int nw = hi - lo_bin + 1;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) hist[i] = __ldcg(&gh[lo_bin + i]);
        __syncthreads();
        unsigned part = 0u;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) part += hist[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red_a[warp] = part;
        __syncthreads();
        unsigned total = 0u;
        for (int v = 0; v < kWarpsF; v++) total += red_a[v];
        if (total >= need_rem) {  // the same decision in every thread
          find_digit(hist, nw, need_rem, &s_digit, &s_above, a.status);
          dig = s_digit + static_cast<uint32_t>(lo_bin);
          abv = s_above + above_acc;
          n_match = hist[s_digit];
          found = true;
          break;
        }
        __syncthreads();  // hist and red_a are rewritten by the next window
        need_rem -= total;
        above_acc += total;
        hi = lo_bin - 1;
      }
      if (!found && threadIdx.x == 0) set_status(a.status, SKV_DEV_COUNT);  // fewer keys than k: not sparse
      __syncthreads();
      P = (P << wb) | dig;
      need -= abv;
      rem = shift;
      pass++;
      continue;
    }
    {  // all loads in flight together: 16-byte pieces, unrolled
      const uint4* g4 = reinterpret_cast<const uint4*>(gh);
      uint4* h4 = reinterpret_cast<uint4*>(hist);
      const int n4 = nb / 4;  // nb >= 4 here: a non-final pass has at least 3 bits... or 1 bin group
      constexpr int kPer = kBins / 4 / kThreads;
      uint4 v[kPer];
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int i = threadIdx.x + j * kThreads;
        v[j] = i < n4 ? __ldcg(&g4[i]) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < kPer; j++) {
        const int i = threadIdx.x + j * kThreads;
        if (i < n4) h4[i] = v[j];
      }
      for (int i = 4 * n4 + threadIdx.x; i < nb; i += blockDim.x) hist[i] = __ldcg(&gh[i]);
    }
    __syncthreads();
    find_digit(hist, nb, need, &s_digit, &s_above, a.status);
    n_match = hist[s_digit];
    __syncthreads();  // every thread has read the bin before the next pass clears hist
    P = (P << wb) | s_digit;
    need -= s_above;
    rem = shift;
    pass++;
  }

  // ---- 3. final pass: K*, ties, and this CTA's offsets ------------------------------
  // The request-wide bins of the last digit go to global memory by atomics.
  // Each CTA also publishes suffix counts rec[d] = (its keys above the prefix)
  // + (its keys in bins >= d), d = 0..nbf, so that a later CTA gets the keys
  // above K* and equal to K* of every earlier chunk from two words each.
  // Each warp histograms its own contiguous piece of the chunk (the piece it
  // writes the picks of in step 4), so that once K* is known its counts of
  // keys above and equal to K* come from its bins, without another pass over
  // the keys; the CTA's bins are the warps' summed.
  constexpr int nbf = kLastBins;  // wlast == kLastBits: bits >= 21 in every mode
  uint32_t* whist = hist + nbf;   // [kWarpsF][nbf]
  static_assert(nbf * (kWarpsF + 1) <= kBins, "per-warp bins fit in the histogram buffer");
  for (int i = threadIdx.x; i < nbf * (kWarpsF + 1); i += blockDim.x) hist[i] = 0u;
  __syncthreads();
  const int sub = ((len + kWarpsF - 1) / kWarpsF + 31) / 32 * 32;  // warp v owns [v*sub, (v+1)*sub)
  const int p0 = min(len, warp * sub), p1 = min(len, p0 + sub);
  uint32_t* myh = whist + warp * nbf;
  // Four keys per lane per step: the tail of the launch runs every warp of
  // the SM at once, so instructions per key count.
  unsigned above_local = 0u;
  for (int i0 = p0; i0 < p1; i0 += 128) {
    const int i = i0 + 4 * lane;
    uint32_t k4[4];
    if (i + 3 < p1) {
      const uint4 v = *reinterpret_cast<const uint4*>(&skey[i]);
      k4[0] = v.x;
      k4[1] = v.y;
      k4[2] = v.z;
      k4[3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; j++) k4[j] = i + j < p1 ? skey[i + j] : base;
    }
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const uint32_t rel = k4[j] - base;
      const uint32_t t = rel >> wlast;
      if (t == P && i + j < p1)
        atomicAdd(&myh[rel & static_cast<uint32_t>(nbf - 1)], 1u);
      else if (t > P)
        above_local++;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) above_local += __shfl_xor_sync(0xffffffffu, above_local, o);
  if (lane == 0) wgt[warp] = static_cast<int>(above_local);
  __syncthreads();
  for (int d = threadIdx.x; d < nbf; d += blockDim.x) {
    unsigned sum = 0u;
#pragma unroll
    for (int v = 0; v < kWarpsF; v++) sum += whist[v * nbf + d];
    hist[d] = sum;
  }
  if (threadIdx.x == 0) {
    unsigned tot = 0u;
    for (int v = 0; v < kWarpsF; v++) tot += static_cast<unsigned>(wgt[v]);
    s_above = tot;
  }
  __syncthreads();
  unsigned* gf = w.fhist(b);
  int* myfin = w.fin(b, c);
  for (int i = threadIdx.x; i < nbf; i += blockDim.x)
    if (hist[i]) atomicAdd(&gf[i], hist[i]);
  if (warp == 0) {  // lane l owns bins [8l, 8l + 8); suffix sums from the top
    constexpr int kPerLane = nbf / 32;
    unsigned v[kPerLane], own = 0u;
#pragma unroll
    for (int j = 0; j < kPerLane; j++) {
      v[j] = hist[kPerLane * lane + j];
      own += v[j];
    }
    unsigned suf = own;  // sum over lanes >= l
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    unsigned acc = s_above + suf - own;
#pragma unroll
    for (int j = kPerLane - 1; j >= 0; j--) {
      acc += v[j];
      myfin[kPerLane * lane + j] = static_cast<int>(tag | acc);
    }
    if (lane == 0) myfin[nbf] = static_cast<int>(tag | s_above);
  }
  // Arrive, then poll the request's final bins with the arrival count: the
  // bins are complete once they sum to the request's keys matching P (they
  // only grow).  No release fence: the records the CTAs read next carry the
  // epoch tag in every word and are checked word by word.
  __syncthreads();
  if (warp == 0) {
    const unsigned target = ++nbar * C;
    if (lane == 0) asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(arrive) : "memory");
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    bool ok = false;
    for (long it = 0; it < kSpinLimit; it++) {
      unsigned arr = 0u;
      if (lane == 0) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(arr) : "l"(arrive) : "memory");
      v0 = ld_relaxed_v4(gf + 8 * lane);
      v1 = ld_relaxed_v4(gf + 8 * lane + 4);
      unsigned sum = v0.x + v0.y + v0.z + v0.w + v1.x + v1.y + v1.z + v1.w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      arr = __shfl_sync(0xffffffffu, arr, 0);
      if (arr >= target && (n_match == kUnknown || sum == n_match)) {
        ok = true;
        break;
      }
      if (it > 64) __nanosleep(32);
    }
    if (n_match == kUnknown) {
      v0 = ld_relaxed_v4(gf + 8 * lane);
      v1 = ld_relaxed_v4(gf + 8 * lane + 4);
    }
    reinterpret_cast<uint4*>(hist)[2 * lane] = v0;
    reinterpret_cast<uint4*>(hist)[2 * lane + 1] = v1;
    if (lane == 0) {
      s_ok = ok;
      if (!ok) set_status(a.status, SKV_DEV_TIMEOUT);
    }
  }
  __syncthreads();
  // Every CTA has read the non-final bins by now (each did before it
  // arrived): each clears its share of them.
  if (s_ok) {
    const int share = (kBins + C - 1) / C;
    const int i0 = c * share, i1 = min(kBins, i0 + share);
    for (int p = 0; p < pass; p++)
      for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) w.hist(p, b)[i] = 0u;
  }
  find_digit(hist, nbf, need, &s_digit, &s_above, a.status);
  const uint32_t dstar = s_digit;
  const uint32_t need_eq = need - s_above;  // keys equal to K* that are taken (lowest index first)
  const uint32_t kstar = base + ((P << wlast) | dstar);
  // keys of the chunks before this one: above K*, and equal to K*
  int gb = 0, eb = 0;
  for (int cc = threadIdx.x; cc < c; cc += blockDim.x) {
    const unsigned* rf = reinterpret_cast<const unsigned*>(w.fin(b, cc));
    unsigned x1 = 0u, x0 = 0u;
    for (long it = 0;; it++) {  // both words from this launch (bounded poll)
      x1 = ld_relaxed_u32(&rf[dstar + 1]);
      x0 = ld_relaxed_u32(&rf[dstar]);
      if ((x1 & 0xffff0000u) == tag && (x0 & 0xffff0000u) == tag) break;
      if (it >= kSpinLimit) {
        set_status(a.status, SKV_DEV_TIMEOUT);
        break;
      }
      if (it > 64) __nanosleep(32);
    }
    const int above_d = static_cast<int>(x1 & 0xffffu);
    gb += above_d;
    eb += static_cast<int>(x0 & 0xffffu) - above_d;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gb += __shfl_xor_sync(0xffffffffu, gb, o);
    eb += __shfl_xor_sync(0xffffffffu, eb, o);
  }
  if (threadIdx.x == 0) s_before[0] = s_before[1] = 0;
  __syncthreads();
  if (lane == 0 && (gb || eb)) {
    atomicAdd(&s_before[0], gb);
    atomicAdd(&s_before[1], eb);
  }
  // This CTA is done with everything the request's CTAs published: it takes
  // an exit ticket now and reads it at the end, where the last CTA clears
  // the window cells, the final bins and the counters, so the workspace is
  // ready for the next launch.
  unsigned ticket = 0u;
  __syncthreads();
  if (threadIdx.x == 0) {  // the high half counts CTAs whose final poll ran out
    __threadfence();
    ticket = atomicAdd(w.bar(b) + 1, s_ok ? 1u : 0x10001u);
  }

  // ---- 4. this CTA's picks, in ascending index order ---------------------------------
  // Warp v owns the contiguous piece [v*sub, (v+1)*sub) of the chunk; its
  // keys above K* are those above the prefix plus those in its bins above
  // d*, its keys equal to K* those in bin d*.
  {
    int ngt = 0;
#pragma unroll
    for (int j = 0; j < nbf / 32; j++) {
      const int d = lane * (nbf / 32) + j;
      if (d > static_cast<int>(dstar)) ngt += static_cast<int>(myh[d]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
    const int neq = static_cast<int>(myh[dstar]);
    __syncwarp();
    if (lane == 0) {
      wgt[warp] += ngt;  // keys above the prefix were counted in the final pass
      weq[warp] = neq;
    }
  }
  __syncthreads();
  const int needi = static_cast<int>(need_eq);
  int eq_run = s_before[1];  // equal keys before this warp's piece
  int pos = s_before[0] + min(s_before[1], needi);
  for (int v = 0; v < warp; v++) {
    pos += wgt[v] + max(0, min(weq[v], needi - eq_run));
    eq_run += weq[v];
  }
  const unsigned lt = (1u << lane) - 1u;
  const int head = pooled ? 0 : a.S;
  for (int bb = p0; bb < p1; bb += 32) {
    const int i = bb + lane;
    const uint32_t key = i < p1 ? skey[i] : 0u;
    // most blocks of 32 keys hold no key >= K*: one vote skips them
    if (!__any_sync(0xffffffffu, i < p1 && key >= kstar)) continue;
    const bool gt = i < p1 && key > kstar;
    const bool eq = i < p1 && key == kstar;
    const unsigned eqb = __ballot_sync(0xffffffffu, eq);
    const int eq_rank = eq_run + __popc(eqb & lt);
    const bool sel = gt || (eq && eq_rank < needi);
    const unsigned selb = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int j = pos + __popc(selb & lt);
      const int64_t t = c0 + i;
      if (j < a.k) {
        for (int u = 0; u < ratio; u++) out[head + ratio * j + u] = static_cast<int32_t>(ratio * t + u);
      } else {
        set_status(a.status, SKV_DEV_COUNT);
      }
    }
    eq_run += __popc(eqb);
    pos += __popc(selb);
  }
  if (c == 0) {
    if (!pooled) {
      for (int i = threadIdx.x; i < a.S; i += blockDim.x) out[i] = i;
      for (int i = threadIdx.x; i < a.W; i += blockDim.x) out[a.S + a.k + i] = static_cast<int32_t>(T - a.W + i);
      if (threadIdx.x == 0) a.count[b] = a.S + a.k + a.W;
    } else {
      const int64_t nbk = T / ratio;
      const int rem_tok = static_cast<int>(T - nbk * ratio);
      for (int i = threadIdx.x; i < rem_tok; i += blockDim.x)
        out[ratio * a.k + i] = static_cast<int32_t>(nbk * ratio + i);
      if (threadIdx.x == 0) a.count[b] = ratio * a.k + rem_tok;
    }
  }
  __shared__ int s_last;
  if (threadIdx.x == 0)
    s_last = (ticket & 0xffffu) != static_cast<unsigned>(C - 1) ? 0 : (ticket >> 16) == 0u && s_ok ? 1 : 2;
  __syncthreads();
  if (s_last) {
    __threadfence();
    // after a poll that ran out the shares above may have been cleared early
    if (s_last == 2)
      for (int p = 0; p < pass; p++)
        for (int i = threadIdx.x; i < kBins; i += blockDim.x) w.hist(p, b)[i] = 0u;
    for (int i = threadIdx.x; i < kLastBins; i += blockDim.x) w.fhist(b)[i] = 0u;
    // Tags repeat every 65,535 launches: when the next launch starts a new
    // cycle, every record of the request is cleared, so that a record last
    // written a whole cycle ago (a slot a smaller grid left unused) cannot
    // pass for one of the next launch.
    if ((epoch + 1u) % 65535u == 0u)
      for (int i = threadIdx.x; i < kCMax * kFin; i += blockDim.x) w.fin(b, 0)[i] = 0;
    if (threadIdx.x == 0) {
      w.rng(b)[0] = 0u;
      w.rng(b)[1] = epoch + 1u;
      w.bar(b)[0] = 0u;
      w.bar(b)[1] = 0u;
    }
  }
}

// CTAs per request of the largest grid whose CTAs are all resident at once
// (two per SM if they fit), with the shared memory each needs; 0 when B
// requests do not fit (too many requests, or a chunk too large for on-chip
// keys).
template <int MODE, int LPT>
int plan_grid(int B, int64_t n_cap, size_t* smem) {
  auto kernel = score_select_kernel<MODE, LPT>;
  static std::atomic<int> configured[kMaxDevices];
  if (smem_limit_once(configured, kernel, kKeyBudget) != SKV_OK) return 0;
  for (int per_sm_try = 2; per_sm_try >= 1; per_sm_try--) {
    const int c_try = per_sm_try * sm_count() / B;
    if (c_try < 1) continue;
    const int c_use = c_try > kCMax ? kCMax : c_try;
    const size_t need = static_cast<size_t>((n_cap + c_use - 1) / c_use) * sizeof(uint32_t);
    int fit = 0;
    if (need > kKeyBudget ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kernel, kThreads, need) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (fit >= per_sm_try) {
      *smem = need;
      return c_use;
    }
  }
  return 0;
}

template <int MODE, int LPT>
int launch(const Args& a, Ws w, cudaStream_t st) {
  auto kernel = score_select_kernel<MODE, LPT>;
  size_t smem = 0;
  const int C = plan_grid<MODE, LPT>(a.B, a.n_cap, &smem);
  if (C < 1) return SKV_EUNSUPPORTED;  // too many requests, or a chunk too large for on-chip keys
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.B, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, a, w) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  return SKV_OK;
}

}  // namespace

// Whether skv_score_select runs as one launch for these shapes (int4 sketch
// scores of the given width); otherwise it returns SKV_EUNSUPPORTED.
bool score_select_fits_int4(int width, int B, int64_t n_cap) {
  size_t smem = 0;
  if (B < 1) return false;
  if (width == 128) return plan_grid<SKV_SCORE_SKETCH_INT4, 4>(B, n_cap, &smem) > 0;
  if (width == 256) return plan_grid<SKV_SCORE_SKETCH_INT4, 8>(B, n_cap, &smem) > 0;
  if (width == 512) return plan_grid<SKV_SCORE_SKETCH_INT4, 16>(B, n_cap, &smem) > 0;
  return false;
}

}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_score_select_workspace_size(int B) { return B > 0 ? ws_bytes(B) : 0; }

SKV_EXPORT int skv_score_select(int mode, int B, int width, const void* query, const void* keys, int64_t n_cap,
                                const int32_t* lengths, int ratio, int k, int S, int W, int32_t* idx,
                                int max_rows, int32_t* count, uint32_t* order_keys, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (B < 0 || B > 65535 || n_cap < 0 || k < 1 || S < 0 || W < 0 || ratio < 1) return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (!query || !keys || !lengths || !idx || !count || !workspace) return SKV_EINVAL;
  if (!aligned16(keys) || !aligned16(query) || !aligned16(workspace)) return SKV_EINVAL;
  if (workspace_bytes < ws_bytes(B)) return SKV_ENOMEM;
  const bool pooled = mode == SKV_SCORE_POOLED_BF16;
  if (pooled ? (ratio > 64 || width != 128 || S != 0 || W != 0) : ratio != 1) return SKV_EINVAL;
  const int64_t need_rows = pooled ? static_cast<int64_t>(ratio) * k + ratio - 1 : static_cast<int64_t>(S) + k + W;
  if (max_rows < need_rows) return SKV_EINVAL;
  Args a{mode, width, query, keys, n_cap, lengths, ratio, k, S, W, idx, max_rows, count, order_keys, dev_status, B};
  Ws w = ws_carve(workspace, B);
  cudaStream_t st = as_stream(stream);
  switch (mode) {
    case SKV_SCORE_SKETCH_INT4:
      if (width == 128) return launch<SKV_SCORE_SKETCH_INT4, 4>(a, w, st);
      if (width == 256) return launch<SKV_SCORE_SKETCH_INT4, 8>(a, w, st);
      if (width == 512) return launch<SKV_SCORE_SKETCH_INT4, 16>(a, w, st);
      return SKV_EUNSUPPORTED;
    case SKV_SCORE_SKETCH_F32:
      if (width <= 0 || width % 4 || width > 1024) return SKV_EINVAL;
      return launch<SKV_SCORE_SKETCH_F32, 32>(a, w, st);
    case SKV_SCORE_POOLED_BF16:
      return launch<SKV_SCORE_POOLED_BF16, 16>(a, w, st);
    default:
      return SKV_EINVAL;
  }
}

SKV_EXPORT int skv_decode_select(int B, int Hq, int Hkv, int d, int r, const uint16_t* q, const uint16_t* new_k,
                                 const uint16_t* new_v, const float* basis, const float* c, const int64_t* new_rows,
                                 uint8_t* sketch, int8_t* k8, uint16_t* k_scale, int8_t* v8, uint16_t* v_scale,
                                 int64_t n_cap, const int32_t* lengths, int k, int S, int W, int32_t* idx,
                                 int max_rows, int32_t* count, int8_t* q8_out, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (B < 0 || B > 65535 || n_cap < 0 || k < 1 || S < 0 || W < 1) return SKV_EINVAL;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || r != fold::kRank || d <= 0 || d % 2) return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  const int width = Hkv * fold::kRank;
  if (width != 128 && width != 256 && width != 512) return SKV_EUNSUPPORTED;
  const size_t ns = (d + 31) / 32;
  if (d > 512 || d % 8 ||
      (Hkv + 2ull) * d + (Hkv + 1ull) * fold::kRank * ns + static_cast<size_t>(width) > kBins)
    return SKV_EUNSUPPORTED;
  if (!q || !new_k || !new_v || !basis || !c || !new_rows || !sketch || !k8 || !k_scale || !v8 || !v_scale ||
      !lengths || !idx || !count || !workspace)
    return SKV_EINVAL;
  if (!aligned16(sketch) || !aligned16(workspace)) return SKV_EINVAL;
  if (workspace_bytes < ws_bytes(B)) return SKV_ENOMEM;
  if (max_rows < static_cast<int64_t>(S) + k + W) return SKV_EINVAL;
  Args a{SKV_SCORE_SKETCH_INT4, width, nullptr, sketch, n_cap, lengths, 1, k, S, W, idx, max_rows, count,
         nullptr, dev_status, B};
  a.prep = Prep{q, new_k, new_v, basis, c, new_rows, sketch, k8, reinterpret_cast<__half*>(k_scale), v8,
                reinterpret_cast<__half*>(v_scale), q8_out, Hq, Hkv, d};
  Ws w = ws_carve(workspace, B);
  cudaStream_t st = as_stream(stream);
  if (width == 128) return launch<SKV_SCORE_SKETCH_INT4, 4>(a, w, st);
  if (width == 256) return launch<SKV_SCORE_SKETCH_INT4, 8>(a, w, st);
  return launch<SKV_SCORE_SKETCH_INT4, 16>(a, w, st);
}
