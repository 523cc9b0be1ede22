// resolve.cu -- a5: map the selected tokens to pool rows (host-tier resolvers)
// and the host-tier write path.
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": the main KV
// cache sits in host RAM as int4 (64-dim groups, fp16 scales, 272 B per
// token-head); the GPU keeps the sketch, the sinks, the recent tail and a 2.5%
// hot buffer managed by windowed CLOCK, and rows fetched from the host are
// dequantised back to int8 rows.
// [P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one block pool":
// resident tokens are read in place, hot tokens refresh their LRU entry, and a
// miss copies one row from pinned host memory into an LRU slot of the hot
// buffer ("What it composes with": the hot buffer holds 2 x top-K rows).
//
// Two launches per call.  First one CTA per request: the resolver state of
// the request is staged in shared memory, the hit pass runs over all threads,
// the sweep (CLOCK) or the victim order (LRU) is computed on chip, and the
// misses are listed.  Then a wide grid with one warp per miss reads the host
// rows with coalesced 16-byte loads, so that many SMs keep host reads in
// flight at once.
#include "common.cuh"

namespace skv {
namespace {

constexpr int kResThreads = 1024;
constexpr int kClockThreads = 512;
constexpr int kMaxTokBytes = 5120;  // host bytes of one token's row (all heads, K and V), CLOCK tier
constexpr int kMaxClockSlots = 16384;
constexpr int kMaxLruSlots = 8192;
constexpr int kMaxResolveRows = 8192;

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// The decode step lives in device memory so that a captured graph replays
// with a new step each time: every CTA reads step[0] at its start; the last
// CTA to finish (ticket step[1]) advances step[0] and resets the ticket.
__device__ __forceinline__ int32_t read_step(const int32_t* step) {
  return *reinterpret_cast<const volatile int32_t*>(step);
}

__device__ __forceinline__ void advance_step(int32_t* step) {
  __threadfence();
  if (atomicAdd(reinterpret_cast<unsigned*>(step + 1), 1u) == gridDim.x - 1) {
    __threadfence();
    step[0] = step[0] + 1;
    step[1] = 0;
    __threadfence();
  }
}

// ---------------------------------------------------------------------------
// Windowed CLOCK over the hot slots of one request.
// ---------------------------------------------------------------------------
struct ClockArgs {
  int64_t t_cap;
  const int32_t* lengths;
  int S, W, Hkv, d, Hs;
  const int32_t* idx;
  int max_rows;
  const int32_t* count;
  int32_t* step;  // [0] decode step, [1] ticket
  int32_t* slot_token;
  uint8_t* ref;
  int32_t* use_step;
  int32_t* token_slot;
  int32_t* hand;
  const uint8_t* host_rows;
  int8_t* k8;
  int8_t* v8;
  __half* k_scale;
  __half* v_scale;
  int64_t req_row_stride;
  int32_t* rows_out;
  int32_t* n_miss;
  int32_t* ws_tok;  // [B][max_rows] miss tokens
  int32_t* ws_row;  // [B][max_rows] their destination pool rows
  int32_t* status;
};

size_t clock_smem_bytes(int Hs, int max_rows) {
  return align16(static_cast<size_t>(Hs) * 9) + static_cast<size_t>(max_rows) * 12 + 64 * sizeof(int);
}

// int4 vector (128 B of codes for 256 dims per 136 B, fp16 group scales after
// the codes) -> int8 row + fp16 scale: x = code * s_g exactly in fp32,
// s8 = fp16(max|x| / 127), q = clamp(rint(x / s8), +-127).  One lane per
// 64-dim group; the ng lanes of a vector are consecutive.
// A code takes one of 16 values, so q is computed once per value and the
// codes are mapped through that table: max|x| = max|code| * s_g (exact),
// q(-c) = -q(c) (IEEE division, rounding to even and the clamp are
// symmetric), q(0) = 0, and q(-8) = -q(8).
__device__ __forceinline__ void requant_group(const uint2 (&c)[4], uint16_t sbits, int ng, int8_t* dst,
                                              __half* sdst, bool store) {
  const float sg = __half2float(__ushort_as_half(sbits));
  const uint32_t w[8] = {c[0].x, c[0].y, c[1].x, c[1].y, c[2].x, c[2].y, c[3].x, c[3].y};
  // largest |code|: per nibble, 8 - n for n >= 8 (code n - 16), else n
  int cmax = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) {
#pragma unroll
    for (int e = 0; e < 8; e++) {
      const int code = static_cast<int>(w[i] << (28 - 4 * e)) >> 28;
      cmax = max(cmax, code < 0 ? -code : code);
    }
  }
  // max_e |code_e * s_g| (a NaN product counts as 0, as fmaxf over the elements would have it)
  float amax = fmaxf(0.f, static_cast<float>(cmax) * fabsf(sg));
  for (int o = 1; o < ng; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const __half s8 = __float2half_rn(__fdiv_rn(amax, 127.f));
  const float sf = __half2float(s8);
  const bool ok = (sf != 0.f) && isfinite(sf);
  if (!store) return;
  // table bytes by nibble n: q(n) for n < 8, q(n - 16) = -q(16 - n) for n >= 8
  int qp[9];
  qp[0] = 0;
#pragma unroll
  for (int m = 1; m <= 8; m++)
    qp[m] = ok ? rint_clamp(__fdiv_rn(static_cast<float>(m) * sg, sf), -127, 127) : 0;
  auto byte_of = [](int v) { return static_cast<uint32_t>(v) & 0xffu; };
  const uint32_t t0 = byte_of(qp[0]) | (byte_of(qp[1]) << 8) | (byte_of(qp[2]) << 16) | (byte_of(qp[3]) << 24);
  const uint32_t t1 = byte_of(qp[4]) | (byte_of(qp[5]) << 8) | (byte_of(qp[6]) << 16) | (byte_of(qp[7]) << 24);
  const uint32_t t2 = byte_of(-qp[8]) | (byte_of(-qp[7]) << 8) | (byte_of(-qp[6]) << 16) | (byte_of(-qp[5]) << 24);
  const uint32_t t3 = byte_of(-qp[4]) | (byte_of(-qp[3]) << 8) | (byte_of(-qp[2]) << 16) | (byte_of(-qp[1]) << 24);
  // four nibbles held one per byte -> their four table bytes
  auto lookup = [&](uint32_t x) {
    const uint32_t sel = (x & 0x7u) | ((x >> 4) & 0x70u) | ((x >> 8) & 0x700u) | ((x >> 12) & 0x7000u);
    const uint32_t lo = prmt(t0, t1, sel), hi = prmt(t2, t3, sel);
    const uint32_t m = ((x & 0x08080808u) >> 3) * 0xffu;  // 0xff in the bytes whose nibble is >= 8
    return (lo & ~m) | (hi & m);
  };
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i2 = 0; i2 < 4; i2++) {
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 2; k++) {
      const uint32_t wi = w[2 * i2 + k];  // nibble e = dim 8 (2 i2 + k) + e
      const uint32_t ev = wi & 0x0f0f0f0fu, od = (wi >> 4) & 0x0f0f0f0fu;  // nibbles 0,2,4,6 and 1,3,5,7
      out[2 * k] = lookup(prmt(ev, od, 0x5140u));      // dims 0..3 of the word
      out[2 * k + 1] = lookup(prmt(ev, od, 0x7362u));  // dims 4..7
    }
    d4[i2] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  if (sdst) *sdst = s8;
}

__global__ __launch_bounds__(kClockThreads) void clock_kernel(ClockArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  allow_dependent_launch();  // the row fetch may be scheduled now; it waits for this grid to finish
  const int b = blockIdx.x, tid = threadIdx.x;
  const int Hs = a.Hs;
  int32_t* s_tok = reinterpret_cast<int32_t*>(smem);
  int32_t* s_use = s_tok + Hs;
  uint8_t* s_ref = reinterpret_cast<uint8_t*>(s_use + Hs);
  int32_t* m_tok = reinterpret_cast<int32_t*>(smem + align16(static_cast<size_t>(Hs) * 9));
  int32_t* m_pos = m_tok + a.max_rows;
  int32_t* m_slot = m_pos + a.max_rows;
  int* scr = reinterpret_cast<int*>(m_slot + a.max_rows);

  int64_t T = a.lengths[b];
  if (T < 0 || T > a.t_cap) {
    if (tid == 0) set_status(a.status, SKV_DEV_RANGE);
    T = T < 0 ? 0 : a.t_cap;
  }
  int n = a.count[b];
  if (n < 0 || n > a.max_rows) {
    if (tid == 0) set_status(a.status, SKV_DEV_COUNT);
    n = n < 0 ? 0 : a.max_rows;
  }
  const int32_t* idx = a.idx + static_cast<int64_t>(b) * a.max_rows;
  int32_t* rows = a.rows_out + static_cast<int64_t>(b) * a.max_rows;
  int32_t* tslot = a.token_slot + static_cast<int64_t>(b) * a.t_cap;
  const int64_t sbase = static_cast<int64_t>(b) * Hs;
  const int S = a.S, W = a.W;
  const int32_t step = read_step(a.step);
  auto is_pick = [&](int64_t t) { return t >= S && t < T - W; };

  // Thread tid owns the contiguous run of rows [tid*run, tid*run + run): its
  // tokens, then the slots of its picks, each round of loads issued together,
  // so that one block-wide scan orders the misses.
  constexpr int kRun = kMaxResolveRows / kClockThreads;
  const int run = (n + kClockThreads - 1) / kClockThreads;
  const int i0 = tid * run;
  int32_t tk[kRun], sk[kRun];
  int picks_local = 0;
#pragma unroll
  for (int k = 0; k < kRun; k++) {
    const int i = i0 + k;
    tk[k] = k < run && i < n ? idx[i] : -1;
  }
#pragma unroll
  for (int k = 0; k < kRun; k++) {
    const int64_t t = tk[k];
    const bool pk = k < run && i0 + k < n && t >= 0 && t < T && is_pick(t);
    picks_local += pk;
    sk[k] = pk ? tslot[t] : -1;
  }
  for (int s = tid; s < Hs; s += kClockThreads) {
    s_tok[s] = a.slot_token[sbase + s];
    s_use[s] = a.use_step[sbase + s];
    s_ref[s] = a.ref[sbase + s];
  }
  // The sweep needs at least as many slots as picks (else nothing changes).
  int n_picks;
  block_exclusive_scan(picks_local, scr, &n_picks);
  const bool fits = n_picks <= Hs;
  if (!fits && tid == 0) set_status(a.status, SKV_DEV_COUNT);
  __syncthreads();

  // Phase 1: sinks, tail and hits; misses listed in ascending token order.
  int miss_local = 0;
  uint32_t miss_bits = 0u;
#pragma unroll
  for (int k = 0; k < kRun; k++) {
    const int i = i0 + k;
    if (k >= run || i >= n) continue;
    const int64_t t = tk[k];
    if (t < 0 || t >= T) {
      set_status(a.status, SKV_DEV_RANGE);
      rows[i] = -1;
    } else if (t < S) {
      rows[i] = static_cast<int32_t>(t);
    } else if (t >= T - W) {
      rows[i] = static_cast<int32_t>(S + t % W);
    } else if (!fits) {
      rows[i] = -1;
    } else {
      const int32_t s = sk[k];
      if (s >= 0 && s < Hs) {
        s_ref[s] = 1;
        s_use[s] = step;
        rows[i] = S + W + s;
      } else {
        if (s >= Hs) set_status(a.status, SKV_DEV_RANGE);
        rows[i] = -1;
        miss_bits |= 1u << k;
        miss_local++;
      }
    }
  }
  int nm;
  int mo = block_exclusive_scan(miss_local, scr, &nm);
#pragma unroll
  for (int k = 0; k < kRun; k++) {
    if (miss_bits & (1u << k)) {
      m_tok[mo] = tk[k];
      m_pos[mo] = i0 + k;
      m_slot[mo] = -1;
      mo++;
    }
  }
  __syncthreads();

  // Phase 2: the hand sweeps windows of up to 512 slots, all threads at once.
  // Visiting slots in order from the hand, the one-slot-at-a-time CLOCK skips
  // slots used in this step, takes slots that are empty or have ref == 0 (one
  // per remaining miss), and clears the ref bit of the others; so within a
  // window the first m candidates are taken (m = misses left), the ref bits
  // of the non-candidates before the last taken slot are cleared, and the
  // hand stops after it.  A window without enough candidates takes all of
  // them, clears every ref bit it passes and hands over to the next window.
  if (nm > 0) {
    __shared__ int s_hand, s_last;
    int h = a.hand[b];
    if (h < 0 || h >= Hs) {
      if (tid == 0) set_status(a.status, SKV_DEV_RANGE);
      h = 0;
    }
    const int win = Hs < kClockThreads ? Hs : kClockThreads;
    const int64_t limit = 3 * static_cast<int64_t>(Hs) + 2 * kClockThreads;  // two turns always suffice
    int64_t moved = 0;
    int j = 0;  // misses placed so far (the same in every thread)
    while (j < nm) {
      if (moved > limit) {
        if (tid == 0) set_status(a.status, SKV_DEV_COUNT);
        break;
      }
      const bool act = tid < win;
      int s = h + tid;
      if (s >= Hs) s -= Hs;
      const bool used = act && s_use[s] == step;
      const int32_t st = act ? s_tok[s] : 0;
      const bool cand = act && !used && (st < 0 || s_ref[s] == 0);
      int total;
      const int rank = block_exclusive_scan(cand ? 1 : 0, scr, &total);
      const int need = nm - j;
      // position of the last slot the hand visits in this window
      if (tid == 0) s_last = win - 1;
      __syncthreads();
      if (total >= need && cand && rank == need - 1) s_last = tid;
      __syncthreads();
      const int last = s_last;
      if (act && tid <= last) {
        if (cand && rank < need) {
          const int jj = j + rank;
          const int32_t tok = m_tok[jj];
          if (st >= 0 && st < a.t_cap) tslot[st] = -1;
          s_tok[s] = tok;
          tslot[tok] = s;
          s_ref[s] = 1;
          s_use[s] = step;
          m_slot[jj] = s;
          rows[m_pos[jj]] = S + W + s;
        } else if (!used && !cand) {
          s_ref[s] = 0;
        }
      }
      j += total < need ? total : need;
      h += last + 1;
      if (h >= Hs) h -= Hs;
      moved += last + 1;
      __syncthreads();  // the window's state changes are visible to the next window
    }
    if (tid == 0) s_hand = h;
    __syncthreads();
    if (tid == 0) a.hand[b] = s_hand;
  }
  __syncthreads();

  // Phase 3: the miss list for the fetch kernel (token, destination pool row).
  for (int j = tid; j < nm; j += kClockThreads) {
    a.ws_tok[static_cast<int64_t>(b) * a.max_rows + j] = m_tok[j];
    a.ws_row[static_cast<int64_t>(b) * a.max_rows + j] =
        m_slot[j] >= 0 ? static_cast<int32_t>(static_cast<int64_t>(b) * a.req_row_stride + S + W + m_slot[j]) : -1;
  }

  // Phase 4: state back to global memory.
  for (int s = tid; s < Hs; s += kClockThreads) {
    a.slot_token[sbase + s] = s_tok[s];
    a.use_step[sbase + s] = s_use[s];
    a.ref[sbase + s] = s_ref[s];
  }
  if (tid == 0) a.n_miss[b] = fits ? nm : -1;
  __syncthreads();
  if (tid == 0) advance_step(a.step);
}

// One warp per miss: the token's host row (Hkv heads x [K | V] int4 vectors,
// contiguous) is read with coalesced 16-byte loads into shared memory, then
// each lane requantises one 64-dim group to int8 and writes it to the pool.
// A lane issues all its loads of the row before it stores any (a host read
// takes microseconds, so the round trips must overlap, not follow each other).
constexpr int kFetchWarps = 8;
constexpr int kFetchPieces = 8;  // 16-byte pieces per lane and row held in registers (rows up to 4 KB)

__global__ __launch_bounds__(32 * kFetchWarps, 3) void fetch_int4_kernel(
    const int32_t* __restrict__ ws_tok, const int32_t* __restrict__ ws_row, const int32_t* __restrict__ n_miss,
    int max_rows, int64_t t_cap, int Hkv, int d, const uint8_t* __restrict__ host_rows, int8_t* __restrict__ k8,
    int8_t* __restrict__ v8, __half* __restrict__ k_scale, __half* __restrict__ v_scale) {
  extern __shared__ __align__(16) unsigned char stage_all[];
  grid_dependency_wait();  // launched early: the state pass's miss list is complete from here on
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * kFetchWarps + warp;
  const int nm = n_miss[b];
  if (j >= nm) return;  // also nm == -1
  const int64_t row = ws_row[static_cast<int64_t>(b) * max_rows + j];
  if (row < 0) return;
  const int32_t tok = ws_tok[static_cast<int64_t>(b) * max_rows + j];
  const int ng = d / 64, rb = d / 2 + 2 * ng, tasks = 2 * Hkv * ng;
  const int tb = 2 * Hkv * rb;
  unsigned char* stage = stage_all + warp * tb;
  const uint4* src = reinterpret_cast<const uint4*>(host_rows + (static_cast<int64_t>(b) * t_cap + tok) * tb);
  const int np = tb / 16;  // 17 d / 16 bytes per vector: a whole number of pieces for d % 256 == 0
  uint4 v[kFetchPieces];
#pragma unroll
  for (int u = 0; u < kFetchPieces; u++)
    if (lane + 32 * u < np) v[u] = ld_nc16(src + lane + 32 * u);
#pragma unroll
  for (int u = 0; u < kFetchPieces; u++)
    if (lane + 32 * u < np) reinterpret_cast<uint4*>(stage)[lane + 32 * u] = v[u];
  for (int c = lane + 32 * kFetchPieces; c < np; c += 32) reinterpret_cast<uint4*>(stage)[c] = ld_nc16(src + c);
  __syncwarp();
  for (int it = 0; it * 32 < tasks; it++) {
    const int task = it * 32 + lane;
    const bool live = task < tasks;
    const int v = live ? task / ng : 0, g = live ? task % ng : 0;
    const unsigned char* vec = stage + v * rb;
    uint2 c[4];
#pragma unroll
    for (int q = 0; q < 4; q++) c[q] = reinterpret_cast<const uint2*>(vec + 32 * g)[q];
    const uint16_t sb = *reinterpret_cast<const uint16_t*>(vec + d / 2 + 2 * g);
    const int hh = v >> 1;
    int8_t* dst = ((v & 1) ? v8 : k8) + (row * Hkv + hh) * d + 64 * g;
    __half* sdst = g == 0 ? ((v & 1) ? v_scale : k_scale) + row * Hkv + hh : nullptr;
    requant_group(c, sb, ng, dst, sdst, live);
  }
}

// One warp per kRowsPerWarp misses: plain row copy host -> pool, every load
// of the warp's rows (up to kFetchPieces / kRowsPerWarp pieces per lane and
// row) issued before the first store.
constexpr int kRowsPerWarp = 2;

__global__ __launch_bounds__(32 * kFetchWarps) void fetch_rows_kernel(
    const int32_t* __restrict__ ws_tok, const int32_t* __restrict__ ws_row, const int32_t* __restrict__ n_miss,
    int max_rows, int64_t t_cap, const uint8_t* __restrict__ host, uint8_t* __restrict__ pool, int64_t row_bytes) {
  grid_dependency_wait();  // launched early: the state pass's miss list is complete from here on
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = (blockIdx.x * kFetchWarps + warp) * kRowsPerWarp;
  const int nm = n_miss[b];
  if (j0 >= nm) return;
  const int chunks = static_cast<int>(row_bytes / 16);
  constexpr int kPer = kFetchPieces / kRowsPerWarp;
  const uint8_t* src[kRowsPerWarp];
  uint4* dst[kRowsPerWarp];
  bool live[kRowsPerWarp];  // a miss whose destination row is known (-1: nothing to write)
#pragma unroll
  for (int u = 0; u < kRowsPerWarp; u++) {
    const int j = j0 + u < nm ? j0 + u : j0;  // j0 < nm
    const int32_t tok = ws_tok[static_cast<int64_t>(b) * max_rows + j];
    const int64_t row = ws_row[static_cast<int64_t>(b) * max_rows + j];
    live[u] = j0 + u < nm && row >= 0;
    src[u] = host + (static_cast<int64_t>(b) * t_cap + tok) * row_bytes;
    dst[u] = reinterpret_cast<uint4*>(pool + (row >= 0 ? row : 0) * row_bytes);
  }
  uint4 v[kRowsPerWarp][kPer];
#pragma unroll
  for (int u = 0; u < kRowsPerWarp; u++)
#pragma unroll
    for (int q = 0; q < kPer; q++)
      if (live[u] && lane + 32 * q < chunks) v[u][q] = ld_nc16(src[u] + 16 * (lane + 32 * q));
#pragma unroll
  for (int u = 0; u < kRowsPerWarp; u++)
#pragma unroll
    for (int q = 0; q < kPer; q++)
      if (live[u] && lane + 32 * q < chunks) dst[u][lane + 32 * q] = v[u][q];
  for (int c = lane + 32 * kPer; c < chunks; c += 32)  // rows above kPer * 512 bytes
    for (int u = 0; u < kRowsPerWarp; u++)
      if (live[u]) dst[u][c] = ld_nc16(src[u] + 16 * c);
}

// ---------------------------------------------------------------------------
// LRU hot buffer behind a block table.
// ---------------------------------------------------------------------------
struct LruArgs {
  int64_t t_cap;
  const int32_t* lengths;
  int page;
  const int32_t* block_table;
  int64_t n_pages;
  int64_t hot_base, hot_stride;
  int n_slots;
  int32_t* step;  // [0] decode step, [1] ticket
  int64_t* stamp;
  int32_t* slot_token;
  int32_t* token_slot;
  int32_t* order;  // [B][n_slots]: the slots by ascending (stamp, slot)
  const uint8_t* host;
  uint8_t* pool;
  int64_t row_bytes, n_pool_rows;
  const int32_t* idx;
  int max_rows;
  const int32_t* count;
  int32_t* rows_out;
  int32_t* n_miss;
  int32_t* ws_tok;
  int32_t* ws_row;
  int32_t* status;
  // Leased hot pages ([P2]: a hot-buffer page is an ordinary block of the
  // pool): slot s of request b is row hot_blocks[b][s / page] * page + s % page.
  // NULL: the reserved region hot_base + b * hot_stride + s.
  const int32_t* hot_blocks;
  int n_hot_pages;
};

size_t lru_smem_bytes(int n_slots, int max_rows) {
  return static_cast<size_t>(n_slots) * 8 + static_cast<size_t>(n_slots) * 4 * 2 + static_cast<size_t>(max_rows) * 8 +
         64 * sizeof(int);
}

__global__ __launch_bounds__(kResThreads) void lru_kernel(LruArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  allow_dependent_launch();  // the row fetch may be scheduled now; it waits for this grid to finish
  const int b = blockIdx.x, tid = threadIdx.x;
  const int ns = a.n_slots;
  int64_t* s_stamp = reinterpret_cast<int64_t*>(smem);
  int32_t* s_order = reinterpret_cast<int32_t*>(s_stamp + ns);  // LRU order on entry
  int32_t* s_new = s_order + ns;                                // victim slots, then the new order
  int32_t* m_tok = s_new + ns;
  int32_t* m_pos = m_tok + a.max_rows;
  int* scr = reinterpret_cast<int*>(m_pos + a.max_rows);

  int64_t T = a.lengths[b];
  if (T < 0 || T > a.t_cap) {
    if (tid == 0) set_status(a.status, SKV_DEV_RANGE);
    T = T < 0 ? 0 : a.t_cap;
  }
  int n = a.count[b];
  if (n < 0 || n > a.max_rows) {
    if (tid == 0) set_status(a.status, SKV_DEV_COUNT);
    n = n < 0 ? 0 : a.max_rows;
  }
  const int32_t* idx = a.idx + static_cast<int64_t>(b) * a.max_rows;
  int32_t* rows = a.rows_out + static_cast<int64_t>(b) * a.max_rows;
  int32_t* tslot = a.token_slot + static_cast<int64_t>(b) * a.t_cap;
  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.n_pages;
  const int64_t sbase = static_cast<int64_t>(b) * ns;
  const int64_t hot = a.hot_base + static_cast<int64_t>(b) * a.hot_stride;
  const int32_t* hb = a.hot_blocks ? a.hot_blocks + static_cast<int64_t>(b) * a.n_hot_pages : nullptr;
  auto hot_row = [&](int s) -> int64_t {  // -1 when the leased page is missing or out of the pool
    if (!hb) return hot + s;
    const int64_t blk = hb[s / a.page];
    const int64_t row = blk * a.page + s % a.page;
    return blk < 0 || row >= a.n_pool_rows ? -1 : row;
  };
  const int64_t step = read_step(a.step);

  for (int s = tid; s < ns; s += kResThreads) s_stamp[s] = a.stamp[sbase + s];
  __syncthreads();

  // Phase 1: resident rows in place, hot hits refresh their stamp, misses
  // listed in ascending token order.
  int nm = 0;
  for (int base = 0; base < n; base += kResThreads) {
    const int i = base + tid;
    int miss = 0;
    int64_t t = -1;
    if (i < n) {
      t = idx[i];
      const int64_t p = t / a.page;
      if (t < 0 || t >= T || p >= a.n_pages) {
        set_status(a.status, SKV_DEV_RANGE);
        rows[i] = -1;
      } else if (bt[p] >= 0) {
        const int64_t row = static_cast<int64_t>(bt[p]) * a.page + t % a.page;
        if (row >= a.n_pool_rows) set_status(a.status, SKV_DEV_RANGE);
        rows[i] = row < a.n_pool_rows ? static_cast<int32_t>(row) : -1;
      } else {
        const int32_t s = tslot[t];
        if (s >= 0 && s < ns) {
          s_stamp[s] = step;
          const int64_t row = hot_row(s);
          if (row < 0) set_status(a.status, SKV_DEV_RANGE);
          rows[i] = static_cast<int32_t>(row);
        } else {
          if (s >= ns) set_status(a.status, SKV_DEV_RANGE);
          rows[i] = -1;
          miss = 1;
        }
      }
    }
    int tot;
    const int ex = block_exclusive_scan(miss, scr, &tot);
    if (miss) {
      m_tok[nm + ex] = static_cast<int32_t>(t);
      m_pos[nm + ex] = i;
    }
    nm += tot;
  }
  __syncthreads();

  // Phase 2: the victims are the first nm untouched slots of the LRU order
  // (ascending (stamp, slot)).  A block scan over the order ranks the
  // untouched slots; rank j < nm is the j-th victim.
  int32_t* order = a.order + sbase;
  for (int pos = tid; pos < ns; pos += kResThreads) {
    int32_t v = order[pos];
    if (v < 0 || v >= ns) {  // not a permutation of the slots: flag it and use the identity there
      set_status(a.status, SKV_DEV_RANGE);
      v = pos;
    }
    s_order[pos] = v;
  }
  __syncthreads();
  constexpr int kPer = 8;  // order positions per thread (n_slots <= 8192)
  int ucnt = 0;
  const int p0 = tid * kPer;
  for (int u = 0; u < kPer; u++) {
    const int pos = p0 + u;
    if (pos < ns && s_stamp[s_order[pos]] != step) ucnt++;
  }
  int n_untouched;
  int urank = block_exclusive_scan(ucnt, scr, &n_untouched);
  const bool ok = n_untouched >= nm;
  if (!ok && tid == 0) set_status(a.status, SKV_DEV_COUNT);
  if (ok && nm > 0) {
    // victims in LRU order; the untouched rest keeps its order at the front
    for (int u = 0; u < kPer; u++) {
      const int pos = p0 + u;
      if (pos < ns) {
        const int sl = s_order[pos];
        if (s_stamp[sl] != step) {
          if (urank < nm)
            s_new[urank] = sl;  // victim urank
          urank++;
        }
      }
    }
    __syncthreads();
    // Phase 3: the i-th miss takes the i-th victim.
    for (int j = tid; j < nm; j += kResThreads) {
      const int sl = s_new[j];
      const int32_t tok = m_tok[j];
      const int32_t old = a.slot_token[sbase + sl];
      if (old >= 0 && old < a.t_cap) tslot[old] = -1;
      a.slot_token[sbase + sl] = tok;
      tslot[tok] = sl;
      const int64_t row = hot_row(sl);  // -1: the fetch skips it
      if (row < 0) set_status(a.status, SKV_DEV_RANGE);
      rows[m_pos[j]] = static_cast<int32_t>(row);
      a.ws_tok[static_cast<int64_t>(b) * a.max_rows + j] = tok;  // the miss list for the fetch kernel
      a.ws_row[static_cast<int64_t>(b) * a.max_rows + j] = static_cast<int32_t>(row);
    }
    __syncthreads();
    for (int j = tid; j < nm; j += kResThreads) s_stamp[s_new[j]] = step;
  }
  __syncthreads();
  {
    // New order: the untouched slots in their old order, then every slot
    // used this step (hits and victims, all with stamp = step) by slot index.
    int keep = 0;
    for (int u = 0; u < kPer; u++) {
      const int pos = p0 + u;
      if (pos < ns && s_stamp[s_order[pos]] != step) keep++;
    }
    int n_keep;
    int krank = block_exclusive_scan(keep, scr, &n_keep);
    int used = 0;
    for (int u = 0; u < kPer; u++) {
      const int sl = p0 + u;
      if (sl < ns && s_stamp[sl] == step) used++;
    }
    int n_used;
    int rrank = block_exclusive_scan(used, scr, &n_used);
    for (int u = 0; u < kPer; u++) {
      const int pos = p0 + u;
      if (pos < ns && s_stamp[s_order[pos]] != step) s_new[krank++] = s_order[pos];
      const int sl = p0 + u;
      if (sl < ns && s_stamp[sl] == step) s_new[n_keep + rrank++] = sl;
    }
    __syncthreads();
    for (int pos = tid; pos < ns; pos += kResThreads) order[pos] = s_new[pos];
  }
  __syncthreads();
  for (int s = tid; s < ns; s += kResThreads) a.stamp[sbase + s] = s_stamp[s];
  if (tid == 0) a.n_miss[b] = ok ? nm : -1;
  __syncthreads();
  if (tid == 0) advance_step(a.step);
}

// ---------------------------------------------------------------------------
// Host-tier write path: int4 rows with 64-dim groups and fp16 group scales.
// ---------------------------------------------------------------------------
// One warp per (row, head) vector of d = 256*m dims: lane l encodes dims
// [8l, 8l+8) of each 256-dim block (group g = l/8 of the block).
__global__ __launch_bounds__(256) void quant_int4_kernel(const uint16_t* __restrict__ x, int64_t n_items,
                                                         int Hkv, int d, const int64_t* __restrict__ out_rows,
                                                         uint8_t* __restrict__ out, int64_t token_pitch,
                                                         int64_t head_pitch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * nw + warp; item < n_items;
       item += static_cast<int64_t>(gridDim.x) * nw) {
    const int64_t t = item / Hkv;
    const int h = static_cast<int>(item % Hkv);
    const int64_t orow = out_rows ? out_rows[t] : t;
    uint8_t* o = out + orow * token_pitch + h * head_pitch;
    const uint16_t* row = x + item * d;
    for (int blk = 0; blk < d; blk += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + blk + 8 * lane);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
      for (int o2 = 1; o2 < 8; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
      const __half sh = __float2half_rn(__fdiv_rn(amax, 7.f));
      const float sf = __half2float(sh);
      const bool ok = (sf != 0.f) && isfinite(sf);
      uint32_t packed = 0;
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const int q = ok ? rint_clamp(__fdiv_rn(f[e], sf), -8, 7) : 0;
        packed |= (static_cast<uint32_t>(q) & 0xfu) << (4 * e);
      }
      *reinterpret_cast<uint32_t*>(o + blk / 2 + 4 * lane) = packed;
      if ((lane & 7) == 0) {
        const int g = blk / 64 + lane / 8;
        *reinterpret_cast<__half*>(o + d / 2 + 2 * g) = sh;
      }
    }
  }
}

// Gather read: one warp per listed row (rows[i] * row_bytes from `base`,
// HBM or a host alias), every 16-byte load of the row issued before any is
// used; the XOR of the words goes to *sink.  The probe for reads of
// scattered rows, the access pattern of the host-tier fetches.
__global__ __launch_bounds__(256) void gather_read_kernel(const uint8_t* __restrict__ base,
                                                          const int64_t* __restrict__ rows, int n, int64_t row_bytes,
                                                          unsigned long long* sink) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= n) return;
  const uint4* src = reinterpret_cast<const uint4*>(base + rows[wid] * row_bytes);
  const int chunks = static_cast<int>(row_bytes / 16);
  uint32_t acc = 0;
  uint4 v[kFetchPieces];
#pragma unroll
  for (int u = 0; u < kFetchPieces; u++)
    v[u] = lane + 32 * u < chunks ? ld_stream16(src + lane + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int u = 0; u < kFetchPieces; u++) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  for (int c = lane + 32 * kFetchPieces; c < chunks; c += 32) {
    const uint4 x = ld_stream16(src + c);
    acc ^= x.x ^ x.y ^ x.z ^ x.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && acc == 0x9e3779b9u) atomicAdd(sink, 1ull);  // keeps the loads; almost never taken
}

// Streaming read of a buffer (HBM or a host alias) with 16-byte loads; the
// XOR of every word goes to *sink so the loads cannot be dropped.
__global__ __launch_bounds__(512) void stream_read_kernel(const uint4* __restrict__ p, int64_t n16,
                                                          unsigned long long* sink) {
  uint32_t acc = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; u++) v[u] = ld_stream16(p + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; u++) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = ld_stream16(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc) atomicXor(sink, static_cast<unsigned long long>(acc));
}

}  // namespace
}  // namespace skv

namespace skv {
namespace {
// A launch that may start while the previous kernel in the stream is still
// running (programmatic dependent launch); the kernel waits for that kernel
// with grid_dependency_wait() before it reads anything the kernel produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(dim3 grid, int threads, size_t smem, cudaStream_t st, void (*kernel)(KArgs...),
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_resolve_workspace_size(int B, int max_rows) {
  if (B < 1 || max_rows < 1) return 0;
  return 2 * static_cast<size_t>(B) * max_rows * sizeof(int32_t);
}

SKV_EXPORT int skv_resolve_rows_clock(int B, int64_t t_cap, const int32_t* lengths, int S, int W, int Hkv, int d,
                                      int Hs, const int32_t* idx, int max_rows, const int32_t* count,
                                      int32_t* step, int32_t* slot_token, uint8_t* ref, int32_t* use_step,
                                      int32_t* token_slot, int32_t* hand, const uint8_t* host_rows, int8_t* k8,
                                      int8_t* v8, uint16_t* k_scale, uint16_t* v_scale, int64_t req_row_stride,
                                      int32_t* rows_out, int32_t* n_miss, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, void* stream) {
  if (B < 0 || B > 65535 || t_cap < 0 || S < 0 || W < 0 || Hkv < 1 || Hs < 1 || max_rows < 1) return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (d < 256 || d % 256 || d > 1024) return SKV_EUNSUPPORTED;
  if (Hs > kMaxClockSlots || max_rows > kMaxResolveRows || t_cap > INT32_MAX) return SKV_EUNSUPPORTED;
  if (!step || req_row_stride < static_cast<int64_t>(S) + W + Hs) return SKV_EINVAL;
  if (!lengths || !idx || !count || !slot_token || !ref || !use_step || !token_slot || !hand || !host_rows ||
      !k8 || !v8 || !k_scale || !v_scale || !rows_out || !n_miss)
    return SKV_EINVAL;
  if (!aligned16(host_rows) || !aligned16(k8) || !aligned16(v8)) return SKV_EINVAL;
  const int tb = 2 * Hkv * (d / 2 + d / 32);
  if (tb > kMaxTokBytes) return SKV_EUNSUPPORTED;
  if (!workspace || workspace_bytes < skv_resolve_workspace_size(B, max_rows)) return SKV_ENOMEM;
  int32_t* ws_tok = static_cast<int32_t*>(workspace);
  int32_t* ws_row = ws_tok + static_cast<size_t>(B) * max_rows;
  const size_t smem = clock_smem_bytes(Hs, max_rows);
  static std::atomic<int> configured[kMaxDevices];
  static std::mutex configured_mu;
  if (smem_limit_at_least(configured, configured_mu, clock_kernel, smem) != SKV_OK) return SKV_EUNSUPPORTED;
  ClockArgs a{t_cap, lengths, S, W, Hkv, d, Hs, idx, max_rows, count, step, slot_token, ref, use_step,
              token_slot, hand, host_rows, k8, v8, reinterpret_cast<__half*>(k_scale),
              reinterpret_cast<__half*>(v_scale), req_row_stride, rows_out, n_miss, ws_tok, ws_row, dev_status};
  cudaStream_t st = as_stream(stream);
  clock_kernel<<<B, kClockThreads, smem, st>>>(a);
  const dim3 fgrid((max_rows + kFetchWarps - 1) / kFetchWarps, B);
  if (launch_dependent(fgrid, 32 * kFetchWarps, kFetchWarps * tb, st, fetch_int4_kernel, ws_tok, ws_row, n_miss,
                       max_rows, t_cap, Hkv, d, host_rows, k8, v8, reinterpret_cast<__half*>(k_scale),
                       reinterpret_cast<__half*>(v_scale)) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  return launch_status();
}

namespace {
int lru_resolve(int B, int64_t t_cap, const int32_t* lengths, int page, const int32_t* block_table, int64_t n_pages,
                int64_t hot_base, int64_t hot_stride, const int32_t* hot_blocks, int n_slots, int32_t* step,
                int64_t* stamp, int32_t* slot_token, int32_t* token_slot, int32_t* order, const uint8_t* host,
                uint8_t* pool, int64_t row_bytes, int64_t n_pool_rows, const int32_t* idx, int max_rows,
                const int32_t* count, int32_t* rows_out, int32_t* n_miss, void* workspace, size_t workspace_bytes,
                int32_t* dev_status, void* stream) {
  if (B < 0 || B > 65535 || t_cap < 0 || page < 1 || n_pages < 0 || n_slots < 1 || max_rows < 1 ||
      row_bytes < 16 || row_bytes % 16 || hot_base < 0 || hot_stride < 0)
    return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (n_slots > kMaxLruSlots || max_rows > kMaxResolveRows || t_cap > INT32_MAX) return SKV_EUNSUPPORTED;
  if (!step) return SKV_EINVAL;
  if (n_pool_rows > INT32_MAX) return SKV_EINVAL;
  if (!hot_blocks && hot_base + static_cast<int64_t>(B - 1) * hot_stride + n_slots > n_pool_rows) return SKV_EINVAL;
  if (!lengths || !block_table || !stamp || !slot_token || !token_slot || !order || !host || !pool || !idx ||
      !count || !rows_out || !n_miss)
    return SKV_EINVAL;
  if (!aligned16(host) || !aligned16(pool)) return SKV_EINVAL;
  if (!workspace || workspace_bytes < skv_resolve_workspace_size(B, max_rows)) return SKV_ENOMEM;
  int32_t* ws_tok = static_cast<int32_t*>(workspace);
  int32_t* ws_row = ws_tok + static_cast<size_t>(B) * max_rows;
  const size_t smem = lru_smem_bytes(n_slots, max_rows);
  static std::atomic<int> configured[kMaxDevices];
  static std::mutex configured_mu;
  if (smem_limit_at_least(configured, configured_mu, lru_kernel, smem) != SKV_OK) return SKV_EUNSUPPORTED;
  LruArgs a{t_cap, lengths, page, block_table, n_pages, hot_base, hot_stride, n_slots, step, stamp, slot_token,
            token_slot, order, host, pool, row_bytes, n_pool_rows, idx, max_rows, count, rows_out, n_miss, ws_tok,
            ws_row, dev_status, hot_blocks, (n_slots + page - 1) / page};
  cudaStream_t st = as_stream(stream);
  lru_kernel<<<B, kResThreads, smem, st>>>(a);
  const int per_cta = kFetchWarps * kRowsPerWarp;
  if (launch_dependent(dim3((max_rows + per_cta - 1) / per_cta, B), 32 * kFetchWarps, 0, st, fetch_rows_kernel,
                       ws_tok, ws_row, n_miss, max_rows, t_cap, host, pool, row_bytes) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  return launch_status();
}
}  // namespace

SKV_EXPORT int skv_resolve_rows_lru(int B, int64_t t_cap, const int32_t* lengths, int page,
                                    const int32_t* block_table, int64_t n_pages, int64_t hot_base,
                                    int64_t hot_stride, int n_slots, int32_t* step, int64_t* stamp,
                                    int32_t* slot_token, int32_t* token_slot, int32_t* order, const uint8_t* host,
                                    uint8_t* pool,
                                    int64_t row_bytes, int64_t n_pool_rows, const int32_t* idx, int max_rows,
                                    const int32_t* count, int32_t* rows_out, int32_t* n_miss, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return lru_resolve(B, t_cap, lengths, page, block_table, n_pages, hot_base, hot_stride, nullptr, n_slots, step,
                     stamp, slot_token, token_slot, order, host, pool, row_bytes, n_pool_rows, idx, max_rows, count,
                     rows_out, n_miss, workspace, workspace_bytes, dev_status, stream);
}

SKV_EXPORT int skv_resolve_rows_lru_leased(int B, int64_t t_cap, const int32_t* lengths, int page,
                                           const int32_t* block_table, int64_t n_pages, const int32_t* hot_blocks,
                                           int n_slots, int32_t* step, int64_t* stamp, int32_t* slot_token,
                                           int32_t* token_slot, int32_t* order, const uint8_t* host, uint8_t* pool,
                                           int64_t row_bytes, int64_t n_pool_rows, const int32_t* idx, int max_rows,
                                           const int32_t* count, int32_t* rows_out, int32_t* n_miss,
                                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
  if (!hot_blocks) return SKV_EINVAL;
  return lru_resolve(B, t_cap, lengths, page, block_table, n_pages, 0, 0, hot_blocks, n_slots, step, stamp,
                     slot_token, token_slot, order, host, pool, row_bytes, n_pool_rows, idx, max_rows, count,
                     rows_out, n_miss, workspace, workspace_bytes, dev_status, stream);
}

SKV_EXPORT int skv_quantize_int4_rows(const uint16_t* x, int64_t n_rows, int Hkv, int d, const int64_t* out_rows,
                                      uint8_t* out, int64_t token_pitch, int64_t head_pitch, void* stream) {
  if (n_rows < 0 || Hkv < 1 || d < 256 || d % 256 || d > 1024) return SKV_EINVAL;
  if (n_rows == 0) return SKV_OK;
  if (!x || !out || !aligned16(x)) return SKV_EINVAL;
  const int64_t rb = d / 2 + 2 * (d / 64);
  if (head_pitch < rb || token_pitch < Hkv * head_pitch) return SKV_EINVAL;
  if ((reinterpret_cast<uintptr_t>(out) | token_pitch | head_pitch) & 3) return SKV_EINVAL;
  const int64_t items = n_rows * Hkv;
  int64_t grid = (items + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (grid > cap && cap > 0) grid = cap;
  quant_int4_kernel<<<static_cast<int>(grid), 256, 0, as_stream(stream)>>>(x, items, Hkv, d, out_rows, out,
                                                                            token_pitch, head_pitch);
  return launch_status();
}

SKV_EXPORT int skv_gather_read(const void* base, const int64_t* rows, int n, int64_t row_bytes,
                               unsigned long long* sink, void* stream) {
  if (!base || !rows || !sink || n < 0 || row_bytes < 16 || row_bytes % 16 || !aligned16(base)) return SKV_EINVAL;
  if (n == 0) return SKV_OK;
  const int64_t blocks = (static_cast<int64_t>(n) * 32 + 255) / 256;
  if (blocks > INT32_MAX) return SKV_EINVAL;
  gather_read_kernel<<<static_cast<int>(blocks), 256, 0, as_stream(stream)>>>(static_cast<const uint8_t*>(base), rows,
                                                                             n, row_bytes, sink);
  return launch_status();
}

SKV_EXPORT int skv_stream_read(const void* src, size_t bytes, unsigned long long* sink, int grid, void* stream) {
  if (!src || !sink || bytes % 16 || !aligned16(src) || grid < 0) return SKV_EINVAL;
  if (bytes == 0) return SKV_OK;
  if (grid == 0) grid = 2 * sm_count();
  stream_read_kernel<<<grid, 512, 0, as_stream(stream)>>>(static_cast<const uint4*>(src),
                                                          static_cast<int64_t>(bytes / 16), sink);
  return launch_status();
}
