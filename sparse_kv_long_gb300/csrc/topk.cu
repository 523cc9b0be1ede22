// topk.cu -- deterministic top-k selection (a4).
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": top 2048 +
// 64 sinks + last 1024 tokens, "deterministic radix select", one pick per
// layer.  [P4] "3.14M Context on 3x 3090 ...", "Why": the pooled indexer
// switches to sparse reads once the context exceeds 4*block_topk + 3 tokens.
//
// Radix select over 32-bit order keys in three digit passes (bits 31..21,
// 20..10, 9..0).  Each pass is one launch of CT CTAs per request: a CTA
// histograms the digit of the keys that still match the prefix found so far
// (shared-memory bins, warp-aggregated increments), adds its bins to the
// request's global histogram, and the last CTA to finish (atomic ticket, no
// waiting) finds the digit holding the k-th key and updates the prefix.  After
// the last pass the k-th key K* is exact and `need` says how many keys equal to
// K* are taken: the lowest-index ones.  A count launch and a write launch then
// emit the selection in ascending index order with an ordered block-wide
// compaction per chunk.  All steps are deterministic.
#include <mutex>

#include "common.cuh"

namespace skv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCTMax = 64;
constexpr int kUnroll = 8;         // keys per thread whose loads are in flight together
constexpr int kFlagWords = 1024;   // write pass: bits marking 32-key groups that hold a pick candidate

// Scratch of one request, at a fixed stride whatever B is, so that one
// zero-filled workspace serves calls with any number of requests: the words
// that must start at zero (histograms, tickets, todo) are returned to zero by
// every call, and the rest is written before it is read.
//   hist   [3][kBins]  digit histograms of the three passes
//   done   [3]         per-pass tickets
//   todo   [1]         the request still needs the radix passes (many-request path)
//   state  [4]         prefix, mask, need, pad
//   cgt, ceq [kCTMax]  per-chunk counts of keys above / equal to K*
constexpr size_t kReqWords = 3ull * kBins + 4 + 4 + 2ull * kCTMax;

struct Ws {
  uint32_t* base;
  __device__ __forceinline__ uint32_t* req(int b) const { return base + static_cast<size_t>(b) * kReqWords; }
  __device__ __forceinline__ uint32_t* hist(int pass, int b) const { return req(b) + static_cast<size_t>(pass) * kBins; }
  __device__ __forceinline__ uint32_t* done(int pass, int b) const { return req(b) + 3 * kBins + pass; }
  __device__ __forceinline__ int32_t* todo(int b) const { return reinterpret_cast<int32_t*>(req(b) + 3 * kBins + 3); }
  __device__ __forceinline__ uint32_t* state(int b) const { return req(b) + 3 * kBins + 4; }
  __device__ __forceinline__ int32_t* cgt(int b) const { return reinterpret_cast<int32_t*>(req(b) + 3 * kBins + 8); }
  __device__ __forceinline__ int32_t* ceq(int b) const { return cgt(b) + kCTMax; }
};

__host__ __device__ inline size_t ws_bytes(int B) { return sizeof(uint32_t) * kReqWords * static_cast<size_t>(B); }

inline Ws ws_carve(void* base, int) { return Ws{static_cast<uint32_t*>(base)}; }

struct Sel {
  const uint32_t* okeys;
  int64_t n_cap;
  const int32_t* lengths;
  int k, S, W, ratio, CT, B;
  int32_t* idx;
  int max_rows;
  int32_t* count;
  int32_t* status;
  int only_todo;  // 0: every request; else only those whose workspace todo word is set
};

// Candidate range [lo, hi) of request b and whether it takes the dense path.
__device__ __forceinline__ bool request_range(const Sel& s, int b, int64_t* T, int64_t* lo, int64_t* hi) {
  int64_t t = s.lengths[b];
  const int64_t cap = s.ratio > 1 ? s.n_cap * s.ratio : s.n_cap;
  if (t > cap) t = cap;
  if (t < 0) t = 0;
  *T = t;
  bool dense;
  if (s.ratio <= 1) {
    dense = t <= static_cast<int64_t>(s.S) + s.W + s.k;
    *lo = s.S;
    *hi = t - s.W;
  } else {
    dense = t <= static_cast<int64_t>(s.ratio) * s.k + s.ratio - 1;
    *lo = 0;
    *hi = t / s.ratio;
  }
  return dense;
}

__device__ __forceinline__ void chunk_of(int64_t lo, int64_t hi, int CT, int c, int64_t* c0, int64_t* c1) {
  const int64_t n = hi - lo;
  const int64_t chunk = (n + CT - 1) / CT;
  *c0 = lo + c * chunk;
  *c1 = (*c0 + chunk < hi) ? *c0 + chunk : hi;
  if (*c0 > hi) *c0 = hi;
}

__device__ __forceinline__ void pass_digits(int pass, int* shift, int* nbins) {
  *shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
  *nbins = pass == 2 ? 1024 : 2048;
}

__global__ __launch_bounds__(kThreads) void topk_hist_kernel(Sel s, Ws w, int pass) {
  __shared__ uint32_t h[kBins];
  __shared__ int scan[33];
  __shared__ int last;
  const int b = blockIdx.y, c = blockIdx.x;
  if (s.only_todo && !*w.todo(b)) return;
  int64_t T, lo, hi;
  if (request_range(s, b, &T, &lo, &hi)) return;  // dense: nothing to select
  int shift, nbins;
  pass_digits(pass, &shift, &nbins);
  uint32_t prefix = 0, mask = 0, need = static_cast<uint32_t>(s.k);
  if (pass > 0) {
    prefix = w.state(b)[0];
    mask = w.state(b)[1];
    need = w.state(b)[2];
  }
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) h[i] = 0;
  __syncthreads();
  int64_t c0, c1;
  chunk_of(lo, hi, s.CT, c, &c0, &c1);
  const uint32_t* ok = s.okeys + static_cast<int64_t>(b) * s.n_cap;
  const int lane = threadIdx.x & 31;
  for (int64_t base = c0; base < c1; base += static_cast<int64_t>(blockDim.x) * kUnroll) {
    uint32_t key[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t i = base + threadIdx.x + u * blockDim.x;
      key[u] = i < c1 ? ok[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t i = base + threadIdx.x + u * blockDim.x;
      uint32_t digit = 0xffffffffu;
      if (i < c1 && (key[u] & mask) == prefix) digit = (key[u] >> shift) & static_cast<uint32_t>(nbins - 1);
      // later passes: most keys left the prefix already, and a warp with none
      // of them skips the (costly) match
      if (pass > 0 && !__any_sync(0xffffffffu, digit != 0xffffffffu)) continue;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (digit != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&h[digit], __popc(peers));
    }
  }
  __syncthreads();
  uint32_t* gh = w.hist(pass, b);
  for (int i = threadIdx.x; i < nbins; i += blockDim.x)
    if (h[i]) atomicAdd(&gh[i], h[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(w.done(pass, b), 1u) == static_cast<unsigned>(s.CT - 1));
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Last CTA of this request: read the full histogram (from L2) and clear it.
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) {
    h[i] = __ldcg(&gh[i]);
    gh[i] = 0;
  }
  __syncthreads();
  // Thread t owns bins_per_thread consecutive bins counted from the top.
  const int bpt = nbins / blockDim.x;
  const int top = nbins - 1 - threadIdx.x * bpt;
  int local = 0;
  for (int j = 0; j < bpt; j++) local += static_cast<int>(h[top - j]);
  int tot;
  int above = block_exclusive_scan(local, scan, &tot);
  if (static_cast<uint32_t>(tot) < need && threadIdx.x == 0) set_status(s.status, SKV_DEV_COUNT);
  for (int j = 0; j < bpt; j++) {
    const int bin = top - j;
    const int cnt = static_cast<int>(h[bin]);
    if (static_cast<uint32_t>(above) < need && static_cast<uint32_t>(above + cnt) >= need) {
      w.state(b)[0] = prefix | (static_cast<uint32_t>(bin) << shift);
      w.state(b)[1] = mask | (static_cast<uint32_t>(nbins - 1) << shift);
      w.state(b)[2] = need - static_cast<uint32_t>(above);
    }
    above += cnt;
  }
  if (threadIdx.x == 0) *w.done(pass, b) = 0;
}

__global__ __launch_bounds__(kThreads) void topk_count_kernel(Sel s, Ws w) {
  __shared__ int red[2][32];
  const int b = blockIdx.y, c = blockIdx.x;
  if (s.only_todo && !*w.todo(b)) return;
  int64_t T, lo, hi;
  if (request_range(s, b, &T, &lo, &hi)) return;
  const uint32_t kstar = w.state(b)[0];
  int64_t c0, c1;
  chunk_of(lo, hi, s.CT, c, &c0, &c1);
  const uint32_t* ok = s.okeys + static_cast<int64_t>(b) * s.n_cap;
  int gt = 0, eq = 0;
  for (int64_t base = c0; base < c1; base += static_cast<int64_t>(blockDim.x) * kUnroll) {
    uint32_t key[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t i = base + threadIdx.x + u * blockDim.x;
      key[u] = i < c1 ? ok[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const bool valid = base + threadIdx.x + u * blockDim.x < c1;
      gt += valid && key[u] > kstar;
      eq += valid && key[u] == kstar;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = gt;
    red[1][warp] = eq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int g = 0, e = 0;
    for (int i = 0; i < (blockDim.x >> 5); i++) {
      g += red[0][i];
      e += red[1][i];
    }
    w.cgt(b)[c] = g;
    w.ceq(b)[c] = e;
  }
}

// Ordered write of this CTA's picks.  Warp v owns the contiguous piece
// [p0, p1) of the CTA's chunk.  A first pass counts each warp's keys above
// K* and equal to K* and marks the 32-key groups that hold any of them; the
// warps' output offsets follow from those counts (ties: lowest index first,
// up to the quota); a second pass revisits only the marked groups and writes
// the picks with warp ballots, so no block-wide scan runs per key.
__global__ __launch_bounds__(kThreads) void topk_write_kernel(Sel s, Ws w) {
  __shared__ int base_s[2];
  __shared__ int wgt[kWarps], weq[kWarps];
  __shared__ unsigned flags[kFlagWords];
  const int b = blockIdx.y, c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (s.only_todo && !*w.todo(b)) return;
  int64_t T, lo, hi;
  const bool dense = request_range(s, b, &T, &lo, &hi);
  int32_t* out = s.idx + static_cast<int64_t>(b) * s.max_rows;
  if (dense) {
    for (int64_t i = static_cast<int64_t>(c) * blockDim.x + threadIdx.x; i < T;
         i += static_cast<int64_t>(s.CT) * blockDim.x)
      out[i] = static_cast<int32_t>(i);
    if (c == 0 && threadIdx.x == 0) s.count[b] = static_cast<int32_t>(T);
    return;
  }
  const uint32_t kstar = w.state(b)[0];
  const int need = static_cast<int>(w.state(b)[2]);
  if (threadIdx.x < 32) {
    int g = 0, e = 0;
    for (int i = threadIdx.x; i < c; i += 32) {
      g += w.cgt(b)[i];
      e += w.ceq(b)[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (threadIdx.x == 0) {
      base_s[0] = g;
      base_s[1] = e;
    }
  }
  int64_t c0, c1;
  chunk_of(lo, hi, s.CT, c, &c0, &c1);
  const uint32_t* ok = s.okeys + static_cast<int64_t>(b) * s.n_cap;
  const int64_t sub = ((c1 - c0 + kWarps - 1) / kWarps + 31) / 32 * 32;  // whole 32-key groups per warp
  const int64_t p0 = c0 + warp * sub < c1 ? c0 + warp * sub : c1;
  const int64_t p1 = p0 + sub < c1 ? p0 + sub : c1;
  const int64_t n_groups = (p1 - p0 + 31) / 32;
  constexpr int kWordsPerWarp = kFlagWords / kWarps;
  const bool marked = n_groups <= 32 * kWordsPerWarp;  // larger pieces revisit every group
  unsigned* myflags = flags + warp * kWordsPerWarp;
  // pass 1: counts and group marks, kUnroll groups' loads in flight per lane
  int ngt = 0, neq = 0;
  for (int64_t g0 = 0; g0 < n_groups; g0 += 32) {
    unsigned word = 0u;
    for (int q = 0; q < 32 && g0 + q < n_groups; q += kUnroll) {
      uint32_t key[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; u++) {
        const int64_t i = p0 + (g0 + q + u) * 32 + lane;
        key[u] = i < p1 ? ok[i] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; u++) {
        const bool valid = p0 + (g0 + q + u) * 32 + lane < p1;
        const bool gt = valid && key[u] > kstar, eq = valid && key[u] == kstar;
        ngt += gt;
        neq += eq;
        if (__ballot_sync(0xffffffffu, gt || eq)) word |= 1u << (q + u);
      }
    }
    if (marked && lane == 0) myflags[g0 / 32] = word;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
    neq += __shfl_xor_sync(0xffffffffu, neq, o);
  }
  if (lane == 0) {
    wgt[warp] = ngt;
    weq[warp] = neq;
  }
  __syncthreads();
  const int ties_before = base_s[1] < need ? base_s[1] : need;
  const int quota = need - ties_before;
  int pos = base_s[0] + ties_before;
  int eq_run = 0;  // keys equal to K* in this CTA before this warp's piece
  for (int v = 0; v < warp; v++) {
    pos += wgt[v] + max(0, min(weq[v], quota - eq_run));
    eq_run += weq[v];
  }
  if (c == s.CT - 1 && threadIdx.x == 0) {  // the request's last chunk: every pick placed
    int end = base_s[0] + ties_before, er = 0;
    for (int v = 0; v < kWarps; v++) {
      end += wgt[v] + max(0, min(weq[v], quota - er));
      er += weq[v];
    }
    if (end != s.k) set_status(s.status, SKV_DEV_COUNT);
  }
  // pass 2: the marked groups again, picks written in ascending index order
  const int ratio = s.ratio > 1 ? s.ratio : 1;
  const int head = s.ratio > 1 ? 0 : s.S;
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t gi = 0; gi < n_groups; gi++) {
    if (marked && !((myflags[gi / 32] >> (gi % 32)) & 1u)) continue;
    const int64_t i = p0 + gi * 32 + lane;
    const uint32_t key = i < p1 ? ok[i] : 0u;
    const bool gt = i < p1 && key > kstar;
    const bool eq = i < p1 && key == kstar;
    const unsigned eqb = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_run + __popc(eqb & lt) < quota);
    const unsigned selb = __ballot_sync(0xffffffffu, sel);
    if (sel) {
      const int j = pos + __popc(selb & lt);
      if (j < s.k) {
        for (int u = 0; u < ratio; u++) out[head + ratio * j + u] = static_cast<int32_t>(ratio * i + u);
      } else {
        set_status(s.status, SKV_DEV_COUNT);
      }
    }
    pos += __popc(selb);
    eq_run += __popc(eqb);
  }
  if (c == 0) {
    if (s.ratio <= 1) {
      for (int i = threadIdx.x; i < s.S; i += blockDim.x) out[i] = i;
      for (int i = threadIdx.x; i < s.W; i += blockDim.x)
        out[s.S + s.k + i] = static_cast<int32_t>(T - s.W + i);
      if (threadIdx.x == 0) s.count[b] = s.S + s.k + s.W;
    } else {
      const int64_t nb = T / s.ratio;
      const int rem = static_cast<int>(T - nb * s.ratio);
      for (int i = threadIdx.x; i < rem; i += blockDim.x)
        out[s.ratio * s.k + i] = static_cast<int32_t>(nb * s.ratio + i);
      if (threadIdx.x == 0) s.count[b] = s.ratio * s.k + rem;
    }
  }
}

// ---- many requests: one CTA each, threshold filter -----------------------------------
// With at least two requests per SM every request has a single CTA, and the
// radix passes would stream its keys five times.  Instead the CTA takes an
// evenly spaced sample of the keys, sorts it, and picks a threshold tau below
// the sample's ~2k/n quantile; every key >= tau (with its index) goes to
// shared memory -- at least k of them hold the k best, ties at K* included,
// since all keys equal to K* >= tau are kept -- and a bitonic sort by (key
// descending, index ascending) of those candidates gives the selection, which
// a second sort puts in index order.  A request whose candidates overflow the
// buffer, or number fewer than k, is marked for the radix passes.
constexpr int kCand = 8192;       // candidates held in shared memory (64-bit: key, inverted index)
constexpr int kSamp = 4096;       // sampled keys
constexpr int kMaxFilterK = 2048;

__device__ void bitonic_desc_u64(unsigned long long* a, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1)), j = i + stride;
        const bool up = (i & size) == 0;  // this run ends descending
        const unsigned long long x = a[i], y = a[j];
        if ((x < y) == up) {
          a[i] = y;
          a[j] = x;
        }
      }
      __syncthreads();
    }
}

template <typename V>
__device__ void bitonic_asc(V* a, int n) {
  for (int size = 2; size <= n; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n / 2; t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1)), j = i + stride;
        const bool up = (i & size) == 0;
        const V x = a[i], y = a[j];
        if ((x > y) == up) {
          a[i] = y;
          a[j] = x;
        }
      }
      __syncthreads();
    }
}

__global__ __launch_bounds__(kThreads) void topk_filter_kernel(Sel s, Ws w) {
  extern __shared__ __align__(16) unsigned long long cand[];  // [kCand]; the sample aliases its front
  __shared__ int32_t picks[kMaxFilterK];
  __shared__ unsigned s_cnt;
  const int b = blockIdx.x, lane = threadIdx.x & 31;
  int64_t T, lo, hi;
  const bool dense = request_range(s, b, &T, &lo, &hi);
  int32_t* out = s.idx + static_cast<int64_t>(b) * s.max_rows;
  if (dense) {
    for (int64_t i = threadIdx.x; i < T; i += blockDim.x) out[i] = static_cast<int32_t>(i);
    if (threadIdx.x == 0) {
      s.count[b] = static_cast<int32_t>(T);
      *w.todo(b) = 0;
    }
    return;
  }
  const int64_t n = hi - lo;
  const uint32_t* ok = s.okeys + static_cast<int64_t>(b) * s.n_cap + lo;
  uint32_t tau = 0u;
  if (n > kCand) {
    uint32_t* samp = reinterpret_cast<uint32_t*>(cand);
    for (int j = threadIdx.x; j < kSamp; j += blockDim.x) samp[j] = ok[static_cast<int64_t>(j) * n / kSamp];
    __syncthreads();
    bitonic_asc(samp, kSamp);
    const int64_t r = (2ll * s.k * kSamp + n - 1) / n + 16;  // from the top
    tau = samp[kSamp - 1 - (r < kSamp ? r : kSamp - 1)];
    __syncthreads();  // the candidates overwrite the sample
  }
  if (threadIdx.x == 0) s_cnt = 0u;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t base = 0; base < n; base += static_cast<int64_t>(blockDim.x) * kUnroll) {
    uint32_t key[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t i = base + threadIdx.x + u * blockDim.x;
      key[u] = i < n ? ok[i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; u++) {
      const int64_t i = base + threadIdx.x + u * blockDim.x;
      const bool keep = i < n && key[u] >= tau;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      unsigned at = 0u;
      if (lane == 0 && m) at = atomicAdd(&s_cnt, static_cast<unsigned>(__popc(m)));
      at = __shfl_sync(0xffffffffu, at, 0);
      if (keep) {
        const unsigned slot = at + __popc(m & lt);
        if (slot < kCand)
          cand[slot] = (static_cast<unsigned long long>(key[u]) << 32) | (0xffffffffu - static_cast<uint32_t>(i));
      }
    }
  }
  __syncthreads();
  const unsigned total = s_cnt;
  if (total < static_cast<unsigned>(s.k) || total > static_cast<unsigned>(kCand)) {  // the same in every thread
    if (threadIdx.x == 0) *w.todo(b) = 1;
    return;
  }
  int N = 1;
  while (N < static_cast<int>(total)) N <<= 1;
  for (int j = static_cast<int>(total) + threadIdx.x; j < N; j += blockDim.x) cand[j] = 0ull;  // sorts last
  __syncthreads();
  bitonic_desc_u64(cand, N);
  int K = 1;
  while (K < s.k) K <<= 1;
  for (int j = threadIdx.x; j < K; j += blockDim.x)
    picks[j] = j < s.k ? static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(cand[j])) : INT32_MAX;
  __syncthreads();
  bitonic_asc(picks, K);
  const int ratio = s.ratio > 1 ? s.ratio : 1;
  const int head = s.ratio > 1 ? 0 : s.S;
  for (int j = threadIdx.x; j < s.k; j += blockDim.x) {
    const int64_t i = lo + picks[j];
    for (int u = 0; u < ratio; u++) out[head + ratio * j + u] = static_cast<int32_t>(ratio * i + u);
  }
  if (s.ratio <= 1) {
    for (int i = threadIdx.x; i < s.S; i += blockDim.x) out[i] = i;
    for (int i = threadIdx.x; i < s.W; i += blockDim.x) out[s.S + s.k + i] = static_cast<int32_t>(T - s.W + i);
    if (threadIdx.x == 0) s.count[b] = s.S + s.k + s.W;
  } else {
    const int64_t nb = T / s.ratio;
    const int rem = static_cast<int>(T - nb * s.ratio);
    for (int i = threadIdx.x; i < rem; i += blockDim.x) out[s.ratio * s.k + i] = static_cast<int32_t>(nb * s.ratio + i);
    if (threadIdx.x == 0) s.count[b] = s.ratio * s.k + rem;
  }
  if (threadIdx.x == 0) *w.todo(b) = 0;
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_topk_workspace_size(int B) { return B > 0 ? ws_bytes(B) : 0; }

SKV_EXPORT int skv_topk_select(int B, const uint32_t* order_keys, int64_t n_cap,
                               const int32_t* lengths, int k, int S, int W, int ratio, int32_t* idx,
                               int max_rows, int32_t* count, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream) {
  if (B < 0 || B > 4096 || k < 1 || S < 0 || W < 0 || ratio < 1 || n_cap < 0) return SKV_EINVAL;
  if (B == 0) return SKV_OK;
  if (!order_keys || !lengths || !idx || !count || !workspace) return SKV_EINVAL;
  if (ratio > 1 && (S != 0 || W != 0)) return SKV_EINVAL;
  const int64_t need_rows = ratio > 1 ? static_cast<int64_t>(ratio) * k + ratio - 1
                                      : static_cast<int64_t>(S) + k + W;
  if (max_rows < need_rows) return SKV_EINVAL;
  if (workspace_bytes < ws_bytes(B)) return SKV_ENOMEM;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return SKV_EINVAL;
  int CT = (2 * sm_count() + B - 1) / B;
  CT = CT < 1 ? 1 : (CT > kCTMax ? kCTMax : CT);
  Sel s{order_keys, n_cap, lengths, k, S, W, ratio, CT, B, idx, max_rows, count, dev_status, 0};
  Ws w = ws_carve(workspace, B);
  cudaStream_t st = as_stream(stream);
  dim3 grid(CT, B);
  if (CT == 1 && k <= kMaxFilterK) {  // one CTA per request: threshold filter, radix passes for the rest
    constexpr size_t smem = kCand * sizeof(unsigned long long);
    static std::atomic<int> configured[kMaxDevices];
    if (smem_limit_once(configured, topk_filter_kernel, smem) != SKV_OK) return SKV_ECUDA;
    topk_filter_kernel<<<B, kThreads, smem, st>>>(s, w);
    s.only_todo = 1;
  }
  for (int pass = 0; pass < 3; pass++) topk_hist_kernel<<<grid, kThreads, 0, st>>>(s, w, pass);
  topk_count_kernel<<<grid, kThreads, 0, st>>>(s, w);
  topk_write_kernel<<<grid, kThreads, 0, st>>>(s, w);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Top-k selection without caller-provided scratch.
//
// Some callers cannot hand this library a workspace: for example an engine
// that reserves all device memory for its own KV pools before decoding starts
// and gives out no side buffers, or a latency-critical decode loop that must
// not call cudaMalloc (which can synchronise the device).  For them the
// selection's scratch (digit histograms, tickets, per-chunk counts) lives in
// a fixed device array compiled into the library, sized for at most
// kNoAllocMaxB requests.  Every device that loads the library holds this
// array until the process exits.
// ---------------------------------------------------------------------------
namespace skv {
namespace {

constexpr int kNoAllocMaxB = 32;
constexpr size_t kNoAllocBytes = sizeof(uint32_t) * kReqWords * kNoAllocMaxB;

static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_topk_scratch on the current device.  The host-side name
// of the array is only a stand-in, so the address is looked up once per device
// (with that device current) and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SKV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return SKV_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SKV_OK;
}

}  // namespace
}  // namespace skv

SKV_EXPORT int skv_topk_select_noalloc(int B, const uint32_t* order_keys, int64_t n_cap,
                                       const int32_t* lengths, int k, int S, int W, int ratio,
                                       int32_t* idx, int max_rows, int32_t* count, int32_t* dev_status,
                                       void* stream) {
  if (B < 0 || k < 1 || S < 0 || W < 0 || ratio < 1 || n_cap < 0) return SKV_EINVAL;
  if (B > kNoAllocMaxB) return SKV_ENOMEM;  // the fixed scratch holds kNoAllocMaxB requests
  if (B == 0) return SKV_OK;
  if (!order_keys || !lengths || !idx || !count) return SKV_EINVAL;
  if (ratio > 1 && (S != 0 || W != 0)) return SKV_EINVAL;
  const int64_t need_rows = ratio > 1 ? static_cast<int64_t>(ratio) * k + ratio - 1
                                      : static_cast<int64_t>(S) + k + W;
  if (max_rows < need_rows) return SKV_EINVAL;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SKV_OK) return rc;
  cudaStream_t st = as_stream(stream);
  // The array keeps whatever the previous call left; the histograms, tickets
  // and todo words must start at zero, so the call's per-request blocks are
  // cleared (no allocation involved).
  const size_t zero_bytes = ws_bytes(B);
  if (cudaMemsetAsync(scratch, 0, zero_bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }
  int CT = (2 * sm_count() + B - 1) / B;
  CT = CT < 1 ? 1 : (CT > kCTMax ? kCTMax : CT);
  Sel s{order_keys, n_cap, lengths, k, S, W, ratio, CT, B, idx, max_rows, count, dev_status, 0};
  Ws w = ws_carve(scratch, B);
  dim3 grid(CT, B);
  for (int pass = 0; pass < 3; pass++) topk_hist_kernel<<<grid, kThreads, 0, st>>>(s, w, pass);
  topk_count_kernel<<<grid, kThreads, 0, st>>>(s, w);
  topk_write_kernel<<<grid, kThreads, 0, st>>>(s, w);
  return launch_status();
}
