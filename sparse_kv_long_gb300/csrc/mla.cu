// mla.cu -- a6 over latent (MLA) rows: exact sparse attention of 128 absorbed
// query heads over fp8 e4m3 rows of 576 values (512 latent + 64 rope, V = the
// latent part), on the 5th-generation tensor cores.
//
// [P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one block pool":
// the attention kernel reads the selected rows wherever the resolver put
// them (in place, hot buffer); the pool rows here are what that resolver
// returns.
//
// Per request the work is S = Q.K^T (M = 128 heads, K = 576) and O = P.V
// (N = 512): 570 MFLOP over 2048 rows, about 480 flop per byte read, so the
// tensor cores set the pace.  The fp32 output O (128 x 512) alone fills a
// whole SM's tensor memory, so a CTA pair (cluster of 2) shares every row
// chunk:
//   * CTA r gathers dims [256 r, 256 r + 320) of each row (fp8 -> fp16, exact)
//     into a 128-byte-swizzled tile that serves both products;
//   * its share of the query (dims [0, 320) or [320, 576)) sits in tensor
//     memory as the A operand of the logit product, so only the row tile is
//     read from shared memory by each MMA;
//   * it computes the partial logits over its share of the contraction, each
//     softmax warp ships its 32 heads' partials to the peer with one bulk
//     copy (completion counted on the peer's barrier) and adds the peer's
//     (a + b on both sides, so both hold the same logits and softmax);
//   * it accumulates O for its half of the value dims ([0, 256) or
//     [256, 512)) in tensor memory.
// Roles in a CTA: warp 0 issues tcgen05.mma (one thread), warps 1-3 gather
// rows into a 3-deep ring, warps 4-7 own one head each (tensor-memory lane =
// head) for the online softmax and the epilogue.  Rows are split across
// clusters; the splits are merged in a fixed order (deterministic): when a
// request has two splits, its two CTA pairs form one cluster of four and merge
// through distributed shared memory at the end, otherwise a merge kernel
// combines the partials.
#include <cstddef>

#include "tc.cuh"

namespace skv {
namespace {

constexpr int kH = 128;
constexpr int kD = 576;
constexpr int kDv = 512;
constexpr int kNr = 64;                         // rows per chunk (N of the logit product)
constexpr int kSlice = 320;                     // dims gathered per CTA
constexpr int kAtoms = kSlice / 64;             // 64-dim swizzle atoms per tile row
constexpr int kPieces = kSlice / 16;            // 16-byte fp8 pieces per row and CTA
constexpr int kBuf = 3;                         // gather ring depth
constexpr int kKVBytes = kAtoms * kNr * 128;    // 40 KB per ring slot
constexpr int kPBytes = kH * 128;               // 16 KB
constexpr int kXBytes = kH * kNr * 4;           // 32 KB (one direction of the exchange)
constexpr int kThreads = 256;
constexpr int kProducers = 96;
constexpr int kPerProducer = (kNr * kPieces + kProducers - 1) / kProducers;
constexpr int kTmemCols = 512;                  // S [0, 64), Q [64, 224), O [256, 512)
constexpr int kSCol = 0;
constexpr int kQCol = 64;
constexpr int kOCol = 256;
constexpr float kRescaleLog2 = 8.f;             // rescale O only when the max grows by > 2^8

struct Aux {
  uint64_t kv_full[kBuf], kv_empty[kBuf];
  uint64_t s_full, s_empty, p_full, pv_done, x_full, x_empty, mma_idle, q_full;
  alignas(16) int32_t prow[kBuf][kNr];  // pool rows of the chunk in slot s (-1: none), staged by the gather warps
  alignas(16) float kl[kBuf][kNr];      // logit factor of each row: row scale x softmax scale x log2(e); 0 if no row
  alignas(16) float madd[kBuf][kNr];    // 0, or -inf for a missing row
  alignas(16) float vsc[kBuf][kNr];     // value factor: the row scale; 0 if no row
  float mrow[kH], lrow[kH];             // in-cluster split merge: running max and row sum per head
  uint32_t tmem_base;
  int abort;
};

// The softmax reads kl / madd / vsc as float4.
static_assert(offsetof(Aux, kl) % 16 == 0 && offsetof(Aux, madd) % 16 == 0 && offsetof(Aux, vsc) % 16 == 0,
              "per-row factor arrays must be 16-byte aligned");
static_assert((kBuf * kKVBytes + kPBytes + 2 * kXBytes) % 16 == 0, "Aux must start 16-byte aligned");

// Prologue and epilogue stage rows in the (then idle) gather ring + P buffer,
// with 16 bytes of padding per row so that thread h's row accesses fall in
// distinct bank groups.
constexpr int kQRowBytes = kSlice * 2;            // a CTA's query share: at most 320 dims, bf16
constexpr int kQStride = kQRowBytes + 16;
constexpr int kORowBytes = 256 * 4;               // a CTA's output share: 256 fp32 values
constexpr int kOStride = kORowBytes + 16;
static_assert(kH * kQStride <= kBuf * kKVBytes && kH * kOStride <= kBuf * kKVBytes + kPBytes,
              "staging fits in the ring and the P buffer");

constexpr int kSmem = 1024 + kBuf * kKVBytes + kPBytes + 2 * kXBytes + static_cast<int>(sizeof(Aux));

struct MlaArgs {
  const uint16_t* q;
  const uint8_t* pool;
  const float* row_scale;
  int64_t req_row_stride, n_pool_rows;
  const int32_t* rows;
  int max_rows;
  const int32_t* count;
  float scale_log2;
  float* out;
  float* ws_o;      // [B][nsplit][128][512] unnormalised partial outputs
  float* ws_ml;     // [B][nsplit][128][2]: running max (log2 units), row sum
  int nsplit;
  int cmerge;       // 1: the two splits of a request are one 4-CTA cluster and merge in it
  int32_t* status;
};

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n)); }

// Named barrier over n threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_sync_and(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbarrier.red.and.pred q, %2, %3, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Launched in clusters of (2, 1, 1) -- a CTA pair -- or (2, 2, 1) when the
// request's two splits merge inside the cluster.
__global__ void __launch_bounds__(kThreads, 1) mla_kernel(MlaArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sKV = sm;
  unsigned char* sP = sKV + kBuf * kKVBytes;
  float* sXin = reinterpret_cast<float*>(sP + kPBytes);   // the peer's partial logits
  float* sXout = sXin + kH * kNr;                         // this CTA's, staged for the bulk copy
  Aux* ax = reinterpret_cast<Aux*>(sP + kPBytes + 2 * kXBytes);

  allow_dependent_launch();  // the split merge may be scheduled onto the SMs this grid leaves free
  const uint32_t crank = tc::cluster_rank();
  const uint32_t rank = crank & 1u, peer = crank ^ 1u;  // position in the pair, the pair partner's cluster rank
  const int split = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int n = a.count[b];
  if (n < 0 || n > a.max_rows) {
    if (tid == 0 && rank == 0 && split == 0) set_status(a.status, SKV_DEV_COUNT);
    n = n < 0 ? 0 : a.max_rows;
  }
  const int per = ((n + a.nsplit - 1) / a.nsplit + kNr - 1) / kNr * kNr;
  const int r0 = split * per;
  const int r1 = min(n, r0 + per);
  const int nchunks = r1 > r0 ? (r1 - r0 + kNr - 1) / kNr : 0;
  const int qdim0 = rank == 0 ? 0 : kSlice;          // this CTA's share of the contraction
  const int qsteps = rank == 0 ? kSlice / 16 : (kD - kSlice) / 16;  // 16-dim MMA steps: 20 or 16

  if (tid == 0) {
    for (int s = 0; s < kBuf; s++) {
      tc::bar_init(&ax->kv_full[s], kProducers);
      tc::bar_init(&ax->kv_empty[s], 1);
    }
    tc::bar_init(&ax->s_full, 1);
    tc::bar_init(&ax->s_empty, kH);
    tc::bar_init(&ax->p_full, kH);
    tc::bar_init(&ax->pv_done, 1);
    tc::bar_init(&ax->x_full, 1);          // one local arm per chunk + kXBytes of bulk data from the peer
    tc::bar_init(&ax->x_empty, kH / 32);   // one remote arrive per peer softmax warp and chunk
    tc::bar_init(&ax->mma_idle, 1);
    tc::bar_init(&ax->q_full, 1);
    ax->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // armed for the 128 query rows copied below, before any copy is issued
    tc::bar_arrive_expect_tx(&ax->q_full, kH * (qsteps * 32));
  }
  if (warp == 0) tc::tmem_alloc<kTmemCols>(&ax->tmem_base);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = ax->tmem_base;

  // Query share -> fp16 -> tensor memory: softmax thread h copies head h's
  // share (one bulk copy of 640 or 512 bytes) into a staging row, then
  // writes it to lane h, columns kQCol + c holding dims 2c, 2c + 1.
  if (warp >= 4) {
    const int h = tid - 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    unsigned char* qst = sKV + h * kQStride;
    tc::bulk_load(qst, a.q + (static_cast<int64_t>(b) * kH + h) * kD + qdim0, qsteps * 32, &ax->q_full);
    if (!__all_sync(0xffffffffu, tc::bar_wait(&ax->q_full, 0, &ax->abort))) set_status(a.status, SKV_DEV_TIMEOUT);
#pragma unroll
    for (int c0 = 0; c0 < kSlice / 2; c0 += 32) {  // 32 columns = 64 dims per store
      if (c0 < qsteps * 8) {
        uint32_t r[32];
#pragma unroll
        for (int m = 0; m < 8; m++) {
          const uint4 w = *reinterpret_cast<const uint4*>(qst + 4 * c0 + 16 * m);
          r[4 * m] = bf16x2_to_f16x2(w.x);
          r[4 * m + 1] = bf16x2_to_f16x2(w.y);
          r[4 * m + 2] = bf16x2_to_f16x2(w.z);
          r[4 * m + 3] = bf16x2_to_f16x2(w.w);
        }
        tc::tmem_st32(tm + lane_base + kQCol + c0, r);
      }
    }
    tc::tmem_wait_st();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  tc::cluster_sync();  // the peer's barriers exist before any remote access
  volatile int* abort = &ax->abort;

  if (warp == 0) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0 && nchunks > 0) {
      const uint32_t aKV = tc::smem_addr(sKV), aP = tc::smem_addr(sP);
      constexpr uint32_t id_qk = tc::idesc_f16(kH, kNr, 0);
      constexpr uint32_t id_pv = tc::idesc_f16(kH, 256, 1);
      bool ok = true;
      for (int i = 0; ok && i <= nchunks; i++) {
        if (i < nchunks) {  // S(i) = Q . K(i)^T, once slot i%3 is full and S(i-1) was read
          const int s = i % kBuf;
          ok = tc::bar_wait(&ax->kv_full[s], (i / kBuf) & 1, abort);
          if (ok && i >= 1) ok = tc::bar_wait(&ax->s_empty, (i - 1) & 1, abort);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t kv = aKV + s * kKVBytes;
          for (int ks = 0; ks < qsteps; ks++) {
            const int dim = qdim0 + 16 * ks - rank * 256;  // dim within this CTA's tile
            tc::mma_f16_ts(tm + kSCol, tm + kQCol + 8 * ks,
                           tc::sw128_desc(kv + (dim >> 6) * (kNr * 128) + ((dim & 63) >> 4) * 32, 16, 1024), id_qk,
                           ks > 0);
          }
          tc::mma_commit(&ax->s_full);
        }
        if (i >= 1) {  // O += P(i-1) . V(i-1)
          const int j = i - 1, s = j % kBuf;
          ok = tc::bar_wait(&ax->p_full, j & 1, abort);
          if (!ok) break;
          tc::tc_fence_after();
          const uint32_t kv = aKV + s * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < 4; kk++)  // 16 rows per step; value dims are the tile's first 4 atoms
            tc::mma_f16(tm + kOCol, tc::sw128_desc(aP + kk * 32, 16, 1024),
                        tc::sw128_desc(kv + kk * 2048, kNr * 128, 1024), id_pv, j > 0 || kk > 0);
          tc::mma_commit(&ax->pv_done);
          tc::mma_commit(&ax->kv_empty[s]);
        }
      }
      // Nothing of this thread's may still be running when the tensor memory
      // is released (also after a wait that gave up).
      tc::mma_commit(&ax->mma_idle);
      if (!tc::bar_drain(&ax->mma_idle, 0, 4000000000ull)) set_status(a.status, SKV_DEV_TIMEOUT);
    }
  } else if (warp < 4) {
    // ---------------- row gather: fp8 -> fp16 swizzled tiles ----------------
    // Row ids of chunk i+1 are fetched while chunk i's rows are in flight.
    const int pt = tid - 32;
    auto row_of = [&](int i) -> int32_t {
      const int gi = r0 + i * kNr + pt;
      if (gi >= r1) return -1;
      const int64_t p = static_cast<int64_t>(b) * a.req_row_stride + a.rows[static_cast<int64_t>(b) * a.max_rows + gi];
      if (p < 0 || p >= a.n_pool_rows) {
        if (rank == 0) set_status(a.status, SKV_DEV_RANGE);
        return -1;
      }
      return static_cast<int32_t>(p);
    };
    if (pt < kNr && nchunks > 0) ax->prow[0][pt] = row_of(0);
    named_sync(1, kProducers);
    for (int i = 0; i < nchunks; i++) {
      const int s = i % kBuf;
      // The chunk's loads are issued before waiting for its slot (they only
      // need the row ids, which the producers keep for themselves).
      uint4 v[kPerProducer];
#pragma unroll
      for (int m = 0; m < kPerProducer; m++) {
        const int u = pt + m * kProducers;
        v[m] = make_uint4(0u, 0u, 0u, 0u);
        if (u < kNr * kPieces) {
          const int jr = u / kPieces, q = u % kPieces;
          const int32_t p = ax->prow[s][jr];
          if (p >= 0) v[m] = ld_nc16(a.pool + static_cast<int64_t>(p) * kD + rank * 256 + 16 * q);
        }
      }
      int32_t next = -1;
      float rsc = 0.f;
      bool have = false;
      if (pt < kNr) {
        const int32_t p = ax->prow[s][pt];
        have = p >= 0;
        if (have) rsc = a.row_scale ? a.row_scale[p] : 1.f;
        if (i + 1 < nchunks) next = row_of(i + 1);
      }
      const bool free_buf = i < kBuf || tc::bar_wait(&ax->kv_empty[s], ((i / kBuf) - 1) & 1, abort);
      if (!named_sync_and(1, kProducers, free_buf)) break;  // the same decision in every producer
      unsigned char* tile = sKV + s * kKVBytes;
#pragma unroll
      for (int m = 0; m < kPerProducer; m++) {
        const int u = pt + m * kProducers;
        if (u < kNr * kPieces) {
          const int jr = u / kPieces, q = u % kPieces;
          const int c0 = (q & 3) * 2;
          const uint2 e0 = tc::e4m3x4_to_f16x4(v[m].x), e1 = tc::e4m3x4_to_f16x4(v[m].y);
          const uint2 e2 = tc::e4m3x4_to_f16x4(v[m].z), e3 = tc::e4m3x4_to_f16x4(v[m].w);
          unsigned char* row = tile + (q >> 2) * (kNr * 128) + jr * 128;
          *reinterpret_cast<uint4*>(row + ((c0 ^ (jr & 7)) << 4)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (jr & 7)) << 4)) = make_uint4(e2.x, e2.y, e3.x, e3.y);
        }
      }
      if (pt < kNr) {
        ax->kl[s][pt] = have ? rsc * a.scale_log2 : 0.f;
        ax->madd[s][pt] = have ? 0.f : -INFINITY;
        ax->vsc[s][pt] = have ? rsc : 0.f;
        ax->prow[(i + 1) % kBuf][pt] = next;  // producers only; slot (i+1)%3 held chunk i-2, long done
      }
      tc::fence_async_smem();
      tc::bar_arrive(&ax->kv_full[s]);
      named_sync(1, kProducers);
    }
  } else {
    // ---------------- softmax + epilogue: thread = head ----------------
    const int h = tid - 128;
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    float* xin = sXin + h * kNr;
    float* xout = sXout + h * kNr;
    for (int i = 0; i < nchunks; i++) {
      const int s = i % kBuf;
      ok = __all_sync(0xffffffffu, tc::bar_wait(&ax->s_full, i & 1, abort));
      if (!ok) break;
      tc::tc_fence_after();
      uint32_t ra[32], rb[32];
      tc::tmem_ld32(tm + lane_base + kSCol, ra);
      tc::tmem_ld32(tm + lane_base + kSCol + 32, rb);
      tc::tmem_wait_ld();
      tc::tc_fence_before();
      tc::bar_arrive(&ax->s_empty);
      // This warp's 32 heads of partial logits: staged in shared memory, then
      // one bulk copy into the peer's buffer (which counts down the peer's
      // receive barrier); the peer's come into sXin the same way.
      if (h == 0) tc::bar_arrive_expect_tx(&ax->x_full, kXBytes);
      if (i >= 1) {
        if (lane == 0) tc::wait_bulk_read();  // the previous copy has left sXout
        ok = __all_sync(0xffffffffu, tc::bar_wait(&ax->x_empty, (i - 1) & 1, abort, true));
        if (!ok) break;
      }
#pragma unroll
      for (int c = 0; c < 16; c++) {
        const uint32_t* r = c < 8 ? &ra[4 * c] : &rb[4 * (c - 8)];
        *reinterpret_cast<float4*>(xout + 4 * (c ^ (h & 7))) =
            make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]), __uint_as_float(r[3]));
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int off = 32 * wq * kNr;  // this warp's 32 heads
        tc::bulk_copy_to_peer(sXin + off, sXout + off, 32 * kNr * 4, &ax->x_full, peer);
        tc::commit_bulk();
      }
      ok = __all_sync(0xffffffffu, tc::bar_wait(&ax->x_full, i & 1, abort));
      if (!ok) break;
      float x[64];
#pragma unroll
      for (int c = 0; c < 16; c++) {
        const float4 o = *reinterpret_cast<const float4*>(xin + 4 * (c ^ (h & 7)));
        const uint32_t* r = c < 8 ? &ra[4 * c] : &rb[4 * (c - 8)];
        x[4 * c] = __uint_as_float(r[0]) + o.x;
        x[4 * c + 1] = __uint_as_float(r[1]) + o.y;
        x[4 * c + 2] = __uint_as_float(r[2]) + o.z;
        x[4 * c + 3] = __uint_as_float(r[3]) + o.w;
      }
      __syncwarp();  // this warp has read its part of the peer's logits
      if (lane == 0) tc::bar_arrive_remote_relaxed(&ax->x_empty, peer);
      // logits in log2 units; eight independent max chains
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; k++) mp[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 16; c++) {
        const float4 f = *reinterpret_cast<const float4*>(&ax->kl[s][4 * c]);
        const float4 m = *reinterpret_cast<const float4*>(&ax->madd[s][4 * c]);
        x[4 * c] = fmaf(x[4 * c], f.x, m.x);
        x[4 * c + 1] = fmaf(x[4 * c + 1], f.y, m.y);
        x[4 * c + 2] = fmaf(x[4 * c + 2], f.z, m.z);
        x[4 * c + 3] = fmaf(x[4 * c + 3], f.w, m.w);
        mp[(2 * c) & 7] = fmaxf(mp[(2 * c) & 7], fmaxf(x[4 * c], x[4 * c + 1]));
        mp[(2 * c + 1) & 7] = fmaxf(mp[(2 * c + 1) & 7], fmaxf(x[4 * c + 2], x[4 * c + 3]));
      }
      const float mc = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      bool rescale = false;
      float alpha = 1.f;
      if (mc > m_ref + kRescaleLog2) {
        alpha = exp2f(m_ref - mc);
        rescale = i > 0;
        m_ref = mc;
      }
      if (i >= 1) {
        ok = __all_sync(0xffffffffu, tc::bar_wait(&ax->pv_done, (i - 1) & 1, abort));
        if (!ok) break;
        tc::tc_fence_after();
      }
      if (rescale) {
        for (int c0 = 0; c0 < 256; c0 += 32) {
          uint32_t o[32];
          tc::tmem_ld32(tm + lane_base + kOCol + c0, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; k++) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tc::tmem_st32(tm + lane_base + kOCol + c0, o);
        }
        tc::tmem_wait_st();
        l *= alpha;
      }
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 16; c++) {
        const float4 vf = *reinterpret_cast<const float4*>(&ax->vsc[s][4 * c]);
        const float p0 = tc::ex2_approx(x[4 * c] - m_use), p1 = tc::ex2_approx(x[4 * c + 1] - m_use);
        const float p2 = tc::ex2_approx(x[4 * c + 2] - m_use), p3 = tc::ex2_approx(x[4 * c + 3] - m_use);
        ls[c & 3] += (p0 + p1) + (p2 + p3);
        pk[2 * c] = pack_f16x2(p0 * vf.x, p1 * vf.y);
        pk[2 * c + 1] = pack_f16x2(p2 * vf.z, p3 * vf.w);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
#pragma unroll
      for (int c = 0; c < 8; c++)
        *reinterpret_cast<uint4*>(sP + h * 128 + ((c ^ (h & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      tc::fence_async_smem();
      tc::tc_fence_before();
      tc::bar_arrive(&ax->p_full);
    }
    if (lane == 0) tc::wait_bulk_done();  // this warp's copies into the peer have completed
    // epilogue: this CTA's 256 value dims of head h
    bool have_o = ok && nchunks > 0;
    if (have_o) {
      have_o = __all_sync(0xffffffffu, tc::bar_wait(&ax->pv_done, (nchunks - 1) & 1, abort));
      tc::tc_fence_after();
    }
    if (!ok || (nchunks > 0 && !have_o)) set_status(a.status, SKV_DEV_TIMEOUT);
    const bool merged = a.nsplit == 1;
    const float inv = (merged && l > 0.f) ? 1.f / l : 0.f;
    // Row h staged in shared memory (the ring and P buffer: the last value
    // product has completed, so no tensor-core read of them is pending); the
    // warp then writes its 32 rows out coalesced (one 1 KB row per step).
    unsigned char* ost = sKV + h * kOStride;
    for (int c0 = 0; c0 < 256; c0 += 32) {
      uint32_t o[32];
      if (have_o) {
        tc::tmem_ld32(tm + lane_base + kOCol + c0, o);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; k++) o[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        float4 v = make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]), __uint_as_float(o[k + 2]),
                               __uint_as_float(o[k + 3]));
        if (merged) v = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
        *reinterpret_cast<float4*>(ost + 4 * (c0 + k)) = v;
      }
    }
    if (a.cmerge) {  // merged with the other split after the cluster barrier below
      ax->mrow[h] = have_o ? m_ref : -INFINITY;
      ax->lrow[h] = have_o ? l : 0.f;
    }
    __syncwarp();
    for (int r = 0; !a.cmerge && r < 32; r++) {
      const int hr = 32 * wq + r;
      const unsigned char* src = sKV + hr * kOStride;
      float* drow = merged ? a.out + (static_cast<int64_t>(b) * kH + hr) * kDv + rank * 256
                           : a.ws_o + ((static_cast<int64_t>(b) * a.nsplit + split) * kH + hr) * kDv + rank * 256;
#pragma unroll
      for (int k = 0; k < 2; k++)
        *reinterpret_cast<float4*>(drow + 4 * (lane + 32 * k)) =
            *reinterpret_cast<const float4*>(src + 16 * (lane + 32 * k));
    }
    if (!merged && !a.cmerge && rank == 0) {
      float* ml = a.ws_ml + ((static_cast<int64_t>(b) * a.nsplit + split) * kH + h) * 2;
      ml[0] = have_o ? m_ref : -INFINITY;
      ml[1] = have_o ? l : 0.f;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc<kTmemCols>(tm);
  }
  tc::cluster_sync();  // the peer's copies into this CTA's shared memory are done; partials staged
  if (a.cmerge) {
    // Split sc of the cluster merges heads [64 sc, 64 sc + 64) of this CTA's
    // 256 value dims from its own staged rows and those of the CTA holding
    // the same dims for the other split (cluster rank crank ^ 2), in split
    // order -- the arithmetic of the merge kernel.
    const uint32_t other = crank ^ 2u;
    const int sc = static_cast<int>(crank >> 1);
    const unsigned char* rows0 = sKV;  // staged rows, head h at h * kOStride
    for (int e = tid; e < 64 * 64; e += kThreads) {
      const int h = 64 * sc + e / 64, dd = 4 * (e % 64);
      const unsigned char* own = rows0 + h * kOStride + 4 * dd;
      const float4 o_own = *reinterpret_cast<const float4*>(own);
      const float4 o_oth = tc::ld_remote16(own, other);
      const float m_own = ax->mrow[h], l_own = ax->lrow[h];
      const float m_oth = tc::ld_remote_f32(&ax->mrow[h], other), l_oth = tc::ld_remote_f32(&ax->lrow[h], other);
      // split 0 first
      const bool first = (crank >> 1) == 0;
      const float m0 = first ? m_own : m_oth, m1 = first ? m_oth : m_own;
      const float l0 = first ? l_own : l_oth, l1 = first ? l_oth : l_own;
      const float4 o0 = first ? o_own : o_oth, o1 = first ? o_oth : o_own;
      const float m = fmaxf(fmaxf(-INFINITY, m0), m1);
      const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - m), w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - m);
      float den = 0.f;
      den += w0 * l0;
      den += w1 * l1;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      acc.x += w0 * o0.x;
      acc.y += w0 * o0.y;
      acc.z += w0 * o0.z;
      acc.w += w0 * o0.w;
      acc.x += w1 * o1.x;
      acc.y += w1 * o1.y;
      acc.z += w1 * o1.z;
      acc.w += w1 * o1.w;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      *reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(b) * kH + h) * kDv + rank * 256 + dd) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    tc::cluster_sync();  // no CTA leaves while another still reads its shared memory
  }
}

// Splits of one (request, head) combined in split order.
__global__ __launch_bounds__(128) void mla_merge_kernel(const float* __restrict__ ws_o,
                                                        const float* __restrict__ ws_ml, int nsplit,
                                                        float* __restrict__ out) {
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  grid_dependency_wait();  // launched early: the attention kernel's partials are complete from here on
  const float* ml = ws_ml + (static_cast<int64_t>(b) * nsplit * kH + h) * 2;
  float m = -INFINITY;
  for (int s = 0; s < nsplit; s++) m = fmaxf(m, ml[static_cast<int64_t>(s) * kH * 2]);
  float den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; s++) {
    const float ms = ml[static_cast<int64_t>(s) * kH * 2], ls = ml[static_cast<int64_t>(s) * kH * 2 + 1];
    const float w = ms == -INFINITY ? 0.f : exp2f(ms - m);
    den += w * ls;
    const float4 o = *reinterpret_cast<const float4*>(
        ws_o + ((static_cast<int64_t>(b) * nsplit + s) * kH + h) * kDv + 4 * t);
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  *reinterpret_cast<float4*>(out + (static_cast<int64_t>(b) * kH + h) * kDv + 4 * t) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// Row splits per request: as many CTA pairs per request as one wave holds.
// A request of more than one 64-row chunk always gets at least two splits,
// merged inside one 4-CTA cluster when there are exactly two: a single split
// streaming several chunks through one CTA pair (and writing the normalised
// output itself) is never launched.  That shape has never been run on a GPU,
// and a variant of this kernel with two softmax threads per head stalled on
// it; with 39 or more requests on 152 SMs the two-split clusters simply take
// more than one wave.
int mla_splits(int B, int max_rows) {
  const int clusters = sm_count() / 2;
  int ns = B > 0 ? clusters / B : 1;
  const int chunks = (max_rows + kNr - 1) / kNr;
  if (ns > chunks) ns = chunks;
  if (ns < 1) ns = 1;
  if (ns == 1 && chunks > 1) ns = 2;
  return ns;
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_mla_workspace_size(int B, int max_rows) {
  if (B < 1 || max_rows < 1) return 0;
  const int ns = mla_splits(B, max_rows);
  if (ns <= 2) return 16;  // one split, or two merged inside their cluster
  return static_cast<size_t>(B) * ns * kH * (kDv + 2) * sizeof(float);
}

SKV_EXPORT int skv_sparse_attend_mla(int B, int Hq, int d, int dv, const uint16_t* q, const uint8_t* kv_pool,
                                     const float* row_scale, int64_t req_row_stride, int64_t n_pool_rows,
                                     const int32_t* rows, int max_rows, const int32_t* count, float softmax_scale,
                                     float* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     void* stream) {
  if (B < 0 || B > 65535 || max_rows < 1 || max_rows > 65536 || n_pool_rows < 1 || req_row_stride < 0)
    return SKV_EINVAL;
  if (Hq != kH || d != kD || dv != kDv) return SKV_EUNSUPPORTED;
  if (B == 0) return SKV_OK;
  if (!q || !kv_pool || !rows || !count || !out) return SKV_EINVAL;
  if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) || n_pool_rows > INT32_MAX) return SKV_EINVAL;
  if (static_cast<int64_t>(B - 1) * req_row_stride > INT32_MAX) return SKV_EINVAL;
  const int ns = mla_splits(B, max_rows);
  if (ns > 2) {
    if (!workspace || !aligned16(workspace) || workspace_bytes < skv_mla_workspace_size(B, max_rows))
      return SKV_ENOMEM;
  }
  static std::atomic<int> configured[kMaxDevices];
  if (smem_limit_once(configured, mla_kernel, kSmem) != SKV_OK) return SKV_EUNSUPPORTED;
  float* ws = static_cast<float*>(workspace);
  const bool cmerge = ns == 2;  // the two splits of a request merge inside one 4-CTA cluster
  MlaArgs a{q, kv_pool, row_scale, req_row_stride, n_pool_rows, rows, max_rows, count,
            softmax_scale * kLog2e, out, ws, ns > 1 ? ws + static_cast<size_t>(B) * ns * kH * kDv : nullptr, ns,
            cmerge ? 1 : 0, dev_status};
  cudaStream_t st = as_stream(stream);
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, ns, B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = cmerge ? 2 : 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla_kernel, a) != cudaSuccess) {
      cudaGetLastError();
      return SKV_ECUDA;
    }
  }
  if (ns > 1 && !cmerge) {
    // Launched as a programmatic dependent of the attention kernel: its
    // blocks take the SMs the attention grid leaves free and wait there
    // (grid_dependency_wait) until that grid has completed.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kH, B, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* wo = a.ws_o;
    const float* wml = a.ws_ml;
    if (cudaLaunchKernelEx(&cfg, mla_merge_kernel, wo, wml, ns, out) != cudaSuccess) {
      cudaGetLastError();
      return SKV_ECUDA;
    }
  }
  return launch_status();
}
