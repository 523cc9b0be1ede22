// layer.cu -- one decode step of one attention layer, every step of the path
// chained on one stream (skv_decode_layer_step).
//
// [P1] "8 agents x 250K context on two 3090s ...", "What shipped": per layer
// the current token is appended (int8 rows, int4 sketch, and with the host
// tier its int4 host row), every cached token is scored through the sketch,
// the top 2048 are unioned with 64 sinks and the last 1024 tokens, rows that
// left HBM come back through the windowed-CLOCK hot buffer, and exact int8
// attention runs on the picked rows; the sparse step is one CUDA-graph
// family.  [P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one
// block pool": nothing in the step waits on a CPU-side decision.
//
// The step is the composition of the library's entry points on one stream:
// the launches are exactly those of the separate calls, and the workspace is
// theirs laid end to end.
#include "common.cuh"
#include "fold.cuh"

namespace skv {

int launch_prepare(const uint16_t* q, const uint16_t* new_k, const uint16_t* new_v, int B, int Hq, int Hkv, int d,
                   const float* basis, const float* c, const fold::Append& ap, uint8_t* sketch, int8_t* k8,
                   uint16_t* k_scale, int8_t* v8, uint16_t* v_scale, int8_t* q8, float* sigma, void* workspace,
                   cudaStream_t st);
bool score_select_fits_int4(int width, int B, int64_t n_cap);
struct KnownRows {
  const int32_t* lengths;
  int S, W, k;
};
size_t attend_workspace_bytes(int kv_kind, int B, int Hq, int Hkv, int max_rows, const KnownRows* known);
int launch_attend(int kv_kind, int B, int Hq, int Hkv, const uint16_t* q, const void* k_pool, const void* v_pool,
                  const uint16_t* k_scale, const uint16_t* v_scale, int64_t req_row_stride, int64_t n_pool_rows,
                  const int32_t* rows, int max_rows, const int32_t* count, float softmax_scale, float* out,
                  void* workspace, size_t workspace_bytes, int32_t* dev_status, const KnownRows* known,
                  cudaStream_t st);

namespace {

inline size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// The workspace laid out region by region (each 256-byte aligned).
struct StepWs {
  size_t q8, prep, sel, keys, res, rows, miss, att, total;
  bool fused;
};

bool shapes_ok(const skv_layer_step& a) {
  if (a.B < 1 || a.B > 65535 || a.d != 256 || a.r != fold::kRank || a.Hq <= 0 || a.Hkv <= 0 || a.Hq % a.Hkv)
    return false;
  const int width = a.Hkv * a.r;
  if (width != 128 && width != 256 && width != 512) return false;
  if (a.k < 1 || a.S < 0 || a.W < 1 || a.n_cap < 1 || a.n_cap > INT32_MAX) return false;
  if (a.policy != SKV_RESIDENT && a.policy != SKV_HOST_CLOCK) return false;
  if (a.policy == SKV_HOST_CLOCK && (a.Hs < a.k || a.Hs > 16384)) return false;
  return static_cast<int64_t>(a.S) + a.k + a.W <= 8192;
}

StepWs plan(const skv_layer_step& a) {
  StepWs w{};
  const int max_rows = a.S + a.k + a.W;
  const int width = a.Hkv * a.r;
  size_t off = 0;
  w.q8 = off;
  off += up256(static_cast<size_t>(a.B) * width);
  w.prep = off;
  off += up256(skv_decode_prepare_workspace_size(a.B, a.Hkv, a.r));
  w.fused = score_select_fits_int4(width, a.B, a.n_cap);
  w.sel = off;
  off += up256(w.fused ? skv_score_select_workspace_size(a.B) : skv_topk_workspace_size(a.B));
  w.keys = off;
  if (!w.fused) off += up256(static_cast<size_t>(a.B) * a.n_cap * sizeof(uint32_t));
  w.res = w.rows = off;
  if (a.policy == SKV_HOST_CLOCK) {
    off += up256(skv_resolve_workspace_size(a.B, max_rows));
    w.rows = off;
    off += up256(static_cast<size_t>(a.B) * max_rows * sizeof(int32_t));
    w.miss = off;
    off += up256(static_cast<size_t>(a.B) * sizeof(int32_t));
  }
  w.att = off;
  // resident rows: the attention takes the sinks and the tail before the
  // selection is complete (its known-rows plan)
  const KnownRows known{a.lengths, a.S, a.W, a.k};
  off += up256(attend_workspace_bytes(SKV_KV_INT8, a.B, a.Hq, a.Hkv, max_rows,
                                      a.policy == SKV_RESIDENT ? &known : nullptr));
  w.total = off;
  return w;
}

}  // namespace
}  // namespace skv

using namespace skv;

SKV_EXPORT size_t skv_decode_layer_step_workspace_size(const skv_layer_step* a) {
  if (!a || !shapes_ok(*a)) return 0;
  return plan(*a).total;
}

SKV_EXPORT int skv_decode_layer_step(const skv_layer_step* ap, void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* stream) {
  if (!ap || !shapes_ok(*ap)) return SKV_EINVAL;
  const skv_layer_step& a = *ap;
  if (!a.basis || !a.c || !a.sketch || !a.k8 || !a.v8 || !a.k_scale || !a.v_scale || !a.q || !a.new_k ||
      !a.new_v || !a.lengths || !a.idx || !a.count || !a.out || !workspace)
    return SKV_EINVAL;
  const bool host = a.policy == SKV_HOST_CLOCK;
  if (host && (!a.host_rows || !a.step || !a.slot_token || !a.ref || !a.use_step || !a.token_slot || !a.hand ||
               (reinterpret_cast<uintptr_t>(a.host_rows) & 3)))
    return SKV_EINVAL;
  if (!aligned16(workspace)) return SKV_EINVAL;
  const StepWs w = plan(a);
  if (workspace_bytes < w.total) return SKV_ENOMEM;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t st = as_stream(stream);
  const int max_rows = a.S + a.k + a.W;
  const int width = a.Hkv * a.r;
  const int64_t R = host ? static_cast<int64_t>(a.S) + a.W + a.Hs : a.n_cap;  // pool rows per request
  int8_t* q8 = reinterpret_cast<int8_t*>(ws + w.q8);

  // 1. append the current token, fold the query
  fold::Append app{};
  app.lengths = a.lengths;
  app.n_cap = a.n_cap;
  app.kv_stride = R;
  app.S = a.S;
  app.W = a.W;
  app.ring = host ? 1 : 0;
  app.host4 = host ? a.host_rows : nullptr;
  int rc = launch_prepare(a.q, a.new_k, a.new_v, a.B, a.Hq, a.Hkv, a.d, a.basis, a.c, app, a.sketch, a.k8,
                          a.k_scale, a.v8, a.v_scale, q8, nullptr, ws + w.prep, st);
  if (rc != SKV_OK) return rc;
  if (a.q8_out && cudaMemcpyAsync(a.q8_out, q8, static_cast<size_t>(a.B) * width, cudaMemcpyDeviceToDevice, st) !=
                      cudaSuccess) {
    cudaGetLastError();
    return SKV_ECUDA;
  }

  // 2. score + select
  if (w.fused) {
    rc = skv_score_select(SKV_SCORE_SKETCH_INT4, a.B, width, q8, a.sketch, a.n_cap, a.lengths, 1, a.k, a.S, a.W,
                          a.idx, max_rows, a.count, nullptr, ws + w.sel, skv_score_select_workspace_size(a.B),
                          dev_status, stream);
  } else {
    uint32_t* keys = reinterpret_cast<uint32_t*>(ws + w.keys);
    rc = skv_index_score(SKV_SCORE_SKETCH_INT4, a.B, width, q8, a.sketch, a.n_cap, a.lengths, 1, a.S, a.W, keys,
                         nullptr, dev_status, stream);
    if (rc == SKV_OK)
      rc = skv_topk_select(a.B, keys, a.n_cap, a.lengths, a.k, a.S, a.W, 1, a.idx, max_rows, a.count, ws + w.sel,
                           skv_topk_workspace_size(a.B), dev_status, stream);
  }
  if (rc != SKV_OK) return rc;

  // 3. resolve through the hot buffer (host tier)
  const int32_t* rows = a.idx;
  if (host) {
    int32_t* r = reinterpret_cast<int32_t*>(ws + w.rows);
    int32_t* n_miss = a.n_miss ? a.n_miss : reinterpret_cast<int32_t*>(ws + w.miss);
    rc = skv_resolve_rows_clock(a.B, a.n_cap, a.lengths, a.S, a.W, a.Hkv, a.d, a.Hs, a.idx, max_rows, a.count,
                                a.step, a.slot_token, a.ref, a.use_step, a.token_slot, a.hand, a.host_rows, a.k8,
                                a.v8, a.k_scale, a.v_scale, R, r, n_miss, ws + w.res,
                                skv_resolve_workspace_size(a.B, max_rows), dev_status, stream);
    if (rc != SKV_OK) return rc;
    rows = r;
  }

  // 4. attention over the selected rows; with resident rows the sinks and
  // the tail (known from the lengths) are attended while the selection is
  // still finishing
  const KnownRows known{a.lengths, a.S, a.W, a.k};
  const KnownRows* kr = host ? nullptr : &known;
  return launch_attend(SKV_KV_INT8, a.B, a.Hq, a.Hkv, a.q, a.k8, a.v8, a.k_scale, a.v_scale, R,
                       static_cast<int64_t>(a.B) * R, rows, max_rows, a.count, a.softmax_scale, a.out, ws + w.att,
                       attend_workspace_bytes(SKV_KV_INT8, a.B, a.Hq, a.Hkv, max_rows, kr), dev_status, kr, st);
}
