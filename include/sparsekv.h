/*
 * sparsekv.h -- C ABI of libsparsekv.so, sparse long-context decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * One decode step of one attention layer, for a batch of requests:
 *   1. indexer score of every cached token (int4 rank-64 key sketch, fp32
 *      sketch, or bf16 indexer keys pooled by blocks of 4),
 *   2. deterministic top-k, one pick shared by every KV head of the layer,
 *   3. union with the sink and recent-tail tokens (or block expansion),
 *   4. exact attention over only the selected rows.
 * Sources (page title, section):
 *   [P1] "8 agents x 250K context on two 3090s: sparse KV decode with a
 *        rank-64 key sketch and a host-RAM tier", "What shipped".
 *   [P2] "vLLM's Hybrid HiSparse Triples Concurrent Requests on Million-Token
 *        Contexts", "Three residency states, one block pool".
 *   [P3] "You can offload most of Qwen3.8-Flash-Next's KV cache to RAM with
 *        little decode slowdown".
 *   [P4] "3.14M Context on 3x 3090: The Power of an Architecture That Puts KV
 *        Cache in Host RAM", sections "Why", "No Need to Rewrite the Kernel",
 *        "What Needs to Stay in VRAM".
 *
 * General rules for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise (for host-tier data
 *    pass the device alias returned by skv_host_register).  The caller owns
 *    every buffer; the library allocates nothing and never synchronises.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and contains no host-side decision that depends on device
 *    data, so a sequence of calls can be captured in a CUDA graph ([P2]: the
 *    decode path stays graph-capturable because nothing waits on a CPU-side
 *    decision; [P4]: capture survived host-resident KV).
 *  - Return value: SKV_OK, or an SKV_E* code.  Argument errors are detected on
 *    the host before anything is launched.  SKV_ECUDA means a launch failed
 *    (the CUDA error is left for cudaGetLastError-style inspection by the
 *    caller's runtime).
 *  - Errors that only the device can see (a NaN score, a row index out of
 *    range, a bounded wait that gave up) are OR-ed into the caller's int32
 *    `dev_status` word (SKV_DEV_* bits) when it is non-NULL; the kernel skips
 *    the offending access and carries on.  The caller reads the word after
 *    synchronising.  No kernel traps.
 *  - Scratch memory ("workspace") is caller-provided, sized by the matching
 *    *_workspace_size call, and must be zero-filled once before its first use.
 *    Every call that completes returns its counters and histograms to zero, so
 *    the workspace is ready for the next call without clearing; the rest is
 *    rewritten before it is read.  Calls that share a workspace must not
 *    overlap on the GPU.
 *  - bf16 / fp16 arguments are passed as uint16_t bit patterns.
 */
#ifndef SPARSEKV_H
#define SPARSEKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define SKV_OK 0
#define SKV_EINVAL 1        /* bad argument (null pointer, size, alignment)    */
#define SKV_EUNSUPPORTED 2  /* valid request this build does not implement     */
#define SKV_ECUDA 3         /* a CUDA runtime call or launch failed            */
#define SKV_ENOMEM 4        /* caller buffer too small                         */

/* ---- device status bits (OR-ed into *dev_status) -------------------------- */
#define SKV_DEV_NAN 1u       /* a score was NaN                                 */
#define SKV_DEV_RANGE 2u     /* a row / token index was out of range            */
#define SKV_DEV_TIMEOUT 4u   /* a bounded device-side wait gave up              */
#define SKV_DEV_COUNT 8u     /* a selection produced an unexpected row count    */

/* ---- enumerations ---------------------------------------------------------- */
/* Indexer modes of skv_index_score. */
#define SKV_SCORE_SKETCH_INT4 0   /* int4 key sketch x int8 folded query, int32 */
#define SKV_SCORE_SKETCH_F32 1    /* fp32 key sketch x fp32 folded query        */
#define SKV_SCORE_POOLED_BF16 2   /* bf16 pooled indexer keys x bf16 query      */

/* KV row encodings of skv_sparse_attend_decode. */
#define SKV_KV_BF16 0   /* bf16 K and V rows                                      */
#define SKV_KV_INT8 1   /* int8 K and V rows, one fp16 scale per (row, head) each  */

/* Returns the ABI version (incremented on any incompatible change). */
int skv_version(void);

/* Short English description of a status code (static storage). */
const char *skv_status_string(int status);

/* Number of streaming multiprocessors of the current device (0 on error). */
int skv_device_sm_count(void);

/* ========================================================================== */
/* a1: key sketch ([P1] "What shipped": each token is scored through a rank-64 */
/* key sketch held as int4; the basis is frozen, fitted once offline).        */
/* ========================================================================== */
/*
 * For every input token i and KV head h:
 *   s[j] = sum_{x=0}^{d-1} basis[x*r + j] * key[i][h][x]        (fp32)
 * With c != NULL the sketch is stored int4: code = clamp(rint(s[j] / c[h*r+j]),
 * -8, 7) (round half to even, IEEE division; c == 0 gives code 0), two codes
 * per byte, dim 2b in the low nibble and dim 2b+1 in the high nibble, heads
 * consecutive: an output row is Hkv*r/2 bytes.  With c == NULL the fp32 sketch
 * itself is stored: an output row is Hkv*r floats.
 *   keys     bf16 [n_tok][Hkv][d]
 *   basis    fp32 [d][r]  (column j is basis vector j)
 *   c        fp32 [Hkv][r] quantiser step, or NULL for the fp32 sketch
 *   out_rows int64 [n_tok] destination row of each token in `out`, or NULL
 *            (token i -> row i).  Used to append decode tokens in place.
 *   out      u8 [rows][Hkv*r/2] (int4) or fp32 [rows][Hkv*r]
 * Constraints: r == 64, d a multiple of 8 and <= 512, n_tok >= 0.
 * Rounding: the projection's summation order is the kernel's; an int4 code may
 * differ by one from a different summation only where s/c lies within a few
 * ulps of a half-integer.
 */
int skv_sketch_project(const uint16_t *keys, int64_t n_tok, int Hkv, int d, int r,
                       const float *basis, const float *c, const int64_t *out_rows,
                       void *out, void *stream);

/* ========================================================================== */
/* a2: folded query ([P1] "What shipped": one pick per layer is shared by all */
/* four KV heads; read as the sum of the per-head sketch scores, with the     */
/* query heads of a KV head's group (kv_head = g / (Hq/Hkv)) summed).         */
/* ========================================================================== */
/*
 * For request b, KV head h, sketch dim j:
 *   qp[b][h*r + j] = c[h*r+j] * sum_{g in group h} sum_x basis[x*r+j] * q[b][g][x]
 * (c omitted when NULL).  int8 mode (c != NULL): sigma[b] = max_m |qp[b][m]| /
 * 127, q8 = clamp(rint(qp / sigma), -127, 127), sigma == 0 gives zeros; out is
 * int8 [B][Hkv*r] and sigma_out fp32 [B] (may be NULL).  fp32 mode (c == NULL):
 * out is fp32 [B][Hkv*r] and sigma_out is unused.
 *   q     bf16 [B][Hq][d]
 * Constraints: r == 64, Hq % Hkv == 0, Hkv*r <= 1024, d <= 512.
 */
int skv_sketch_query(const uint16_t *q, int B, int Hq, int Hkv, int d, int r,
                     const float *basis, const float *c, void *out, float *sigma_out,
                     void *stream);

/* ========================================================================== */
/* a1 + a2 + int8 append fused: the per-layer work before the score scan.      */
/* ========================================================================== */
/*
 * For every request b: appends the current token -- its int4 key sketch
 * (skv_sketch_project with c) and its int8 K and V rows (skv_quantize_int8_rows)
 * -- at pool row new_rows[b], and folds the query into q8 / sigma
 * (skv_sketch_query with c), in one launch.  The folded query is computed as
 * c[h][j] * (basis^T (sum of the group's query heads))[j], the same linear map
 * as skv_sketch_query; codes may differ from it by one only at rounding ties.
 *   q       bf16 [B][Hq][d]         new_k, new_v  bf16 [B][Hkv][d]
 *   basis   fp32 [d][r]             c  fp32 [Hkv][r]
 *   new_rows int64 [B]: pool row of the current token of request b
 *   sketch  u8 [rows][Hkv*r/2]      k8, v8  int8 [rows][Hkv][d]
 *   k_scale, v_scale  fp16 [rows][Hkv]
 *   q8      int8 [B][Hkv*r]         sigma  fp32 [B] (may be NULL)
 *   workspace  skv_decode_prepare_workspace_size(B, Hkv, r) bytes, zero-filled
 *              before first use (its tickets return to zero).
 * Constraints: r == 64, Hq % Hkv == 0, d <= 512.
 */
size_t skv_decode_prepare_workspace_size(int B, int Hkv, int r);
int skv_decode_prepare(const uint16_t *q, const uint16_t *new_k, const uint16_t *new_v, int B,
                       int Hq, int Hkv, int d, int r, const float *basis, const float *c,
                       const int64_t *new_rows, uint8_t *sketch, int8_t *k8, uint16_t *k_scale,
                       int8_t *v8, uint16_t *v_scale, int8_t *q8, float *sigma, void *workspace,
                       size_t workspace_bytes, void *stream);

/* ========================================================================== */
/* a2': pooled indexer keys ([P3]: indexer keys compressed by ratio 4; [P4]   */
/* "What Needs to Stay in VRAM": keys pooled per block, kept in HBM).         */
/* ========================================================================== */
/*
 * pooled[b][blk][x] = bf16_rne( (((k0 + k1) + k2) + k3) / 4 ) with k_u =
 * keys[b][4*blk + u][x] in fp32, for blk in [first_block, first_block +
 * n_blocks) of every request b.  The caller passes only complete blocks.
 *   keys    bf16 [B][t_cap][D]       (t_cap tokens of capacity per request)
 *   pooled  bf16 [B][t_cap/4][D]
 * Constraints: ratio == 4, D a multiple of 8, first_block >= 0, and
 * 4*(first_block + n_blocks) <= t_cap.  The result is bit-exact.
 */
int skv_pool_keys(const uint16_t *keys, int B, int64_t t_cap, int D, int ratio,
                  int64_t first_block, int64_t n_blocks, uint16_t *pooled, void *stream);

/* ========================================================================== */
/* a3: indexer scores ([P1]: score every token through the sketch each decode */
/* step; [P4] "What Needs to Stay in VRAM": the indexer scores all blocks at  */
/* every step -- the only read that grows with the context).                  */
/* ========================================================================== */
/*
 * Candidates of request b (T = lengths[b]):
 *   sketch modes: tokens t in [S, T - W)  (sinks and tail do not compete);
 *   pooled mode : complete blocks blk in [0, T / ratio).
 * For each candidate, in the same row index space as `keys`:
 *   SKETCH_INT4 : score = sum_m q8[b][m] * code(t, m)   (exact int32)
 *   SKETCH_F32  : score = sum_m qp[b][m] * s[t][m]      (fp32)
 *   POOLED_BF16 : score = sum_x q_idx[b][x] * pooled[blk][x]  (fp32 accumulate)
 * and order_keys[b][t] = order key of the score: an unsigned 32-bit value
 * whose order is the score's order (int32: sign bit flipped; fp32: -0 taken
 * as +0, negative values bit-inverted, others with the sign bit set).  Entries
 * of non-candidates are not written.  A NaN fp32 score sets SKV_DEV_NAN.
 *   query  int8 [B][width] | fp32 [B][width] | bf16 [B][width]
 *   keys   u8 [B][n_cap][width/2] | fp32 [B][n_cap][width] | bf16 [B][n_cap][width]
 *   order_keys  u32 [B][n_cap]
 *   raw_scores  int32 (INT4) or fp32 (other modes) [B][n_cap], or NULL
 * width: Hkv*r for the sketch modes, the indexer dim for pooled mode.
 * Constraints: INT4 width in {128, 256, 512}; F32 width a multiple of 4 and
 * <= 1024; POOLED width == 128; ratio == 1 for sketch modes; for pooled
 * mode 1 <= ratio <= 64 (4: keys pooled by skv_pool_keys; 1: raw indexer
 * keys, one per token, as a latent-attention indexer scores them);
 * lengths[b] <= n_cap (sketch) or n_cap*ratio (pooled) (else SKV_DEV_RANGE
 * and the request is clamped).  Keys rows must be 16-byte aligned.
 */
int skv_index_score(int mode, int B, int width, const void *query, const void *keys,
                    int64_t n_cap, const int32_t *lengths, int ratio, int S, int W,
                    uint32_t *order_keys, void *raw_scores, int32_t *dev_status,
                    void *stream);

/* ========================================================================== */
/* a4: deterministic top-k with sink/tail union ([P1]: top 2048 + 64 sinks +  */
/* last 1024 tokens, deterministic radix select) and the pooled expansion     */
/* ([P4] "Why": sparse once the context exceeds 4*block_topk + 3 tokens).     */
/* ========================================================================== */
/*
 * For request b with T = lengths[b]:
 *  sketch (ratio == 1): if T <= S + W + k every token 0..T-1 is selected
 *    (dense fallback); otherwise the k best candidates of [S, T - W) by (order
 *    key descending, index ascending), and idx[b] = [0..S) ++ picks ascending
 *    ++ [T-W..T), count[b] = S + k + W.
 *  pooled (ratio > 1, S = W = 0): if T <= ratio*k + ratio - 1 every token;
 *    otherwise the k best complete blocks, each expanded to its `ratio` tokens
 *    in ascending order, then the tokens of the incomplete last block;
 *    count[b] = ratio*k + T % ratio.
 *   order_keys u32 [B][n_cap] (skv_index_score output; n_cap in candidates)
 *   idx        int32 [B][max_rows]   count int32 [B]
 *   workspace  skv_topk_workspace_size(B) bytes, zero-filled before first use.
 *              Each request's scratch sits at a fixed stride whatever B is and
 *              every call returns its counters to zero, so a workspace sized
 *              for B_max serves later calls with any B <= B_max, in any order.
 * Constraints: k >= 1; max_rows >= S + k + W (sketch) or ratio*k + ratio - 1
 * (pooled); B <= 4096.  The result is unique and bit-exact.
 */
size_t skv_topk_workspace_size(int B);
int skv_topk_select(int B, const uint32_t *order_keys, int64_t n_cap,
                    const int32_t *lengths, int k, int S, int W, int ratio,
                    int32_t *idx, int max_rows, int32_t *count, void *workspace,
                    size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * skv_topk_select_noalloc -- the same selection as skv_topk_select, for
 * callers that cannot give this library any scratch memory: for example an
 * engine that reserves all device memory for its own KV pools before decoding
 * starts and hands out no side buffers, or a latency-critical decode loop
 * that must not call cudaMalloc (an allocation can synchronise the device).
 * The pages have no counterpart of this call; it is a library convenience.
 * Its scratch is a fixed array compiled into the library (about 0.8 MB, held
 * by every device that loads the library until the process exits), enough for
 * at most 32 requests: B > 32 returns SKV_ENOMEM before anything is launched.
 * The call allocates nothing.  Its first call on a device looks up that
 * array's device address (with the device current) and caches it, so make
 * the first call on each device before any stream capture.  Every call reuses
 * the same array and clears the parts that must start at zero, so two calls
 * that overlap on the GPU (different streams, or different host threads on
 * one device) race and give wrong results: serialise them.
 * Arguments, results and errors are otherwise those of skv_topk_select.
 */
int skv_topk_select_noalloc(int B, const uint32_t *order_keys, int64_t n_cap,
                            const int32_t *lengths, int k, int S, int W, int ratio,
                            int32_t *idx, int max_rows, int32_t *count,
                            int32_t *dev_status, void *stream);

/* ========================================================================== */
/* a3 + a4 fused: one launch scores the candidates and selects the top-k.      */
/* ========================================================================== */
/*
 * Same result as skv_index_score followed by skv_topk_select with the same
 * arguments (the scores are computed by the same code, so the selection is
 * identical), in one cooperative launch: each CTA keeps its chunk's order
 * keys on chip, the CTAs of a request agree on the radix digits through
 * request-wide barriers, and the key range found during the scan lets the
 * digit passes skip the bits all keys share.  `order_keys` ([B][n_cap], may be
 * NULL) receives a copy of the keys of the candidates.
 *   workspace  skv_score_select_workspace_size(B) bytes, zero-filled before
 *              first use; each call returns its counters to zero and advances
 *              a per-request launch counter (the tag of the per-CTA records it
 *              writes).  Per-request scratch sits at a fixed stride, so a
 *              workspace sized for B_max serves later calls with any B <=
 *              B_max, in any order.
 * Errors: as skv_index_score and skv_topk_select; SKV_EUNSUPPORTED when B is
 * larger than the GPU can hold one resident CTA per request for, or when a
 * request's chunk of keys does not fit on chip (more than about 24K rows per
 * CTA); use the two separate calls then.  A barrier wait that runs out (it
 * cannot on a GPU running only this launch) sets SKV_DEV_TIMEOUT, after which
 * the workspace must be zero-filled again.
 */
size_t skv_score_select_workspace_size(int B);
int skv_score_select(int mode, int B, int width, const void *query, const void *keys,
                     int64_t n_cap, const int32_t *lengths, int ratio, int k, int S, int W,
                     int32_t *idx, int max_rows, int32_t *count, uint32_t *order_keys,
                     void *workspace, size_t workspace_bytes, int32_t *dev_status,
                     void *stream);

/*
 * skv_decode_select -- skv_decode_prepare followed by skv_score_select
 * (SKETCH_INT4) on the same sketch, in one cooperative launch: the per-layer
 * path before attention.  Every CTA folds its request's query itself (the
 * arithmetic of skv_decode_prepare, so the same q8 bits), and CTA h < Hkv of
 * each request appends head h of the current token (sketch codes, int8 K and
 * V rows at new_rows[b]).  Arguments as in those two calls; the sketch is
 * both the append target ([rows][Hkv*r/2], rows = b*n_cap + t) and the scored
 * keys ([B][n_cap][Hkv*r/2]).
 *   q8_out  int8 [B][Hkv*r] copy of the folded query, or NULL
 * The appended token must be in its request's recent tail (new_rows[b] =
 * b*n_cap + t with t >= T_b - W), as the newest token is: tail tokens are not
 * scored, so no CTA reads the row being written.  A row inside the scored
 * range sets SKV_DEV_RANGE.
 * Constraints: r == 64, W >= 1, Hkv*r in {128, 256, 512},
 * Hkv*d + d + 5*Hkv*r + 256 <= 8192; others as skv_score_select.
 */
int skv_decode_select(int B, int Hq, int Hkv, int d, int r, const uint16_t *q,
                      const uint16_t *new_k, const uint16_t *new_v, const float *basis,
                      const float *c, const int64_t *new_rows, uint8_t *sketch, int8_t *k8,
                      uint16_t *k_scale, int8_t *v8, uint16_t *v_scale, int64_t n_cap,
                      const int32_t *lengths, int k, int S, int W, int32_t *idx, int max_rows,
                      int32_t *count, int8_t *q8_out, void *workspace, size_t workspace_bytes,
                      int32_t *dev_status, void *stream);

/* ========================================================================== */
/* One decode step of one attention layer, every step of the path chained on   */
/* one stream: append the current token, fold the query, score and select,    */
/* resolve the rows, attend ([P1] "8 agents x 250K context on two 3090s ...",  */
/* "What shipped": the sparse step is captured as one CUDA-graph family;      */
/* [P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one block      */
/* pool": nothing in the step waits on a decision made on the CPU).           */
/* ========================================================================== */
/* Residency of the layer's int8 K/V rows (skv_layer_step.policy). */
#define SKV_RESIDENT 0    /* every token's rows in HBM: request b, token t at row b*n_cap + t */
#define SKV_HOST_CLOCK 1  /* int4 rows in a host tier; HBM holds per request S sink rows,    */
                          /* a ring of the last W tokens and Hs hot slots (windowed CLOCK)   */

/*
 * Arguments of skv_decode_layer_step (all pointers are device pointers;
 * host_rows is the device alias of the registered host tier).
 * Shapes: d == 256, r == 64, Hq % Hkv == 0, Hkv*r in {128, 256, 512}, k >= 1,
 * S >= 0, W >= 1, 1 <= lengths[b] <= n_cap.
 */
typedef struct skv_layer_step {
  int B, Hq, Hkv, d, r;
  int64_t n_cap;        /* token capacity per request (sketch and host-tier rows)      */
  int k, S, W;          /* top-k, sinks, recent tail                                   */
  float softmax_scale;
  int policy;           /* SKV_RESIDENT or SKV_HOST_CLOCK                              */
  int Hs;               /* hot slots per request (SKV_HOST_CLOCK; else unused)         */
  /* frozen per-layer artifacts */
  const float *basis;   /* fp32 [d][r]                                                 */
  const float *c;       /* fp32 [Hkv][r] sketch quantiser step                         */
  /* the layer's caches */
  uint8_t *sketch;      /* u8 [B][n_cap][Hkv*r/2] int4 key sketch                      */
  int8_t *k8, *v8;      /* int8 [B*R][Hkv][d], R = n_cap (SKV_RESIDENT) or S + W + Hs  */
  uint16_t *k_scale, *v_scale;  /* fp16 [B*R][Hkv]                                     */
  uint8_t *host_rows;   /* SKV_HOST_CLOCK: int4 host tier [B][n_cap][Hkv][2][d/2+d/32] */
  /* windowed-CLOCK state (SKV_HOST_CLOCK), as skv_resolve_rows_clock */
  int32_t *step;        /* int32 [2]: decode step, advanced by every call; ticket      */
  int32_t *slot_token;  /* int32 [B][Hs]  */
  uint8_t *ref;         /* u8 [B][Hs]     */
  int32_t *use_step;    /* int32 [B][Hs]  */
  int32_t *token_slot;  /* int32 [B][n_cap] */
  int32_t *hand;        /* int32 [B]      */
  /* per-step inputs */
  const uint16_t *q;                /* bf16 [B][Hq][d]                                 */
  const uint16_t *new_k, *new_v;    /* bf16 [B][Hkv][d]: the current token, T - 1       */
  const int32_t *lengths;           /* int32 [B]: T, the current token included         */
  /* outputs */
  int32_t *idx;         /* int32 [B][S+k+W]: the selection, ascending                  */
  int32_t *count;       /* int32 [B]                                                   */
  int32_t *n_miss;      /* int32 [B] hot-buffer misses (SKV_HOST_CLOCK), or NULL       */
  int8_t *q8_out;       /* int8 [B][Hkv*r] copy of the folded query, or NULL           */
  float *out;           /* fp32 [B][Hq][d] attention output                             */
} skv_layer_step;

/*
 * skv_decode_layer_step -- for every request b with T = lengths[b]:
 *  1. append the current token T - 1: its int4 sketch at sketch row
 *     b*n_cap + T - 1, its int8 K and V rows (skv_quantize_int8_rows
 *     encoding) at pool row b*n_cap + T - 1 (SKV_RESIDENT) or at the ring row
 *     b*(S+W+Hs) + S + (T-1) mod W (SKV_HOST_CLOCK, which also writes the
 *     token's int4 host row, skv_quantize_int4_rows encoding, at host row
 *     b*n_cap + T - 1); fold the query into int8 (skv_decode_prepare);
 *  2. score the candidates through the sketch and select the top k, with the
 *     sinks and the tail (skv_score_select, SKETCH_INT4; when that does not
 *     fit one launch, skv_index_score then skv_topk_select);
 *  3. SKV_HOST_CLOCK: resolve the selection through the hot buffer, fetching
 *     misses from the host tier (skv_resolve_rows_clock);
 *  4. attend over the selected int8 rows (skv_sparse_attend_decode).
 * The appended rows and the selection are those of the separate calls made
 * one after the other; with SKV_RESIDENT the attention takes each split's
 * share of the sinks and the tail before its share of the picks, so its
 * output equals theirs up to the order of the floating-point sums.  Every launch
 * goes to `stream`; the call has no host-side decision that depends on
 * device data, so a sequence of layer steps can be captured in a CUDA graph.
 *   workspace  skv_decode_layer_step_workspace_size(a) bytes, zero-filled
 *              before first use; every call leaves it ready for the next call
 *              with the same shapes (B, Hq, Hkv, n_cap, k, S, W, policy, Hs).
 *              Zero-fill it again before using it for other shapes.
 * Errors: SKV_EINVAL for null pointers, shapes outside the constraints, or a
 * short workspace (SKV_ENOMEM); the device status bits of the chained calls.
 */
size_t skv_decode_layer_step_workspace_size(const skv_layer_step *a);
int skv_decode_layer_step(const skv_layer_step *a, void *workspace, size_t workspace_bytes,
                          int32_t *dev_status, void *stream);

/* ========================================================================== */
/* KV row encoding (write path).                                               */
/* ========================================================================== */
/*
 * int8 rows with one fp16 scale per (row, head): scale = fp16_rne(max|x| /
 * 127) (fp32 division), code = clamp(rint(x / scale), -127, 127); a zero scale
 * gives zero codes.  Bit-exact.
 *   x          bf16 [n_rows][Hkv][d]
 *   out_rows   int64 [n_rows] destination row, or NULL (identity)
 *   q          int8 [rows][Hkv][d]     scale  fp16 [rows][Hkv]
 * Constraints: d a multiple of 8, <= 1024.
 */
int skv_quantize_int8_rows(const uint16_t *x, int64_t n_rows, int Hkv, int d,
                           const int64_t *out_rows, int8_t *q, uint16_t *scale,
                           void *stream);

/* ========================================================================== */
/* a6: exact attention over the selected rows ([P1]: exact int8 attention on  */
/* the picked tokens; [P4] "No Need to Rewrite the Kernel": each row is found */
/* by adding an offset to the base, layout [token][kv_head][dim]).            */
/* ========================================================================== */
/*
 * For request b, query head g (KV head h = g / (Hq/Hkv)) and the count[b]
 * selected rows i with physical row p_i = b*req_row_stride + rows[b][i]:
 *   logit_i = softmax_scale * sum_x q[b][g][x] * K(p_i, h, x)
 *   out[b][g][:] = sum_i softmax(logit)_i * V(p_i, h, :)
 * K(p, h, x) = k_pool[(p*Hkv + h)*d + x] (bf16), or int8 code times
 * k_scale[p*Hkv + h] (fp16) for SKV_KV_INT8; V likewise with v_pool/v_scale.
 * The split-K partial results are combined in a fixed order, so the output is
 * deterministic.  count[b] == 0 gives a zero output.
 *   q        bf16 [B][Hq][d]
 *   out      fp32 [B][Hq][d]
 *   workspace  skv_attend_workspace_size(...) bytes
 *   n_pool_rows  rows in the pools; a physical row outside [0, n_pool_rows)
 *            is skipped and sets SKV_DEV_RANGE
 * Constraints: d == 256, Hq % Hkv == 0, 1 <= max_rows <= 32768, n_pool_rows >= 1,
 * pools, out and workspace 16-byte aligned.
 * Accuracy: logits accumulate exact products in fp32; the probabilities are
 * rounded to fp16 (int8 rows) or split into two bf16 terms (bf16 rows) for
 * the tensor-core P.V product; max abs error well below 2e-3 for
 * unit-variance values.
 */
size_t skv_attend_workspace_size(int B, int Hq, int Hkv, int d, int max_rows);
int skv_sparse_attend_decode(int kv_kind, int B, int Hq, int Hkv, int d,
                             const uint16_t *q, const void *k_pool, const void *v_pool,
                             const uint16_t *k_scale, const uint16_t *v_scale,
                             int64_t req_row_stride, int64_t n_pool_rows,
                             const int32_t *rows, int max_rows, const int32_t *count,
                             float softmax_scale, float *out, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * skv_sparse_attend_mla -- a6 over latent (MLA) rows: 128 absorbed query
 * heads attend over fp8 e4m3 rows of d = 576 values (512 latent + 64 rope,
 * RoPE already applied); V is the first dv = 512 values of the same row
 * ([P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one block
 * pool": the kernel reads each selected row where the resolver placed it).
 * For request b, head g and the count[b] rows p_i = b*req_row_stride +
 * rows[b][i], with x_i = fp8 value times row_scale[p_i] (1 when row_scale is
 * NULL):
 *   logit_i = softmax_scale * sum_{j<576} q[b][g][j] * x_i[j]
 *   out[b][g][:] = sum_i softmax(logit)_i * x_i[0:512]
 *   q          bf16 [B][128][576] (converted to fp16 on chip: |q| <= 65504)
 *   kv_pool    fp8 e4m3 bytes [n_pool_rows][576]
 *   row_scale  fp32 [n_pool_rows] or NULL
 *   out        fp32 [B][128][512]
 *   workspace  skv_mla_workspace_size(B, max_rows) bytes (no zero-fill needed)
 * A row outside [0, n_pool_rows) is skipped and sets SKV_DEV_RANGE.  The
 * row splits are merged in a fixed order: the output is deterministic (two
 * splits merge inside one thread-block cluster and need no workspace).  A
 * request of more than 64 rows always runs as at least two splits (with more
 * than half as many requests as SMs, two per request in 4-CTA clusters, in
 * more than one wave); one CTA pair never streams several 64-row chunks on
 * its own.
 * Runs on the tcgen05 tensor cores with fp16 operands (fp8 -> fp16 exact),
 * fp32 accumulation; probabilities rounded to fp16.
 * Errors: SKV_EUNSUPPORTED unless Hq = 128, d = 576, dv = 512; SKV_EINVAL for
 * null or unaligned (16 B) q, kv_pool, out or workspace, max_rows outside
 * [1, 65536]; SKV_ENOMEM for a short workspace.
 */
size_t skv_mla_workspace_size(int B, int max_rows);
int skv_sparse_attend_mla(int B, int Hq, int d, int dv, const uint16_t *q, const uint8_t *kv_pool,
                          const float *row_scale, int64_t req_row_stride, int64_t n_pool_rows,
                          const int32_t *rows, int max_rows, const int32_t *count,
                          float softmax_scale, float *out, void *workspace, size_t workspace_bytes,
                          int32_t *dev_status, void *stream);

/* ========================================================================== */
/* a5: resolve the selected tokens to pool rows.  RESIDENT is the identity    */
/* (attention's req_row_stride addressing); the two calls below resolve       */
/* through a hot buffer in front of a host tier.                              */
/* ========================================================================== */
/*
 * skv_resolve_rows_clock -- windowed CLOCK over a host int4 tier ([P1] "What
 * shipped": the main KV cache is int4 in host RAM -- 64-dim groups, fp16
 * scales, 272 B per token-head -- and the GPU keeps the sketch, the sinks, the
 * recent tail and a 2.5 % hot buffer managed by windowed CLOCK; rows fetched
 * from the host are dequantised back to int8 rows).
 *
 * Per request b (one CTA each), with T = lengths[b] and the count[b] selected
 * tokens idx[b][i] (ascending, unique, as skv_topk_select writes them):
 *   sink  t < S          -> row t
 *   tail  t >= T - W     -> row S + (t mod W)   (the recent-token ring)
 *   pick  S <= t < T - W -> row S + W + slot, slot from the CLOCK:
 *     1. a pick whose token has a slot is a hit: ref = 1, use_step = step;
 *     2. the misses, in ascending token order, sweep the hand: a slot used
 *        in this step is skipped; an empty slot or one with ref == 0 is taken
 *        (its previous token loses it); a slot with ref == 1 gets ref = 0 and
 *        the hand moves on.  A taken slot gets the token, ref = 1, use_step =
 *        step, and the token's host row is fetched through host_rows,
 *        requantised to int8 (x = code * group scale, exact in fp32; s8 =
 *        fp16(max|x| / 127); q = clamp(rint(x / s8), +-127); zero s8 gives
 *        zero codes) and written to the slot's pool rows, every head, K and V.
 * Row ids are relative to the request: physical row = b*req_row_stride + row,
 * as skv_sparse_attend_decode reads them.
 *   state (device, caller-owned, per request; start: slot_token = -1, ref = 0,
 *   use_step = -1, token_slot = -1, hand = 0):
 *     slot_token int32 [B][Hs]   ref u8 [B][Hs]   use_step int32 [B][Hs]
 *     token_slot int32 [B][t_cap]   hand int32 [B]
 *   host_rows  u8 [B][t_cap][Hkv][2][d/2 + d/32] -- per token and head the K
 *              then the V vector in skv_quantize_int4_rows layout (136 B each
 *              for d = 256, 1088 B per token at Hkv = 4); the device alias of
 *              registered host memory (skv_host_register) or device memory
 *   k8, v8     int8 [B*req_row_stride][Hkv][d]; k_scale, v_scale fp16
 *              [B*req_row_stride][Hkv]: the request's pool (sinks, tail ring,
 *              hot slots); only hot-slot rows of misses are written
 *   rows_out   int32 [B][max_rows]; n_miss int32 [B] (misses placed; -1 when
 *              the request has more picks than slots)
 *   step       int32 [2] (device): step[0] = this call's decode step (>= 0),
 *              read by every CTA and advanced by one when the call completes
 *              (so a captured graph replays with a fresh step); step[1] = 0, a
 *              ticket the call returns to zero
 *   workspace  skv_resolve_workspace_size(B, max_rows) bytes (the miss list
 *              passed from the state pass to the fetch pass; no zero-fill)
 * Two launches: one CTA per request runs the state machine and lists the
 * misses, then one warp per miss fetches and requantises its host row.
 * Errors: SKV_EINVAL for bad sizes, null pointers, a req_row_stride below
 * S + W + Hs or unaligned pools; SKV_EUNSUPPORTED unless d is 256, 512, 768
 * or 1024, Hs <= 16384, max_rows <= 8192 and a token's host row (2 Hkv
 * vectors) is at most 5120 bytes; SKV_ENOMEM for a short workspace.  On the device: a token outside
 * [0, T) gives row -1 and SKV_DEV_RANGE; more picks than slots leave the state
 * unchanged, give row -1 for every pick and set SKV_DEV_COUNT.
 */
/* Scratch bytes for either resolver call below. */
size_t skv_resolve_workspace_size(int B, int max_rows);

int skv_resolve_rows_clock(int B, int64_t t_cap, const int32_t *lengths, int S, int W, int Hkv,
                           int d, int Hs, const int32_t *idx, int max_rows, const int32_t *count,
                           int32_t *step, int32_t *slot_token, uint8_t *ref, int32_t *use_step,
                           int32_t *token_slot, int32_t *hand, const uint8_t *host_rows,
                           int8_t *k8, int8_t *v8, uint16_t *k_scale, uint16_t *v_scale,
                           int64_t req_row_stride, int32_t *rows_out, int32_t *n_miss,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           void *stream);

/*
 * skv_resolve_rows_lru -- mixed residency behind a block table with an LRU
 * hot buffer ([P2] "Three residency states, one block pool": resident tokens
 * are read in place, hot tokens are read and refresh their LRU entry, a miss
 * copies one row from pinned host memory into an LRU slot; "What it composes
 * with": the hot buffer holds 2 x top-K rows).  One fused kernel, one CTA per
 * request.
 * Per request b and selected token t (ascending, unique):
 *   block_table[b][t / page] = p >= 0  -> row p*page + t mod page (in place)
 *   else a hot hit (token_slot[b][t] = s >= 0) -> row hot(b) + s, stamp = step
 *   else a miss: the misses, in ascending token order, take the slots NOT
 *   touched in this step with the smallest (stamp, slot index); the old token
 *   loses the slot; row_bytes are copied from host + (b*t_cap + t)*row_bytes
 *   to pool row hot(b) + s; stamp = step.
 * hot(b) = hot_base + b*hot_stride.  Row ids are absolute pool rows
 * (attention with req_row_stride = 0).
 *   state: stamp int64 [B][n_slots] (-1 empty), slot_token int32
 *          [B][n_slots] (-1 none), token_slot int32 [B][t_cap] (-1 none),
 *          order int32 [B][n_slots]: the slots by ascending (stamp, slot),
 *          maintained by the call (start: 0, 1, ..., n_slots - 1, since all
 *          stamps start at -1), so the victims are read off its front instead
 *          of sorting every step
 *   block_table int32 [B][n_pages]; host u8 [B][t_cap][row_bytes] (device
 *   alias); pool u8 [n_pool_rows][row_bytes]
 *   step   int32 [2] (device), as for skv_resolve_rows_clock: step[0] is the
 *          decode step, advanced by one when the call completes; step[1] = 0
 *   workspace  skv_resolve_workspace_size(B, max_rows) bytes (miss list)
 * Two launches: the state pass (one CTA per request), then one warp per miss
 * copies the host row.
 * Errors: SKV_EINVAL for bad sizes, null or unaligned pointers, row_bytes not
 * a multiple of 16, a hot buffer past n_pool_rows; SKV_EUNSUPPORTED for
 * n_slots > 8192 or max_rows > 8192; SKV_ENOMEM for a short workspace.  On the device: bad tokens give row -1
 * and SKV_DEV_RANGE; fewer untouched slots than misses leave the misses
 * unresolved (row -1), set n_miss[b] = -1 and SKV_DEV_COUNT.
 */
int skv_resolve_rows_lru(int B, int64_t t_cap, const int32_t *lengths, int page,
                         const int32_t *block_table, int64_t n_pages, int64_t hot_base,
                         int64_t hot_stride, int n_slots, int32_t *step, int64_t *stamp,
                         int32_t *slot_token, int32_t *token_slot, int32_t *order, const uint8_t *host,
                         uint8_t *pool, int64_t row_bytes, int64_t n_pool_rows,
                         const int32_t *idx, int max_rows, const int32_t *count,
                         int32_t *rows_out, int32_t *n_miss, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, void *stream);
/*
 * skv_resolve_rows_lru_leased -- the same, with the hot buffer made of blocks
 * leased from the pool ([P2] "Three residency states, one block pool": a hot
 * buffer page is an ordinary KV-cache block, leased from the same pool as the
 * resident pages): slot s of request b is pool row
 *   hot_blocks[b][s / page] * page + s mod page,
 * hot_blocks int32 [B][ceil(n_slots / page)] (see skv_residency_lease_hot).  A
 * slot whose block is negative or past n_pool_rows gives row -1 and
 * SKV_DEV_RANGE (its miss is not copied).
 */
int skv_resolve_rows_lru_leased(int B, int64_t t_cap, const int32_t *lengths, int page,
                                const int32_t *block_table, int64_t n_pages, const int32_t *hot_blocks,
                                int n_slots, int32_t *step, int64_t *stamp, int32_t *slot_token,
                                int32_t *token_slot, int32_t *order, const uint8_t *host, uint8_t *pool,
                                int64_t row_bytes, int64_t n_pool_rows, const int32_t *idx, int max_rows,
                                const int32_t *count, int32_t *rows_out, int32_t *n_miss, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * skv_quantize_int4_rows -- host-tier row encoding ([P1]: int4 with 64-dim
 * groups and fp16 scales, 272 B per token-head for K and V).  Per (row, head)
 * vector of d dims: for each 64-dim group, scale = fp16_rne(max|x| / 7) (fp32
 * division), code = clamp(rint(x / scale), -8, 7) (zero scale: zero codes);
 * bytes [0, d/2) hold the codes (byte i: dim 2i in the low nibble, 2i+1 in
 * the high nibble, two's complement), then d/64 fp16 scales.  Bit-exact.
 *   x        bf16 [n_rows][Hkv][d] (device)
 *   out      vector (t, h) at out + orow*token_pitch + h*head_pitch, orow =
 *            out_rows[t] (int64, device) or t when out_rows is NULL; out may
 *            be a host alias
 * Constraints: d in {256, 512, 768, 1024}; head_pitch >= d/2 + d/32;
 * token_pitch >= Hkv*head_pitch; pitches and out 4-byte aligned.
 */
int skv_quantize_int4_rows(const uint16_t *x, int64_t n_rows, int Hkv, int d,
                           const int64_t *out_rows, uint8_t *out, int64_t token_pitch,
                           int64_t head_pitch, void *stream);

/*
 * skv_stream_read -- reads `bytes` at `src` (device memory or a host alias)
 * with 16-byte loads and XORs the words into *sink: the probe that measures
 * the bandwidth a zero-copy gather can reach.  grid = 0 picks 2 CTAs per SM.
 * Errors: SKV_EINVAL for a null pointer, bytes not a multiple of 16 or src
 * not 16-byte aligned.
 */
int skv_stream_read(const void *src, size_t bytes, unsigned long long *sink, int grid,
                    void *stream);

/*
 * skv_gather_read -- reads the n rows rows[i] (int64, device) of row_bytes
 * each at base + rows[i] * row_bytes (device memory or a host alias), one
 * warp per row with every load of the row in flight at once, and XORs the
 * words into *sink: the probe for the access pattern of the host-tier
 * fetches (scattered rows of about a kilobyte), whose rate on registered
 * host memory depends on how many rows are read at once and on how much
 * host memory is registered, unlike a streaming read.
 * Errors: SKV_EINVAL for null pointers, n < 0, row_bytes not a multiple of
 * 16, or base not 16-byte aligned.
 */
int skv_gather_read(const void *base, const int64_t *rows, int n, int64_t row_bytes,
                    unsigned long long *sink, void *stream);

/* ========================================================================== */
/* Chunked sparse prefill ([P4] "3.14M Context on 3x 3090 ...", "The Downside */
/* to Keep in Mind": every prefill token picks its own top blocks, so the     */
/* loops are swapped -- the history is staged chunk by chunk into a small HBM */
/* buffer once, every query of the prefill chunk attends to its own picks     */
/* inside it, and the partial softmax states are merged).                     */
/* ========================================================================== */
/*
 * skv_prefill_index_scores -- pooled indexer scores of a chunk of prefill
 * queries that share one request's pooled keys:
 *   order_keys[i][blk] = order key of sum_x q_idx[i][x] * pooled[blk][x]
 * (fp32 accumulate of bf16 products, the POOLED_BF16 key map of
 * skv_index_score) for every query i < nq and block blk < n_blocks; entries
 * blk >= n_blocks are not written.  skv_topk_select with B = nq, lengths[i] =
 * (position of query i) + 1 and ratio 4 then gives every query its causal
 * selection.  The products are summed in tensor-core tiles, so a score agrees
 * with skv_index_score's to fp32 rounding.  A NaN score sets SKV_DEV_NAN.
 *   q_idx       bf16 [nq][128]           pooled  bf16 [n_blocks][128]
 *   order_keys  u32 [nq][key_stride]
 * Constraints: key_stride >= n_blocks and even; q_idx, pooled 16-byte
 * aligned, order_keys 8-byte aligned.  Errors: SKV_EINVAL otherwise.
 */
int skv_prefill_index_scores(int nq, const uint16_t *q_idx, const uint16_t *pooled,
                             int64_t n_blocks, uint32_t *order_keys, int64_t key_stride,
                             int32_t *dev_status, void *stream);

/*
 * skv_prefill_attend -- exact attention of each query of a prefill chunk over
 * its own selected tokens, loops swapped: the history below n_tokens is taken
 * chunk by chunk, each chunk's K and V rows copied once into the staging
 * buffers; one launch attends every query head to the query's selected
 * tokens inside the chunk and merges the partial softmax state (running max
 * m, sum l, accumulator acc) into `state`; a last launch writes out = acc / l.
 * When the sources are device-readable (device memory, or host memory
 * registered with skv_host_register) the buffers are used as two halves of
 * chunk_tokens / 2 rows and the launch that attends one half also copies the
 * next chunk into the other, overlapping the copies with the attention;
 * otherwise each chunk of chunk_tokens rows goes in with cudaMemcpyAsync on
 * `stream` before its launch.  For
 * query i and query head g (KV head g / (Hq / Hkv)) the result is
 *   out[i][g] = sum_{t in S_i} softmax_t(scale * q[i][g] . k[t]) v[t],
 * S_i = idx[i][0 .. count[i]), which is what skv_sparse_attend_decode gives
 * for one request with those rows, to fp32 rounding.  Host-link bytes per call:
 * n_tokens * Hkv * d * 4 when the sources are host memory, independent of nq.
 *   q              bf16 [nq][Hq][d]
 *   k_src, v_src   bf16 [n_tokens][Hkv][d]: host memory registered with
 *                  skv_host_register (HOST pointer), or device memory
 *   k_stage, v_stage  bf16 [chunk_tokens][Hkv][d], device, caller-owned
 *   idx            int32 [nq][max_rows], each row ascending
 *   count          int32 [nq]
 *   state          fp32 [nq][Hq][d + 4] scratch (no initial contents needed)
 *   out            fp32 [nq][Hq][d]; a query with count 0 gets zeros
 * A selected token >= n_tokens sets SKV_DEV_RANGE and is skipped.
 * Constraints: d == 256, Hq % Hkv == 0, Hq / Hkv <= 32, chunk_tokens >= 1;
 * q, stages 16-byte aligned.
 */
int skv_prefill_attend(int nq, int Hq, int Hkv, int d, const uint16_t *q, const uint16_t *k_src,
                       const uint16_t *v_src, int64_t n_tokens, uint16_t *k_stage,
                       uint16_t *v_stage, int64_t chunk_tokens, const int32_t *idx, int max_rows,
                       const int32_t *count, float softmax_scale, float *state, float *out,
                       int32_t *dev_status, void *stream);

/* ========================================================================== */
/* Pressure-driven residency ([P2] "vLLM's Hybrid HiSparse ...", "Three       */
/* residency states, one block pool": KV stays on the GPU while there is room */
/* and gives up residency page by page as the pool runs short; completed      */
/* prefix pages are copied to host memory ahead of need).                     */
/* ========================================================================== */
/*
 * The residency manager is host state (not thread-safe; one per block pool):
 * the pool's free blocks and, per request slot, one entry per page of `page`
 * tokens -- a pool block, or -1, a placeholder whose rows live only in host
 * memory.  That table is the `block_table` of skv_resolve_rows_lru (copy it
 * to the device with skv_residency_block_table + cudaMemcpyAsync).  Rules:
 *  - a page may be released only after its host copy was issued: completed
 *    resident pages are listed by skv_residency_pending, copied with
 *    skv_materialize_pages and then marked with skv_residency_mark_copied;
 *  - release picks, among the releasable pages (resident, copied, neither the
 *    request's newest page nor among its last `tail_pages` pages), the oldest
 *    page of the request that holds the most resident pages (ties: the lowest
 *    slot);
 *  - taking a block when none is free releases one page that way; the call
 *    fails with SKV_ENOMEM when nothing is releasable;
 *  - hot buffers are leased from the same pool (skv_residency_lease_hot): a
 *    block freed by one request can become another request's hot capacity;
 *  - a request added with host_prefix = 1 (a prefix that exists only in host
 *    memory) starts with placeholders for its complete pages; a partial last
 *    page gets a block whose first rows must be brought in (listed by
 *    skv_residency_fills, copied by skv_fill_pages, then marked with
 *    skv_residency_mark_filled) before anything is appended into that page:
 *    the fill copies the whole page.
 * Every call returns SKV_OK or SKV_EINVAL (bad slot, page or size) /
 * SKV_ENOMEM (out array or pool too small).
 */
typedef struct skv_residency skv_residency;
#define SKV_RESIDENCY_FULL 0   /* every page of the request is resident          */
#define SKV_RESIDENCY_MIXED 1  /* some pages are placeholders                     */
#define SKV_RESIDENCY_NONE 2   /* no page is resident                             */
int skv_residency_create(int n_blocks, int page, int max_requests, int64_t max_pages, int tail_pages,
                         skv_residency **out);
void skv_residency_destroy(skv_residency *r);
/* Starts slot b with n_tokens tokens: every page resident (host_prefix = 0) or
 * placeholders (host_prefix = 1). */
int skv_residency_add(skv_residency *r, int b, int64_t n_tokens, int host_prefix);
/* Ends slot b; its blocks return to the pool. */
int skv_residency_remove(skv_residency *r, int b);
/* Appends n tokens to slot b; a token that opens a page takes a block. */
int skv_residency_append(skv_residency *r, int b, int64_t n);
/* Complete resident pages of slot b without a host copy (ascending). */
int skv_residency_pending(const skv_residency *r, int b, int32_t *pages, int max_out, int *n_out);
int skv_residency_mark_copied(skv_residency *r, int b, const int32_t *pages, int n);
/* Resident pages of slot b whose first rows must come from host memory. */
int skv_residency_fills(const skv_residency *r, int b, int32_t *pages, int max_out, int *n_out);
int skv_residency_mark_filled(skv_residency *r, int b, const int32_t *pages, int n);
/* Leases n_pages blocks as slot b's hot buffer (releasing pages under the rule
 * above when none is free) and writes their numbers to blocks[0 .. n_pages);
 * they stay leased until skv_residency_remove.  A second lease for the same
 * slot is SKV_EINVAL. */
int skv_residency_lease_hot(skv_residency *r, int b, int n_pages, int32_t *blocks);
/* Releases up to n_wanted pages under the rule above; released[2i], [2i+1] =
 * (slot, page); *n_out of them. */
int skv_residency_reclaim(skv_residency *r, int n_wanted, int32_t *released, int *n_out);
/* The block table, int32 HOST array [max_requests][max_pages] (-1: placeholder
 * or unused). */
int skv_residency_block_table(const skv_residency *r, int32_t *table);
/* SKV_RESIDENCY_* of slot b, or -1 for a free slot. */
int skv_residency_state(const skv_residency *r, int b);
int skv_residency_free_blocks(const skv_residency *r);

/*
 * skv_materialize_pages / skv_fill_pages -- whole-page copies between the
 * pool and the host tier, one CTA per listed page: materialize writes the
 * rows of a resident page to the host (the copy ahead of need), fill brings
 * a page's host rows into its block.  Page (b, p) = pages[2j], pages[2j+1]:
 * pool rows block_table[b][p] * page + r, host rows b * t_cap + p * page + r,
 * r < page.  A page out of range, or not resident, sets SKV_DEV_RANGE and is
 * skipped.
 *   pages        int32 [n][2] (device)   block_table int32 [B][n_pages]
 *   pool         u8 [n_pool_rows][row_bytes]
 *   host         u8 [B][t_cap][row_bytes] (the host tier's device alias)
 * Constraints: row_bytes a multiple of 16; pool and host 16-byte aligned.
 */
int skv_materialize_pages(int n, const int32_t *pages, int B, int page, const int32_t *block_table,
                          int64_t n_pages, const uint8_t *pool, int64_t row_bytes,
                          int64_t n_pool_rows, uint8_t *host, int64_t t_cap, int32_t *dev_status,
                          void *stream);
int skv_fill_pages(int n, const int32_t *pages, int B, int page, const int32_t *block_table,
                   int64_t n_pages, uint8_t *pool, int64_t row_bytes, int64_t n_pool_rows,
                   const uint8_t *host, int64_t t_cap, int32_t *dev_status, void *stream);

/* ========================================================================== */
/* Host tier ([P4] "No Need to Rewrite the Kernel": allocate with anonymous    */
/* mmap, cudaHostRegister(ptr, n, PORTABLE | MAPPED), use the device pointer). */
/* ========================================================================== */
/*
 * Page-locks `bytes` of existing host memory at `host` (HOST pointer, owned by
 * the caller) for every device and returns in *dev_alias the device pointer
 * through which kernels read it zero-copy.  Synchronous; not for the hot path.
 */
int skv_host_register(void *host, size_t bytes, void **dev_alias);
/* Undoes skv_host_register.  The caller ensures no kernel still reads it. */
int skv_host_unregister(void *host);

#ifdef __cplusplus
}
#endif

#endif /* SPARSEKV_H */
