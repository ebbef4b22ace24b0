/*
 * lora.h -- C ABI of the GB300 composite multi-LoRA delta library
 * (libtclora.so).
 *
 * The library computes, for every token t of a mixed batch,
 *
 *     y_t  +=  sum over the pairs (i, alpha) of token t of  alpha * (x_t A_i[:, :k_i]) B_i[:k_i, :]
 *
 * with A_i in R^{d_in x r_max}, B_i in R^{r_max x d_out} held in a device
 * pool, k_i <= r_max the retained rank of adapter i, bf16 operands, fp32
 * accumulation and one round-to-nearest-even to bf16 of the result.
 *
 * Where the operation comes from:
 *  - the composite update dW = sum_i alpha_i B_i A_i^T, with weights fixed per
 *    request (LoRA-Soup style) or computed per token (MoE-LoRA style), served
 *    on one path: DyMerge-LoRA summary page, "Core idea" (paper Sec. 3.1, M1);
 *  - post-merge fusion: only the base factors are cached and all token-LoRA
 *    pairs of a batch are fused in one pass at kernel time, with the pairs
 *    reordered by LoRA id in a mapping stage: same page, "One-minute summary"
 *    and "Core idea" (paper Sec. 4.3, Algorithm 2, Figure 8);
 *  - one LoRA on one projection, W' = W + A B: ELORA summary page, Sec. 1.2
 *    (Eq. 1) and Sec. 1.3 (Eq. 2);
 *  - the retained-rank contract (a sorted factor prefix plus an effective
 *    rank k_m per module carried as device metadata) and the shrink /
 *    RowExpand split with phase-, rank- and shape-aware dispatch: LoRAForge
 *    summary page, "Key contributions" and "Approach" (1), (4), (5).
 *
 * Conventions (all entry points):
 *  - Row form: y (T x d_out) += x (T x d_in) . A (d_in x k) . B (k x d_out).
 *  - All device arrays are row-major and C-contiguous.  bf16 arrays are passed
 *    as void* holding IEEE bfloat16 bit patterns.  Device pointers must be
 *    16-byte aligned (any cudaMalloc'd base is).
 *  - lora_stream_t is a cudaStream_t (NULL = the legacy default stream).
 *    Every call is stream-ordered and asynchronous unless stated otherwise;
 *    the caller keeps every buffer it passes alive until the stream reaches
 *    the call.
 *  - Errors that the host can see (NULL pointers, sizes out of range, a
 *    mismatched object) return a status and launch nothing.  Errors that only
 *    the device can see (an adapter id outside the pool, an unregistered
 *    slot, a retained rank above r_max, malformed CSR offsets) make the
 *    offending pairs contribute nothing and set bits in the mapping's device
 *    status word, read with lora_mapping_status().  No kernel traps.
 *  - Objects are tied to the CUDA device that was current when they were
 *    created; call with that device current.
 *  - Host threads: distinct pools and mappings may be created and used from
 *    several threads at once (one-time set-up, such as the tensor-map encoder
 *    lookup, the kernels' launch attributes and the cached SM count, is kept
 *    per host thread or done once under a lock, so it is safe to race).  One
 *    object is used by one thread at a time.
 */
#ifndef TCLORA_LORA_H
#define TCLORA_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,
    LORA_ERR_OUT_OF_MEMORY = 2,
    LORA_ERR_CUDA = 3,
    LORA_ERR_BAD_ADAPTER = 4,
    LORA_ERR_NOT_SUPPORTED = 5
} lora_status;

/* Bits of the mapping's device status word (lora_mapping_status). */
#define LORA_DEV_BAD_ID 1       /* a pair's adapter id is outside [0, capacity) */
#define LORA_DEV_BAD_OFFSETS 2  /* CSR offsets not a row pointer for P pairs    */
#define LORA_DEV_UNREGISTERED 4 /* a pair names a slot never registered          */
#define LORA_DEV_BAD_RANK 8     /* a retained rank outside [0, r_max]            */
#define LORA_DEV_TIMEOUT 16     /* a bounded on-chip wait gave up                */

/* Limits of this implementation. */
#define LORA_MAX_RANK 64          /* r_max                                    */
#define LORA_MAX_CAPACITY 49152   /* adapters per pool / mapping key range    */
#define LORA_MAX_PAIRS (1 << 24)
#define LORA_MAX_TOKENS (1 << 24)
#define LORA_DIM_MULTIPLE 64      /* d_in and d_out must be multiples of this */

/* Execution paths of lora_delta_apply_path (LoRAForge page, "Approach" (5):
 * the path is fixed per phase, rank and shape). */
typedef enum {
    LORA_PATH_AUTO = 0,    /* the dispatch table chooses                       */
    LORA_PATH_SPLIT = 1,   /* segment shrink, then token-block RowExpand (PDL) */
    LORA_PATH_FUSED = 2,   /* one-launch decode kernel (small T)               */
    LORA_PATH_MMA = 3,     /* tensor-core prefill (many tokens per adapter)    */
    LORA_PATH_DECODE = 4   /* per-pair shrink, then per-token RowExpand (PDL)  */
} lora_path;

typedef void *lora_stream_t;
typedef struct lora_pool lora_pool;       /* opaque, library-owned device storage   */
typedef struct lora_mapping lora_mapping; /* opaque, library-owned device workspace */

/*
 * lora_pool_create: a device pool of `capacity` adapter slots, each holding
 * A_i (d_in x r_max) and B_i (r_max x d_out) in bf16 and a retained rank.
 * Storage is zeroed and every slot starts unregistered.  Synchronous.
 *   d_in, d_out : multiples of LORA_DIM_MULTIPLE, >= 64
 *   r_max       : 1..LORA_MAX_RANK
 *   capacity    : 1..LORA_MAX_CAPACITY
 *   out         : receives the pool; release with lora_pool_destroy.
 * Returns LORA_ERR_INVALID_ARG / LORA_ERR_NOT_SUPPORTED on bad sizes,
 * LORA_ERR_OUT_OF_MEMORY if the device allocation fails.
 * (DyMerge-LoRA page, "Core idea": only the base {A_i, B_i} are cached on the
 * GPU; ELORA page, Sec. 1.2.3: adapters are stored sliced along the rank.)
 */
lora_status lora_pool_create(int d_in, int d_out, int r_max, int capacity, lora_pool **out);

/*
 * lora_pool_register: copy adapter `slot`'s factors into the pool and set its
 * retained rank k (LoRAForge page, "Approach" (1): the factors are a sorted
 * prefix, k_m directions are live, padding beyond k_m is inert).
 *   A_dev : device bf16 [d_in][r_max] (A_i in R^{d_in x r})
 *   B_dev : device bf16 [r_max][d_out]
 *   k     : 0..r_max; rows/columns at index >= k are never read by the delta
 * The pool stores A transposed (r_max x d_in) so that the first k rows of
 * both factors are contiguous.  Stream-ordered; the caller keeps ownership of
 * A_dev and B_dev, which must stay valid until the stream reaches the call.
 * Re-registering a slot replaces it (order it after any delta still reading it).
 */
lora_status lora_pool_register(lora_pool *pool, int slot, const void *A_dev, const void *B_dev,
                               int k, lora_stream_t stream);

/* lora_pool_unregister: mark `slot` unregistered (stream-ordered). */
lora_status lora_pool_unregister(lora_pool *pool, int slot, lora_stream_t stream);

/* lora_pool_destroy: synchronise the device and free the pool.  NULL is a no-op. */
lora_status lora_pool_destroy(lora_pool *pool);

/*
 * lora_mapping_create: device workspace for batches of up to max_tokens
 * tokens and max_pairs (token, adapter) pairs over adapter ids in
 * [0, capacity).  Holds the adapter-ordered tuples, their inverse
 * permutation, the segments, the shrink output z (max_pairs x LORA_MAX_RANK
 * fp32) and the device status word.  Synchronous.
 */
lora_status lora_mapping_create(int max_tokens, int max_pairs, int capacity, lora_mapping **out);

/*
 * lora_build_mapping: the mapping stage of the fused kernel (DyMerge-LoRA
 * page, "Core idea" and "Reading map": tuples (i, j, k, w) built per batch,
 * reordered by LoRA id so that one CTA processes one adapter's tokens
 * together; paper Sec. 4.3, Algorithm 2, Figure 8).
 *   offsets_dev : int32 [T+1], CSR row pointer of each token's pair list
 *   ids_dev     : int32 [P], adapter id of pair p (CSR order)
 *   alpha_dev   : fp32 [P], weight of pair p
 *   T, P        : 0 <= T <= max_tokens, 0 <= P <= max_pairs
 * Result (device, inside the mapping): tuples (token, adapter, alpha, src=p)
 * ordered by (adapter, p) -- a stable sort on adapter id --, the inverse
 * permutation pos[p] (-1 for a pair left out), the distinct adapters in
 * ascending order with their segment starts.  Pairs with an id outside
 * [0, capacity) are left out and set LORA_DEV_BAD_ID; malformed offsets give
 * an empty mapping and set LORA_DEV_BAD_OFFSETS.  Clears the status word.
 * This call enqueues one kernel that copies the batch into the mapping in
 * CSR order (token, adapter, alpha per pair) and checks it; the decode path
 * reads only that copy.  The sorted tuples are produced from the copy by a
 * second kernel that the first apply needing them (the split, tensor-core
 * and fused paths, the ablation variants that use them, and
 * lora_mapping_export) enqueues before its own kernels; later calls on the
 * same build find them there (a device-side build counter decides, so this
 * also holds inside CUDA graphs; an eager call on the stream of an earlier
 * eager sort of the same build does not launch it at all, unless a build of
 * this mapping was ever enqueued into a graph, whose replays the host does
 * not see).
 * One mapping serves every lora_delta_apply on the same batch (all
 * projections and layers).  The input arrays need to stay valid only until
 * the stream reaches this call.
 */
lora_status lora_build_mapping(lora_mapping *m, const int32_t *offsets_dev, const int32_t *ids_dev,
                               const float *alpha_dev, int T, int P, lora_stream_t stream);

/*
 * lora_delta_apply: y += sum over each token's pairs of alpha (x A[:, :k]) B[:k, :]
 * (the composite delta above), in place, fused over all pairs of the batch.
 *   x_dev     : device bf16 [T][d_in]  (T of the last lora_build_mapping)
 *   y_dev     : device bf16 [T][d_out], read and written; must not alias x
 *   pool      : adapters; its capacity must equal the mapping's
 *   ranks_dev : device int32 [capacity] retained rank per slot, or NULL to use
 *               the ranks given at registration.  A value outside [0, r_max]
 *               sets LORA_DEV_BAD_RANK and that adapter contributes nothing.
 *   m         : a mapping built for this batch
 * Accumulates in fp32 and rounds once to bf16 (nearest even).  Chooses its
 * kernels with the dispatch table of lora_dispatch_choose.  Stream-ordered,
 * no host synchronisation, no allocation: safe to capture in a CUDA graph.
 */
lora_status lora_delta_apply(const void *x_dev, void *y_dev, const lora_pool *pool,
                             const int32_t *ranks_dev, const lora_mapping *m, lora_stream_t stream);

/*
 * lora_delta_apply_multi: lora_delta_apply for several projections of one
 * batch at once -- e.g. the q, k, v and o projections of a layer, each with
 * its own pool (any d_in, d_out, r_max) -- sharing one mapping.  The pages
 * apply LoRA to every dense projection of the model (DyMerge-LoRA page,
 * "What they did", paper Sec. 5.1) and build the token-LoRA mapping once per
 * batch (same page, "Core idea", Sec. 4.3); this entry point runs all the
 * projections' shrinks in one launch and all their expands in a second one.
 *   projs  : host array of n_proj descriptors; each x_dev / y_dev / pool /
 *            ranks_dev has the meaning and layout of lora_delta_apply's, and
 *            every pool's capacity must equal the mapping's
 *   n_proj : 1 .. LORA_MAX_PROJECTIONS
 * The projections' y buffers must not overlap one another or any x.
 * Result per projection: what lora_delta_apply on that projection gives on
 * the decode path -- the same shrink and the same (token, 256 columns)
 * expand, so the same bits, except where a single call takes the wide-rank
 * expand (r_max > 16 with few (token, column) items), whose summation order
 * differs (last-bit differences, within the stated tolerance).  Batches for
 * which the dispatch table picks the decode path for every projection, and
 * whose sum of round4(r_max) over the projections is at most 256, take the
 * two shared launches; other batches run one lora_delta_apply per
 * projection, in order.  Stream-ordered; no allocation.
 * Returns LORA_ERR_INVALID_ARG for NULL or mismatched arguments or aliased
 * outputs, LORA_ERR_NOT_SUPPORTED above LORA_MAX_PROJECTIONS.
 */
#define LORA_MAX_PROJECTIONS 8
typedef struct {
    const void *x_dev;
    void *y_dev;
    const lora_pool *pool;
    const int32_t *ranks_dev;
} lora_projection;
lora_status lora_delta_apply_multi(const lora_projection *projs, int n_proj, const lora_mapping *m,
                                   lora_stream_t stream);

/*
 * The pages' kernel ablation (DyMerge-LoRA page, "How far to trust it":
 * the fused kernel against Copy+SGMV and a naive for-loop, paper Sec. 5.4 -
 * 5.5, Figs. 14 and 16; pre-merging the composite weight, Figs. 3 - 4),
 * reproduced as baselines for timing.  Each computes the same result as
 * lora_delta_apply (fp32 accumulation, y rounded once) by the method named:
 *   LORA_ABLATION_NAIVE     : per adapter of the batch, a shrink launch over
 *                             its pairs and an expand launch adding into an
 *                             fp32 copy of y (the host reads the segments
 *                             back first: the call synchronises the stream);
 *   LORA_ABLATION_COPY_SGMV : gather x into adapter order (a row per pair),
 *                             segment shrink and expand into per-pair rows,
 *                             then add each token's rows back into y (the
 *                             host reads the valid pair count: synchronises);
 *   LORA_ABLATION_PREMERGE  : per token dW_t = sum alpha A[:, :k] B[:k, :]
 *                             (fp32, d_in x d_out), then y_t += x_t dW_t.
 * workspace_dev: device scratch of at least lora_ablation_workspace_bytes()
 * bytes for this batch (16-byte aligned, caller-owned).  Unusable adapters
 * contribute nothing but set no status bit.  Returns LORA_ERR_INVALID_ARG
 * for bad arguments or a short workspace, LORA_ERR_NOT_SUPPORTED for an
 * unknown variant.
 */
#define LORA_ABLATION_NAIVE 1
#define LORA_ABLATION_COPY_SGMV 2
#define LORA_ABLATION_PREMERGE 3
size_t lora_ablation_workspace_bytes(int variant, int T, int P, int d_in, int d_out, int r_max);
lora_status lora_delta_apply_ablation(const void *x_dev, void *y_dev, const lora_pool *pool,
                                      const int32_t *ranks_dev, const lora_mapping *m, int variant,
                                      void *workspace_dev, size_t workspace_bytes, lora_stream_t stream);

/* lora_delta_apply_path: lora_delta_apply with the execution path forced
 * (LORA_PATH_AUTO = the dispatch table).  Returns LORA_ERR_NOT_SUPPORTED if the
 * path cannot run this shape. */
lora_status lora_delta_apply_path(const void *x_dev, void *y_dev, const lora_pool *pool,
                                  const int32_t *ranks_dev, const lora_mapping *m, int path,
                                  lora_stream_t stream);

/*
 * lora_dispatch_choose: the dispatch table, host only (no device work).
 * Returns the lora_path that lora_delta_apply takes for T tokens, P pairs,
 * the given r_max, d_in and d_out.  (LoRAForge page, "Approach" (5): the
 * path fixed by phase, rank and shape.)  The tensor-core path from 8192
 * tokens at r_max <= 8, 3072 at r_max <= 16 and 384 above (batches that long
 * are taken for prefill chunks, whose tokens share adapters); otherwise the
 * decode path; the split path where neither takes the shape.  The thresholds
 * are the measured crossovers of a sweep of all paths over tokens, rank and
 * adapter sharing on GB300.
 */
int lora_dispatch_choose(int T, int P, int r_max, int d_in, int d_out);

/*
 * lora_delta_apply_host: one whole step from HOST buffers (pinned memory
 * recommended): copy offsets, ids, alpha, x and y to the device, build the
 * mapping, apply the delta and copy y back into y_host.  Device staging is
 * allocated inside the mapping on the first call for a given (d_in, d_out)
 * and reused after.  Stream-ordered: y_host is valid after the stream
 * synchronises.  Same element layouts as the device calls.
 * When all five host buffers are page-locked (device-addressable) and the
 * dispatch table picks the decode path, one copy kernel brings x into the
 * device staging (each byte crosses the host link once, overlapped by the
 * mapping stage) and the step's own kernels read the pair lists and y from
 * host memory and write y back there (no copy launch after the step);
 * other page-locked steps move the buffers with two launches of a copy
 * kernel that reads and writes host memory directly (one in, one out);
 * pageable buffers take one cudaMemcpyAsync each.  A step may take as x the
 * y of the step before it on the same stream.
 * A call that repeats the previous call's arguments exactly (pointers, T, P,
 * pool, ranks, stream) is captured into a CUDA graph of the whole step, and
 * later calls with those arguments replay it (one graph launch instead of
 * five to nine API calls); the buffers' contents may change between calls.  Every call
 * looks up again whether each buffer is page-locked and at which device
 * address; a replay happens only when that is unchanged since the capture.
 * Calls on a default stream, or on a stream that is being captured, always
 * run eagerly, as does a step whose capture fails (e.g. copies from
 * pageable memory).  The mapping holds the staging and the graph: calls
 * with one mapping must not run concurrently from several host threads.
 */
lora_status lora_delta_apply_host(const void *x_host, void *y_host, const int32_t *offsets_host,
                                  const int32_t *ids_host, const float *alpha_host, int T, int P,
                                  const lora_pool *pool, const int32_t *ranks_dev, lora_mapping *m,
                                  lora_stream_t stream);

/* lora_mapping_status: synchronise `stream` and return the device status word
 * (LORA_DEV_* bits) accumulated since the last lora_build_mapping. */
lora_status lora_mapping_status(const lora_mapping *m, lora_stream_t stream, int *device_error);

/*
 * lora_mapping_export: sort the mapping's current build if no apply has yet
 * (on `stream`), synchronise `stream` and copy the mapping into HOST
 * buffers (for checking it; any pointer may be NULL to skip that array):
 *   tok, adapter, alpha, src : [P_valid]   the ordered tuples
 *   pos                      : [P]         inverse permutation (-1 = left out)
 *   seg_adapter : [U], seg_start : [U+1]
 *   counts : int32 [3] = { U, P_valid, status word }
 */
lora_status lora_mapping_export(const lora_mapping *m, lora_stream_t stream, int32_t *tok,
                                int32_t *adapter, float *alpha, int32_t *src, int32_t *pos,
                                int32_t *seg_adapter, int32_t *seg_start, int32_t *counts);

/* lora_mapping_destroy: synchronise the device and free the mapping. */
lora_status lora_mapping_destroy(lora_mapping *m);

/* lora_status_string: a static description of a status code. */
const char *lora_status_string(lora_status s);

/* lora_version: the library version string. */
const char *lora_version(void);

/*
 * lora_delta_apply_noalloc: one whole batch -- the mapping, then the
 * segment shrink and the token-block RowExpand (the split path) -- with
 * every scratch array in one fixed, statically allocated device buffer of
 * LORA_NOALLOC_SCRATCH_BYTES, so the call allocates no device memory and
 * needs no lora_mapping.  The pages describe no such interface: it is an
 * operational variant of lora_build_mapping + lora_delta_apply_path(SPLIT).
 *
 * For callers that cannot allocate per call: a serving loop whose caching
 * allocator already holds the spare device memory (cudaMalloc would fail),
 * or code that must not call cudaMalloc / cudaFree, which may synchronise
 * the device.
 *   x_dev, y_dev, pool, ranks_dev : as for lora_delta_apply
 *   offsets_dev, ids_dev, alpha_dev, T, P : as for lora_build_mapping
 *   status_dev : NULL, or a device int32 that receives this call's
 *                LORA_DEV_* bits (stream-ordered)
 * Scratch for a batch: about P * (42 + 4 * round4(r_max)) + 64 * min(P,
 * capacity) + 8 * capacity + 4 * T bytes, in 256-byte aligned pieces.  A batch whose layout
 * exceeds LORA_NOALLOC_SCRATCH_BYTES returns LORA_ERR_NOT_SUPPORTED before
 * launching anything.  The scratch header (status word and counters) is
 * zeroed on the stream at the start of every call; every other scratch
 * array is written before it is read.
 * The first call on a device does set-up (looks up the buffer's device
 * address, sets kernel attributes); make it before any stream capture.
 * There is one buffer per device: calls whose work overlaps in time (on
 * different streams, or from several host threads) race on it and must be
 * serialised, e.g. by issuing them on one stream.
 */
#define LORA_NOALLOC_SCRATCH_BYTES (4 << 20)
lora_status lora_delta_apply_noalloc(const void *x_dev, void *y_dev, const lora_pool *pool,
                                     const int32_t *ranks_dev, const int32_t *offsets_dev,
                                     const int32_t *ids_dev, const float *alpha_dev, int T, int P,
                                     int32_t *status_dev, lora_stream_t stream);

/*
 * MoE-LoRA gating on the device: the step before the mapping in the sparse
 * (MoE-LoRA) scenario (DyMerge-LoRA page, MoE-LoRA scenario and code
 * release notes, paper Sec. 5.3 and Appendix A: each token weights its
 * request's adapters with a gate over padded, masked candidate lists, keeps
 * the top-k and renormalises their softmax weights).  The outputs are the
 * CSR pair lists lora_build_mapping takes, with P = T * top_k.
 *
 * lora_gate_logits: logits[t][e] = sum_d x[t][d] * Wg[req[t]][e][d]
 *   x_dev      : device bf16 [T][d_in] (the tokens' hidden states)
 *   wg_dev     : device bf16 [R][E][d_in], a router per request
 *   req_dev    : device int32 [T], the request of each token, in [0, R)
 *                (not checked: the caller's layout)
 *   logits_dev : device fp32 [T][E] (written); fp32 accumulation
 * d_in a multiple of 8, x and Wg 16-byte aligned.
 *
 * lora_gate_topk: per token, among the candidates e with cand[t][e] >= 0,
 * the top_k by logit (largest first; equal logits: the lower e first), with
 * alpha_i = exp(l_i - l_max) / sum over the kept of exp(l_j - l_max) -- the
 * softmax over all candidates renormalised over the kept ones, whose full
 * denominator cancels.
 *   logits_dev : device fp32 [T][E];  cand_dev : device int32 [T][E]
 *                (adapter id, or -1 for a padded slot)
 *   offsets_dev: device int32 [T+1] = t * top_k
 *   ids_dev, alpha_dev : device [T * top_k]; a token with fewer valid
 *                candidates repeats its best one with alpha 0 (a no-op
 *                pair); a token with none emits id -1 (which the mapping
 *                leaves out, setting LORA_DEV_BAD_ID)
 *   1 <= top_k <= min(E, 8), E <= 64 (else LORA_ERR_NOT_SUPPORTED).
 * Both are stream-ordered and allocate nothing.
 */
lora_status lora_gate_logits(const void *x_dev, const void *wg_dev, const int32_t *req_dev, int T, int E, int d_in,
                             float *logits_dev, lora_stream_t stream);
lora_status lora_gate_topk(const float *logits_dev, const int32_t *cand_dev, int T, int E, int top_k,
                           int32_t *offsets_dev, int32_t *ids_dev, float *alpha_dev, lora_stream_t stream);

/*
 * Batched recompression of a fleet of adapters (LoRAForge summary page,
 * "Key contributions" and "Approach" (2)-(3): FlashTSQR factor construction
 * and the two rank-allocation policies); it produces the sorted factor
 * prefixes and retained ranks k_m that lora_pool_register takes.
 *
 * lora_recompress: for M modules of one shape, dW_m = A_m B_m, computes
 * singular values sigma_m (descending) and balanced factors F_m, T_m with
 * F_m T_m = A_m B_m, F_m^T F_m = T_m T_m^T = diag(sigma_m), and the first k
 * directions equal to the rank-k truncated SVD -- via a tall-skinny QR of
 * A_m (row tiles as independent leaf QRs, then level-wise merges of the
 * triangular factors; Q is never formed), H = R B_m, and the
 * eigen-decomposition of H H^T (fp32 throughout).  Directions with
 * sigma^2 <= 1e-6 sigma_0^2 are dead: sigma 0, zero column / row.
 *   A_dev     : device bf16 [M][d_in][r]  (the pool's A layout per adapter)
 *   B_dev     : device bf16 [M][r][d_out]
 *   F_dev     : device fp32 [M][d_in][r];  T_dev : device fp32 [M][r][d_out]
 *   sigma_dev : device fp32 [M][r]
 *   workspace_dev: device scratch of lora_recompress_workspace_bytes(M, d_in, r)
 *   1 <= r <= LORA_MAX_RANK, r <= d_in.  Stream-ordered.
 *
 * lora_rank_allocate (host only): retained ranks k_m from the sigmas.
 *   sigma_host : [M][r_stride], each row descending (zeros: dead directions)
 *   rank_host  : original rank r_m;  cost_host : d_in + d_out of module m
 *   LORA_RANK_UNIFORM  : k_m = min(max(1, floor(r_m / d)), live directions)
 *                        (LoRAForge-U);
 *   LORA_RANK_SPECTRAL : the uniform policy's parameter budget
 *                        sum k_m cost_m spent greedily: every module keeps
 *                        min(floor_k, live) directions, then directions are
 *                        taken by sigma^2 / cost descending (ties: lower m,
 *                        then lower j) while they extend their module's
 *                        prefix and fit the budget (LoRAForge-S).
 */
#define LORA_RANK_UNIFORM 0
#define LORA_RANK_SPECTRAL 1
size_t lora_recompress_workspace_bytes(int M, int d_in, int r);
lora_status lora_recompress(const void *A_dev, const void *B_dev, int M, int d_in, int d_out, int r, float *F_dev,
                            float *T_dev, float *sigma_dev, void *workspace_dev, size_t workspace_bytes,
                            lora_stream_t stream);
lora_status lora_rank_allocate(const float *sigma_host, int M, int r_stride, const int32_t *rank_host,
                               const int32_t *cost_host, int policy, int d, int floor_k, int32_t *k_host);

/*
 * lora_diag_wait_expiry: diagnostic.  Every on-chip wait of the library is
 * bounded; this launches one kernel whose single wait can never be
 * satisfied, so that the expiry path can be observed: the wait gives up
 * after limit_ns, sets LORA_DEV_TIMEOUT and the kernel returns normally,
 * leaving the context usable.  (The pages have no counterpart: bounded
 * waits are this library's rule for any wait between CTAs.)
 *   kind      : 0 = an mbarrier phase with no arrival (the wait of the TMA
 *               pipelines), 1 = a counter in global memory that nothing
 *               increments (the wait of the cooperative kernels)
 *   limit_ns  : 1e3 .. 1e8 (1 us .. 100 ms)
 *   words_dev : device int32 [4]; words[1] must hold 0 for kind 1.  On
 *               return (stream-ordered): words[0] |= LORA_DEV_TIMEOUT,
 *               words[2] = 1 if the wait was satisfied else 0, words[3] =
 *               microseconds waited.
 * Returns LORA_ERR_INVALID_ARG for other kinds or limits.
 */
lora_status lora_diag_wait_expiry(int kind, long long limit_ns, int32_t *words_dev, lora_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TCLORA_LORA_H */
