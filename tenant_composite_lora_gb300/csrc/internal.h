// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "lora.h"

namespace tcl {

// Shrink tile: at most SHRINK_TT pairs (tokens) of one adapter segment.
constexpr int SHRINK_TT = 8;
constexpr int SHRINK_THREADS = 256;
constexpr int SHRINK_RING_BYTES = 64 * 1024;   // split path (beside an expand CTA)
constexpr int SHRINK_MIN_ENTRY = 12 * 64 * 2;  // a 64-element chunk of the largest unit
constexpr int SHRINK_ROUND_TILES = 1024;       // tile records scanned per round
constexpr int SHRINK_MAX_INFLIGHT = 8;

// Expand (RowExpand) tile: W in {32, 64, 128} output columns x a token block
// of tb tokens (tb * W <= EXP_TILE_ELEMS) x one of ng segment groups (a
// cluster); jobs of at most EXP_JP pairs of one segment.
constexpr int EXP_TILE_ELEMS = 8192;
constexpr int EXP_JP = 16;
constexpr int EXP_THREADS = 256;
constexpr int EXP_MAX_JOBS = 256;
constexpr int EXP_WIN_PAIRS = 1024;
constexpr int EXP_B_BYTES = 48 * 1024;
constexpr int EXP_Z_BYTES = 12 * 1024;
constexpr int EXP_SMEM_MAX = 136 * 1024;

struct ExpandPlan {
    int tb, w, ng;
};

constexpr int MAP_THREADS = 1024;
constexpr int MAP_SMEM_BYTES = 200 * 1024;
// Pools whose per-warp histograms do not fit in shared memory (one warp's
// row plus two per-bin arrays above MAP_SMEM_BYTES) keep them in global
// memory, MAP_GHIST_WARPS rows of `capacity` words plus the two per-bin arrays.
constexpr int MAP_GHIST_WARPS = 8;
// Words of global histogram scratch a mapping over `capacity` ids needs (0: none).
int map_global_hist_words(int capacity);
// Scratch words of the several-CTA sort of long batches (0: pools too large for it).
int map_wide_sort_words(int capacity);

// Ranks of pools up to this capacity are staged in shared memory by the
// apply kernels (one coalesced read instead of a dependent lookup).
constexpr int RANK_TAB_MAX = 2048;

// Header words of the mapping (device int32).
// HDR_BAR, HDR_BAR_BASE, HDR_EXIT: grid-barrier counters of the fused kernel.
// HDR_NMTILES: tensor-core shrink tiles (MMA_TM pairs of one segment).
// HDR_EPOCH, HDR_DEXIT: launches of the fused decode kernel since the mapping
// was built, and its CTAs that have exited in the current launch.
// HDR_BUILD: builds of this mapping (advanced by the CSR stage); HDR_SORTED:
// the build whose tuples the sort stage last produced.  HDR_U, HDR_PVALID,
// HDR_NTILES and HDR_NMTILES belong to the sort stage.  HDR_CSR_DONE,
// HDR_CSR_FLAGS: the several-CTA CSR stage's finished CTAs and their status
// bits, zero between builds (its last CTA writes the status and clears them).
// HDR_SORT_DONE: the several-CTA sort's counting CTAs that have finished,
// zero between sorts (its last CTA clears it); HDR_SORT_GO: 1 when its
// counting kernel prepared this launch's scatter, 0 when it found the build
// sorted already (the scatter's own decision, which its first CTA's update
// of HDR_SORTED cannot change under its other CTAs).
enum { HDR_U = 0, HDR_PVALID = 1, HDR_STATUS = 2, HDR_NTILES = 3, HDR_T = 4, HDR_BAR = 5, HDR_BAR_BASE = 6,
       HDR_EXIT = 7, HDR_NMTILES = 8, HDR_EPOCH = 9, HDR_DEXIT = 10, HDR_BUILD = 11, HDR_SORTED = 12,
       HDR_CSR_DONE = 13, HDR_CSR_FLAGS = 14, HDR_SORT_DONE = 15, HDR_SORT_GO = 16, HDR_WORDS = 17 };

// Tensor-core (tcgen05) prefill path: tiles of MMA_TM rows (pairs of one
// segment for the shrink, consecutive tokens for the expand).
constexpr int MMA_TM = 128;
// Dispatch: batches of at least this many tokens take the tensor-core path,
// by rank class (r_max <= 8, <= 16, larger): the measured crossovers of the
// decode and tensor-core paths on prefill-like batches (runs of consecutive
// tokens sharing their adapters), between the swept sizes 4096 / 8192,
// 2048 / 3250 (the sparse prefill workload) and 256 / 384 tokens.
constexpr int MMA_FROM_R8 = 8192;
constexpr int MMA_FROM_R16 = 3072;
constexpr int MMA_FROM_R64 = 384;

// Fused decode kernel: one CTA per SM; dynamic shared memory = the expand
// layout + an entry ring of at most FUSED_RING_MAX bytes (less if the
// device's per-block limit minus the kernel's static shared memory is lower).
constexpr int FUSED_RING_MAX = 96 * 1024;

struct PoolDev {
    const __nv_bfloat16 *At;  // [capacity][r_max][d_in]
    const __nv_bfloat16 *B;   // [capacity][r_max][d_out]
    const int32_t *reg_rank;  // [capacity], -1 = unregistered
    int d_in, d_out, r_max, capacity;
};

// The mapping on the device.  The CSR stage fills toff, pc, calpha and the
// header's status; the sort stage the ordered tuples and everything after them.
struct MapDev {
    int32_t *tok, *adapter, *src, *pos;  // [max_pairs]
    float *alpha;                        // [max_pairs]
    int32_t *seg_adapter, *seg_start;    // [capacity], [capacity+1]
    int4 *tile;                          // [max_pairs] shrink tiles {adapter, q0, n, segment}
    int32_t *tile_tok;                   // [max_pairs][SHRINK_TT] tokens of each tile's pairs
    int32_t *hdr;                        // [HDR_WORDS]
    int4 *mtile;                         // [mma_tile_bound] tensor-core shrink tiles {adapter, q0, n, segment}
    int32_t *toff;                       // [max_tokens+1] copy of the batch's CSR offsets
    int2 *pc;                            // [max_pairs] per CSR pair: {token, adapter}, adapter -1 if left out
    float *calpha;                       // [max_pairs] per CSR pair: alpha
    int32_t *zcnt;                       // [max_pairs] per CSR pair: z row groups written (fused decode)
    float *z;                            // [max_pairs][Z_ROW_FLOATS] shrink output: a row per sorted
                                         // pair (split, tensor-core paths) or per CSR pair (decode)
    float *partial;                      // [partial_ctas][EXP_TILE_ELEMS] fused-kernel tiles
    int partial_ctas;
    int32_t *ghist;                      // [map_global_hist_words(capacity)] or null: mapping
                                         // histograms of pools too large for shared memory
    int32_t *gsort;                      // [map_wide_sort_words(capacity)] or null: the
                                         // several-CTA sort's per-CTA bin counts and per-bin arrays
};

// Launchers (each returns cudaGetLastError()).
// The mapping's CSR stage (every build) and sort stage (before a path that
// reads the sorted tuples; it does nothing when the current build is sorted);
// launch_build_mapping enqueues both.
cudaError_t launch_map_csr(const MapDev &m, const int32_t *offsets, const int32_t *ids, const float *alpha, int T,
                           int P, int capacity, cudaStream_t st);
cudaError_t launch_map_sort(const MapDev &m, int T, int P, int capacity, cudaStream_t st);
cudaError_t launch_build_mapping(const MapDev &m, const int32_t *offsets, const int32_t *ids,
                                 const float *alpha, int T, int P, int capacity, int max_pairs,
                                 cudaStream_t st);
cudaError_t launch_shrink(const __nv_bfloat16 *x, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int P, int grid, cudaStream_t st);

// Floats per pair in the mapping's z buffer: one projection uses the
// first round4(r_max); several projections applied in one launch place
// their columns side by side (at most this many in total).
constexpr int Z_ROW_FLOATS = 256;

// z row stride (floats): r_max rounded up to a multiple of 4 (16-byte rows).
inline int z_stride(int r_max) { return (r_max + 3) & ~3; }
cudaError_t launch_expand(__nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int T, const ExpandPlan &plan, bool pdl, cudaStream_t st);
size_t expand_smem_bytes(int tb, int w, int capacity);
int expand_cpt(int tb, int w);
cudaError_t launch_transpose_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int rows, int cols,
                                  cudaStream_t st);
cudaError_t launch_set_int(int32_t *p, int v, cudaStream_t st);

int sm_count();

// Upper bound of the number of shrink tiles of P pairs over `capacity` ids
// (host-computable; the mapping fills unused tile slots with empty records).
int shrink_tile_bound(int P, int capacity);

// Upper bound of the number of tensor-core shrink tiles (MMA_TM pairs of one segment).
int mma_tile_bound(int P, int capacity);

bool fused_supported(int T, int d_out);

// Decode path: per-pair shrink, then a warp per (token, 256 columns) expand.
bool decode_supported(int d_in, int d_out);
cudaError_t launch_decode(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int T, int P, cudaStream_t st);
// Several projections (pools of any shapes, one shared mapping) in one
// decode launch pair: their z columns sit side by side in the mapping's z
// rows of Z_ROW_FLOATS floats.
constexpr int MULTI_MAX_PROJ = 8;
struct MultiDecProj {
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    int zoff;  // first z column of this projection (set by the launcher)
    int nc;    // 256-column chunks of d_out (set by the launcher)
};
struct MultiDecArgs {
    MultiDecProj p[MULTI_MAX_PROJ];
    int n;
    MapDev m;
    int T;
    int gpre[MULTI_MAX_PROJ + 1];  // prefix of the shrink's row groups per projection
    int wpre[MULTI_MAX_PROJ + 1];  // prefix of the expand's (token, chunk) warps per projection
};
cudaError_t launch_decode_multi(const MultiDecArgs &a, int P, cudaStream_t st);
// The pages' kernel ablation (naive loop, Copy + SGMV, pre-merge).
size_t ablation_workspace_bytes(int variant, int T, int P, int d_in, int d_out, int r_max);
cudaError_t run_ablation(int variant, const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool,
                         const int32_t *ranks, const MapDev &m, int T, int P, void *ws, cudaStream_t st);
// Batched recompression (FlashTSQR factor construction) and rank policies.
size_t recompress_workspace_bytes(int M, int d_in, int r);
cudaError_t launch_recompress(const __nv_bfloat16 *A, const __nv_bfloat16 *B, int M, int d_in, int d_out, int r,
                              float *F, float *Tout, float *sigma, void *ws, cudaStream_t st);
int rank_allocate(const float *sigma, int M, int r_stride, const int32_t *rank, const int32_t *cost, int policy,
                  int d, int floor_k, int32_t *k_out);
// The same decode work as one cooperative launch (a CTA per SM): shrink
// items first, then expand warps that wait on per-pair counters.
cudaError_t launch_decode_fused(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                                const MapDev &m, int T, int P, cudaStream_t st);
cudaError_t launch_fused(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                         const MapDev &m, int T, int P, const ExpandPlan &plan, int grid, cudaStream_t st);

// Tensor-core prefill path (tcgen05): segment shrink with the K dimension
// split over a cluster, then a token-tile expand; chained with programmatic
// dependent launch.  Tensor maps of the pool are encoded once per pool.
struct MmaMaps {
    alignas(64) unsigned char At[128];  // CUtensorMap over At: [capacity * r_max][d_in]
    alignas(64) unsigned char B[128];   // CUtensorMap over B:  {64, capacity * r_max, d_out / 64}
    bool ready;
};
cudaError_t mma_encode_maps(const PoolDev &pool, MmaMaps &maps);
bool mma_supported(int d_in, int d_out, int r_max);
cudaError_t launch_mma(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const MmaMaps &maps,
                       const int32_t *ranks, const MapDev &m, int T, int P, cudaStream_t st);

}  // namespace tcl
