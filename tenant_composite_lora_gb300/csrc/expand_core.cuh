// Expand phase (RowExpand), shared by the split path (k_expand) and the fused
// decode kernel (k_fused):
//
//   y[t, c] = bf16( y[t, c] + sum_{q: tok_q = t} sum_{j < k_q} z_q[j] * B_{a_q}[j, c] )
//
// LoRAForge summary page, "Approach" (4) and "Developer view": the expand
// keeps each thread's slice of the B rows in registers, reuses it across the
// tokens that share the adapter, and takes z from a shared tile.  DyMerge-
// LoRA summary page, "Core idea" (paper Sec. 4.3): pairs are walked in adapter
// order, so each adapter's B tile is staged once for all of its tokens.
//
// CTA = (token block [t0, t0 + tb), blockIdx.y) x (W output columns) x
// (segment group g of ng).  The ng CTAs of one column tile form a thread-block
// cluster: each sums the pairs of its share of the segments into an fp32
// accumulator tile in shared memory, then the cluster reduces the ng tiles
// through distributed shared memory in a fixed order, adds y and rounds once
// to bf16.  The result does not depend on timing and needs no global atomics.
// For a decode batch the token block is the whole batch (no search); for
// longer batches the block's pairs of a segment are found by binary search
// (tokens are ascending inside a segment) and ng = 1.
//
// Segment ranges are cut into jobs of <= EXP_JP pairs; a window of jobs is
// staged with 16-byte cp.async copies (the k retained B rows x W columns of
// each job, the jobs' z rows, their tokens).  On its first visit of a segment
// that is unlikely to fit the first window, the CTA also prefetches that
// segment's B rows into L2 (per-line prefetches from many threads), so later
// windows hit L2.  Warp w owns the block tokens with
// (t - t0) % 8 == w; each lane owns W / 32 columns and keeps its slice of up
// to 16 B rows in registers while it walks the job's pairs.
//
// Everything that does not depend on z (metadata, the first window's B
// tiles, the y tile, the per-token pair lists) happens before the `before_z`
// hook: griddepcontrol.wait on the split path, the shrink phase and a grid
// barrier in the fused kernel.
#pragma once

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace tcl {

constexpr int NWARP = EXP_THREADS / 32;
constexpr int B_ELEMS = EXP_B_BYTES / 2;
constexpr int Z_FLOATS = EXP_Z_BYTES / 4;
constexpr int WIN_PAIRS = EXP_WIN_PAIRS;
static_assert(NWARP == 8, "eight warps per CTA");
static_assert(EXP_JP <= 32, "one lane per pair of a job");

struct ExpandArgs {
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int T, tb, zs;
    int w;        // tile width (columns)
    int ng;       // segment groups = cluster size along x
    int use_tab;  // ranks staged in shared memory
};

// Dynamic shared memory layout (byte offsets), identical on host and device.
struct ExpLayout {
    int yin, B, Z, tok, pjob, plist, jobA, jobB, rank, total;
    __host__ __device__ ExpLayout(int tb, int w, int cap_tab)
    {
        yin = 0;
        B = (yin + tb * w * 2 + 127) & ~127;  // also the fp32 tile (tb * w * 4 <= EXP_B_BYTES) at the end
        Z = B + EXP_B_BYTES;
        tok = Z + EXP_Z_BYTES;
        pjob = tok + WIN_PAIRS * 4;
        plist = pjob + WIN_PAIRS * 4;
        jobA = plist + WIN_PAIRS * 4;
        jobB = jobA + EXP_MAX_JOBS * 16;
        rank = jobB + EXP_MAX_JOBS * 16;
        total = rank + ((cap_tab + 3) & ~3) * 4;
    }
};

__device__ __forceinline__ int lower_bound_tok(const int32_t *tok, int lo, int hi, int v)
{
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (tok[mid] < v)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Block-wide exclusive scan of an int4 over EXP_THREADS threads.
__device__ __forceinline__ int4 block_scan4(int4 v, int4 &total, int4 *sh /* [NWARP] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4 inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int4 o;
        o.x = __shfl_up_sync(0xffffffffu, inc.x, off);
        o.y = __shfl_up_sync(0xffffffffu, inc.y, off);
        o.z = __shfl_up_sync(0xffffffffu, inc.z, off);
        o.w = __shfl_up_sync(0xffffffffu, inc.w, off);
        if (lane >= off) {
            inc.x += o.x;
            inc.y += o.y;
            inc.z += o.z;
            inc.w += o.w;
        }
    }
    if (lane == 31)
        sh[warp] = inc;
    __syncthreads();
    int4 before = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
        const int4 s = sh[w];
        if (w < warp) {
            before.x += s.x;
            before.y += s.y;
            before.z += s.z;
            before.w += s.w;
        }
        tot.x += s.x;
        tot.y += s.y;
        tot.z += s.z;
        tot.w += s.w;
    }
    __syncthreads();
    total = tot;
    return make_int4(before.x + inc.x - v.x, before.y + inc.y - v.y, before.z + inc.z - v.z,
                     before.w + inc.w - v.w);
}

// CPT: columns of the tile owned by one thread (2, 4, 8, 16 or 32); the
// tile width W and the threads per token TPT = W / CPT are runtime values.

// Static shared state of the expand phase.
struct ExpandShared {
    int4 scan[NWARP];
    int cutjob, cur_s, cur_p;
    int cnt[EXP_THREADS], start[EXP_THREADS], cursor[EXP_THREADS];
};

// Stages the y rows [r0, r1) of the tile and the rank table; returns U.
__device__ __forceinline__ int expand_prologue(const ExpandArgs &a, unsigned char *smem_raw, int c0, int t0, int r0,
                                               int r1)
{
    const int W = a.w, VPR = W / 8, tid = threadIdx.x;
    const ExpLayout L(a.tb, W, a.use_tab ? a.pool.capacity : 0);
    __nv_bfloat16 *yin = reinterpret_cast<__nv_bfloat16 *>(smem_raw + L.yin);
    int *rank_tab = reinterpret_cast<int *>(smem_raw + L.rank);
    for (int i = tid; i < (r1 - r0) * VPR; i += EXP_THREADS) {
        const int t = r0 + i / VPR, v = i % VPR;
        cp_async16(&yin[t * W + v * 8], a.y + (size_t)(t0 + t) * a.pool.d_out + c0 + v * 8);
    }
    cp_async_commit();
    if (a.use_tab)
        for (int i = tid; i < a.pool.capacity; i += EXP_THREADS)
            rank_tab[i] = effective_rank(a.pool, a.ranks, i);
    return a.m.hdr[HDR_U];
}

// Accumulates, for this thread's token my_t and columns [my_c, my_c + CPT) of
// the tile (c0, t0, nt), the pairs of segments [s_begin, s_end) into racc.
// Calls before_z() exactly once, uniformly, before the first z read (also
// when there is no work).  Ends with every copy landed and the CTA synced.
template <int CPT, class BeforeZ>
__device__ __forceinline__ void expand_accumulate(const ExpandArgs &a, unsigned char *smem_raw, ExpandShared &es,
                                                  int c0, int t0, int nt, bool full_range, int s_begin,
                                                  int s_end, float (&racc)[CPT], BeforeZ before_z)
{
    const int W = a.w;
    const int VPR = W / 8;
    const int TPT = W / CPT;
    const ExpLayout L(a.tb, W, a.use_tab ? a.pool.capacity : 0);
    __nv_bfloat16 *sB = reinterpret_cast<__nv_bfloat16 *>(smem_raw + L.B);
    float *sZ = reinterpret_cast<float *>(smem_raw + L.Z);
    int *sTok = reinterpret_cast<int *>(smem_raw + L.tok);
    int4 *jobA = reinterpret_cast<int4 *>(smem_raw + L.jobA);  // {adapter, q, len, k}
    int4 *jobB = reinterpret_cast<int4 *>(smem_raw + L.jobB);  // {B offset, Z offset, tok offset, kp}
    int *rank_tab = reinterpret_cast<int *>(smem_raw + L.rank);
    int *pjob = reinterpret_cast<int *>(smem_raw + L.pjob);    // window pair -> job
    int *plist = reinterpret_cast<int *>(smem_raw + L.plist);  // window pairs grouped by token
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d_out = a.pool.d_out, r_max = a.pool.r_max;
    const int my_t = tid / TPT, my_c = (tid % TPT) * CPT;
    const int t1 = t0 + nt;

    bool waited = false;
    int s_next = s_begin, piece_next = 0;
    while (s_next < s_end) {
        // ---- build a window of jobs from segments s_next .. s_next + 255 of the group
        const int s = s_next + tid;
        int k = 0, lo = 0, hi = 0, adapter = 0, pfirst = 0, np = 0;
        if (s < s_end) {
            adapter = a.m.seg_adapter[s];
            const int sa = a.m.seg_start[s], sb = a.m.seg_start[s + 1];
            k = a.use_tab ? rank_tab[adapter] : effective_rank(a.pool, a.ranks, adapter);
            if (k < 0)
                k = 0;
            if (k > 0) {
                if (full_range) {
                    lo = sa;
                    hi = sb;
                } else {
                    lo = lower_bound_tok(a.m.tok, sa, sb, t0);
                    hi = lower_bound_tok(a.m.tok, lo, sb, t1);
                }
            }
            if (hi > lo) {
                pfirst = (tid == 0) ? piece_next : 0;
                np = (hi - lo + EXP_JP - 1) / EXP_JP - pfirst;
            }
        }
        const int kp = (k + 3) & ~3;
        const int my_pairs = np > 0 ? (hi - lo - pfirst * EXP_JP) : 0;
        const int4 mine = make_int4(np, np * k * W, my_pairs * kp, my_pairs);
        if (tid == 0) {
            es.cutjob = INT_MAX;
            es.cur_s = s_next + EXP_THREADS;
            es.cur_p = 0;
        }
        int4 total;
        const int4 ex = block_scan4(mine, total, es.scan);  // its barriers order the s_* writes above
        {
            int pairs_before = 0;
            for (int pi = 0; pi < np; ++pi) {
                const int qs = lo + (pfirst + pi) * EXP_JP;
                const int len = min(EXP_JP, hi - qs);
                const int job = ex.x + pi;
                const int bo = ex.y + pi * k * W;
                const int zo = ex.z + pairs_before * kp;
                const int to = ex.w + pairs_before;
                const bool fits = job < EXP_MAX_JOBS && bo + k * W <= B_ELEMS && zo + len * kp <= Z_FLOATS &&
                                  to + len <= WIN_PAIRS;
                if (!fits) {
                    atomicMin(&es.cutjob, job);
                    break;
                }
                jobA[job] = make_int4(adapter, qs, len, k);
                jobB[job] = make_int4(bo, zo, to, kp);
                pairs_before += len;
            }
        }
        __syncthreads();
        const int njobs = min(total.x, es.cutjob);
        if (es.cutjob != INT_MAX) {
            // the thread whose first excluded piece is the cut resumes there
            for (int pi = 0; pi < np; ++pi)
                if (ex.x + pi == es.cutjob) {
                    es.cur_s = s;
                    es.cur_p = pfirst + pi;
                }
        }

        // ---- tokens of the window's pairs (mapping data), one lane per pair
        for (int j = warp; j < njobs; j += NWARP) {
            const int4 ja = jobA[j];
            const int to = jobB[j].z;
            if (lane < ja.z) {
                sTok[to + lane] = a.m.tok[ja.y + lane];
                pjob[to + lane] = j;
            }
        }
        // ---- stage B tiles (pool data: legal before the dependency wait)
        for (int j = warp; j < njobs; j += NWARP) {
            const int4 ja = jobA[j];
            const int bo = jobB[j].x;
            const __nv_bfloat16 *src = a.pool.B + (size_t)ja.x * r_max * d_out + c0;
            for (int i = lane; i < ja.w * VPR; i += 32) {
                const int r = i / VPR, v = i % VPR;
                cp_async16(&sB[bo + r * W + v * 8], src + (size_t)r * d_out + v * 8);
            }
        }
        // ---- list the window's pairs per token (stable, window order kept)
        const int npw = njobs > 0 ? jobB[njobs - 1].z + jobA[njobs - 1].z : 0;
        es.cnt[tid] = 0;
        __syncthreads();  // also publishes the tokens staged above
        for (int e = tid; e < npw; e += EXP_THREADS)
            atomicAdd(&es.cnt[sTok[e] - t0], 1);
        __syncthreads();
        {
            int4 tot4;
            const int4 ex4 = block_scan4(make_int4(es.cnt[tid], 0, 0, 0), tot4, es.scan);
            es.start[tid] = ex4.x;
            es.cursor[tid] = ex4.x;
        }
        __syncthreads();
        if (warp == 0) {
            const unsigned lt = (1u << lane) - 1u;
            for (int base = 0; base < npw; base += 32) {
                const int e = base + lane;
                const bool valid = e < npw;
                const int t = valid ? sTok[e] - t0 : -1 - lane;
                const unsigned peers = __match_any_sync(0xffffffffu, t);
                const int cur = valid ? es.cursor[t] : 0;
                if (valid)
                    plist[cur + __popc(peers & lt)] = e;
                __syncwarp();
                if (valid && lane == __ffs(peers) - 1)
                    es.cursor[t] = cur + __popc(peers);
                __syncwarp();
            }
        }
        __syncthreads();
        if (!waited) {
            before_z();
            waited = true;
        }
        for (int j = warp; j < njobs; j += NWARP) {
            const int4 ja = jobA[j], jb = jobB[j];
            const int nv = jb.w >> 2;
            for (int i = lane; i < ja.z * nv; i += 32) {
                const int r = i / nv, v = i - r * nv;
                cp_async16(&sZ[jb.y + r * jb.w + v * 4], a.m.z + (size_t)(ja.y + r) * a.zs + v * 4);
            }
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();

        // ---- accumulate this thread's token over its pairs of the window
        if (my_t < nt) {
            const int i0 = es.start[my_t], i1 = i0 + es.cnt[my_t];
            for (int idx = i0; idx < i1; ++idx) {
                const int e = plist[idx];
                const int j = pjob[e];
                const int4 ja = jobA[j], jb = jobB[j];
                const float *zr = &sZ[jb.y + (e - jb.z) * jb.w];
                const __nv_bfloat16 *bb = &sB[jb.x + my_c];
                for (int r = 0; r < ja.w; ++r) {
                    const float zz = zr[r];
                    const __nv_bfloat16 *br = bb + r * W;
                    if constexpr (CPT == 2) {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(br);
                        racc[0] = fmaf(zz, bf16lo(w), racc[0]);
                        racc[1] = fmaf(zz, bf16hi(w), racc[1]);
                    } else if constexpr (CPT == 4) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(br);
                        racc[0] = fmaf(zz, bf16lo(w.x), racc[0]);
                        racc[1] = fmaf(zz, bf16hi(w.x), racc[1]);
                        racc[2] = fmaf(zz, bf16lo(w.y), racc[2]);
                        racc[3] = fmaf(zz, bf16hi(w.y), racc[3]);
                    } else {
#pragma unroll
                        for (int v = 0; v < CPT / 8; ++v) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(br + v * 8);
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                racc[v * 8 + 2 * h] = fmaf(zz, bf16lo(ww[h]), racc[v * 8 + 2 * h]);
                                racc[v * 8 + 2 * h + 1] = fmaf(zz, bf16hi(ww[h]), racc[v * 8 + 2 * h + 1]);
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
        s_next = es.cur_s;
        piece_next = es.cur_p;
        __syncthreads();
    }
    if (!waited)
        before_z();
    cp_async_wait_all();
    __syncthreads();
}

}  // namespace tcl
