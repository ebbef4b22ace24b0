// Expand (RowExpand): y[t, c] = bf16( y[t, c] + sum_{q: tok_q = t} sum_{j < k_q} z_q[j] * B_{a_q}[j, c] )
//
// LoRAForge summary page, "Approach" (4) and "Developer view": the expand
// keeps each thread's slice of the B rows in registers, reuses it across the
// tokens that share the adapter, and takes z from a shared tile.  DyMerge-
// LoRA summary page, "Core idea" (paper Sec. 4.3): pairs are walked in adapter
// order, so each adapter's B tile is staged once for all of its tokens.
//
// CTA = (token block [t0, t0 + tb), blockIdx.x) x (32 or 64 output
// columns, blockIdx.y).  The CTA owns
// its y tile outright: every pair of every token of the block is summed into
// an fp32 accumulator tile in shared memory, in a fixed order (segment
// ascending, then pair order), and the tile is rounded once to bf16 and
// written.  No global atomics; the result does not depend on timing.
//
// Inside a segment the pairs are ordered by token, so the block's pairs of a
// segment are one contiguous range (found by binary search).  Ranges are cut
// into jobs of <= EXP_JP pairs; a window of jobs is staged with 16-byte
// cp.async copies: the k retained B rows x EXP_W columns of each job, the
// jobs' z rows, the tokens.  Warp w owns the block tokens with
// (t - t0) % 8 == w; each lane owns one or two columns.  The segment list,
// the header and a shared-memory table of retained ranks are read at entry in
// one round trip; a decode batch (T <= token block) needs no search.
//
// Launched with programmatic dependent launch after the shrink kernel: the
// first window's B tiles and the y tile (neither written by the shrink) are
// staged before griddepcontrol.wait, overlapping the shrink; z is read after.
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int NWARP = EXP_THREADS / 32;
constexpr int WMAX = EXP_W;
constexpr int B_ELEMS = EXP_B_BYTES / 2;
constexpr int Z_FLOATS = EXP_Z_BYTES / 4;
constexpr int WIN_PAIRS = 1024;
static_assert(NWARP == 8, "warp owns tokens mod 8");

struct ExpandArgs {
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int T, tb, zs;
    int seg_bound;  // host-known bound on the number of segments
    int use_tab;    // ranks staged in shared memory
};

struct Smem {
    float acc[EXP_TB_MAX * WMAX];
    __nv_bfloat16 yin[EXP_TB_MAX * WMAX];
    __nv_bfloat16 B[B_ELEMS];
    float Z[Z_FLOATS];
    int tok[WIN_PAIRS];
    int4 jobA[EXP_MAX_JOBS];  // {adapter, q, len, k}
    int4 jobB[EXP_MAX_JOBS];  // {B offset (elements), Z offset (floats), tok offset, kp}
    int rank_tab[RANK_TAB_MAX];
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
__device__ int4 block_scan4(int4 v, int4 &total, int4 *sh /* [NWARP] */)
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

// W output columns per CTA: 64 (lane owns 2 columns) or 32 (lane owns 1).
template <int W>
__global__ void __launch_bounds__(EXP_THREADS, 1) k_expand(ExpandArgs a)
{
    static_assert(W == 32 || W == 64, "tile width");
    constexpr int VPR = W / 8;  // 16-byte vectors per tile row
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    __shared__ int4 s_scan[NWARP];
    __shared__ int s_cutjob, s_cur_s, s_cur_p;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d_out = a.pool.d_out, r_max = a.pool.r_max;
    const int c0 = blockIdx.y * W;
    const int t0 = blockIdx.x * a.tb, t1 = min(a.T, t0 + a.tb), nt = t1 - t0;
    const bool full_range = (t0 == 0 && t1 >= a.T);

    // y tile (not written by the shrink: legal before the dependency wait)
    for (int i = tid; i < nt * VPR; i += EXP_THREADS) {
        const int t = i / VPR, v = i % VPR;
        cp_async16(&sm.yin[t * W + v * 8], a.y + (size_t)(t0 + t) * d_out + c0 + v * 8);
    }
    cp_async_commit();
    if (a.use_tab)
        for (int i = tid; i < a.pool.capacity; i += EXP_THREADS)
            sm.rank_tab[i] = effective_rank(a.pool, a.ranks, i);
    for (int i = tid; i < nt * W; i += EXP_THREADS)
        sm.acc[i] = 0.f;
    const int U = min(a.m.hdr[HDR_U], a.seg_bound);
    __syncthreads();

    bool waited = false;
    int s_next = 0, piece_next = 0;
    while (s_next < U) {
        // ---- build a window of jobs from segments s_next .. s_next + 255
        const int s = s_next + tid;
        int k = 0, lo = 0, hi = 0, adapter = 0, pfirst = 0, np = 0;
        if (s < U) {
            adapter = a.m.seg_adapter[s];
            const int sa = a.m.seg_start[s], sb = a.m.seg_start[s + 1];
            k = a.use_tab ? sm.rank_tab[adapter] : effective_rank(a.pool, a.ranks, adapter);
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
        int4 mine = make_int4(np, np * k * W, my_pairs * kp, my_pairs);
        if (tid == 0) {
            s_cutjob = INT_MAX;
            s_cur_s = s_next + EXP_THREADS;
            s_cur_p = 0;
        }
        int4 total;
        const int4 ex = block_scan4(mine, total, s_scan);  // its barriers order the s_* writes above
        {
            int pairs_before = 0;
            for (int pi = 0; pi < np; ++pi) {
                const int qs = lo + (pfirst + pi) * EXP_JP;
                const int len = min(EXP_JP, hi - qs);
                const int job = ex.x + pi;
                const int bo = ex.y + pi * k * W;
                const int zo = ex.z + pairs_before * kp;
                const int to = ex.w + pairs_before;
                const bool fits = job < EXP_MAX_JOBS && bo + k * W <= B_ELEMS &&
                                  zo + len * kp <= Z_FLOATS && to + len <= WIN_PAIRS;
                if (!fits) {
                    atomicMin(&s_cutjob, job);
                    break;
                }
                sm.jobA[job] = make_int4(adapter, qs, len, k);
                sm.jobB[job] = make_int4(bo, zo, to, kp);
                for (int i = 0; i < len; ++i)
                    sm.tok[to + i] = a.m.tok[qs + i];
                pairs_before += len;
            }
        }
        __syncthreads();
        const int njobs = min(total.x, s_cutjob);
        if (s_cutjob != INT_MAX) {
            // the thread whose first excluded piece is the cut resumes there
            for (int pi = 0; pi < np; ++pi)
                if (ex.x + pi == s_cutjob) {
                    s_cur_s = s;
                    s_cur_p = pfirst + pi;
                }
        }

        // ---- stage B tiles (pool data: legal before the dependency wait)
        for (int j = warp; j < njobs; j += NWARP) {
            const int4 ja = sm.jobA[j];
            const int bo = sm.jobB[j].x;
            const __nv_bfloat16 *src = a.pool.B + (size_t)ja.x * r_max * d_out + c0;
            for (int i = lane; i < ja.w * VPR; i += 32) {
                const int r = i / VPR, v = i % VPR;
                cp_async16(&sm.B[bo + r * W + v * 8], src + (size_t)r * d_out + v * 8);
            }
        }
        if (!waited) {
            pdl_wait();  // z comes from the shrink kernel
            waited = true;
        }
        for (int j = warp; j < njobs; j += NWARP) {
            const int4 ja = sm.jobA[j], jb = sm.jobB[j];
            const int nv = jb.w >> 2;
            for (int i = lane; i < ja.z * nv; i += 32) {
                const int r = i / nv, v = i - r * nv;
                cp_async16(&sm.Z[jb.y + r * jb.w + v * 4], a.m.z + (size_t)(ja.y + r) * a.zs + v * 4);
            }
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();

        // ---- accumulate: warp owns tokens (t - t0) % 8 == warp, lane owns W/32 columns
        for (int j = 0; j < njobs; ++j) {
            const int4 ja = sm.jobA[j], jb = sm.jobB[j];
            for (int i = 0; i < ja.z; ++i) {
                const int t = sm.tok[jb.z + i] - t0;
                if ((t & (NWARP - 1)) != warp)
                    continue;
                const float *zr = &sm.Z[jb.y + i * jb.w];
                if (W == 64) {
                    const uint32_t *brow = reinterpret_cast<const uint32_t *>(&sm.B[jb.x]) + lane;
                    float d0 = 0.f, d1 = 0.f;
                    for (int jj = 0; jj < ja.w; ++jj) {
                        const uint32_t b = brow[jj * (W / 2)];
                        const float zz = zr[jj];
                        d0 = fmaf(zz, bf16lo(b), d0);
                        d1 = fmaf(zz, bf16hi(b), d1);
                    }
                    float2 *ap = reinterpret_cast<float2 *>(&sm.acc[t * W]) + lane;
                    float2 cur = *ap;
                    cur.x += d0;
                    cur.y += d1;
                    *ap = cur;
                } else {
                    const unsigned short *brow = reinterpret_cast<const unsigned short *>(&sm.B[jb.x]) + lane;
                    float d0 = 0.f;
                    for (int jj = 0; jj < ja.w; ++jj)
                        d0 = fmaf(zr[jj], __uint_as_float((uint32_t)brow[jj * W] << 16), d0);
                    sm.acc[t * W + lane] += d0;
                }
            }
        }
        __syncthreads();
        s_next = s_cur_s;
        piece_next = s_cur_p;
        __syncthreads();
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- y = bf16(y_in + acc), one rounding
    for (int i = tid; i < nt * VPR; i += EXP_THREADS) {
        const int t = i / VPR, v = i % VPR;
        const uint4 yi = *reinterpret_cast<const uint4 *>(&sm.yin[t * W + v * 8]);
        const float *ac = &sm.acc[t * W + v * 8];
        const uint32_t w[4] = {yi.x, yi.y, yi.z, yi.w};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(bf16lo(w[h]) + ac[2 * h]);
            const __nv_bfloat16 hi = __float2bfloat16_rn(bf16hi(w[h]) + ac[2 * h + 1]);
            o[h] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
        *reinterpret_cast<uint4 *>(a.y + (size_t)(t0 + t) * d_out + c0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace

cudaError_t launch_expand(__nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks, const MapDev &m, int T,
                          int P, int tb, int w, bool pdl, cudaStream_t st)
{
    const size_t smem = sizeof(Smem);
    static int attr_done = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_expand<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_expand<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    const int seg_bound = P < pool.capacity ? P : pool.capacity;
    ExpandArgs a{y, pool, ranks, m, T, tb, z_stride(pool.r_max), seg_bound, pool.capacity <= RANK_TAB_MAX ? 1 : 0};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((T + tb - 1) / tb, pool.d_out / w, 1);
    cfg.blockDim = dim3(EXP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (w == 32)
        return cudaLaunchKernelEx(&cfg, k_expand<32>, a);
    return cudaLaunchKernelEx(&cfg, k_expand<64>, a);
}

}  // namespace tcl
