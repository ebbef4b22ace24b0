// Mapping stage: per-token pair lists (CSR) -> tuples ordered by adapter id.
//
// DyMerge-LoRA summary page, "Core idea" and "Reading map" (paper Sec. 4.3,
// Algorithm 2, Figure 8): the fused kernel first builds tuples for every
// token-LoRA pair of the batch and reorders them by LoRA id, so that one CTA
// processes the tokens of one adapter back to back and each adapter's A and
// B are read once.
//
// One CTA of 1024 threads performs a stable counting sort on the adapter id
// (the key range is the pool capacity, a few thousand at most):
//   1. check the CSR offsets; expand them into the token of each pair;
//   2. per-warp histograms of the adapter ids over contiguous chunks of the
//      pairs (warp-level match + popcount, no atomics);
//   3. one block scan over (bin, warp) gives every warp's first output slot
//      per bin, the segment starts, and the shrink tiles (<= SHRINK_TT pairs
//      of one segment);
//   4. each warp rescans its chunk and scatters: rank among equal keys =
//      earlier lanes with the same key + the warp's running cursor.
// Stability: chunks are in CSR order, warps are ranked by chunk, lanes by
// pair index, so ties keep CSR order -- the tuples come out ordered by
// (adapter, p).  The result does not depend on timing.
#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

struct Scan3 {
    int a, b, c;
};

// Block-wide exclusive scan of three ints (1024 threads); returns the
// exclusive prefix and writes the block totals.
__device__ Scan3 block_exclusive_scan3(Scan3 v, Scan3 &total, int *sh /* [3][32] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    Scan3 inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int a = __shfl_up_sync(0xffffffffu, inc.a, off);
        int b = __shfl_up_sync(0xffffffffu, inc.b, off);
        int c = __shfl_up_sync(0xffffffffu, inc.c, off);
        if (lane >= off) {
            inc.a += a;
            inc.b += b;
            inc.c += c;
        }
    }
    if (lane == 31) {
        sh[warp] = inc.a;
        sh[32 + warp] = inc.b;
        sh[64 + warp] = inc.c;
    }
    __syncthreads();
    if (warp == 0) {
        int a = sh[lane], b = sh[32 + lane], c = sh[64 + lane];
        int ia = a, ib = b, ic = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int xa = __shfl_up_sync(0xffffffffu, ia, off);
            int xb = __shfl_up_sync(0xffffffffu, ib, off);
            int xc = __shfl_up_sync(0xffffffffu, ic, off);
            if (lane >= off) {
                ia += xa;
                ib += xb;
                ic += xc;
            }
        }
        sh[lane] = ia - a;  // exclusive warp offsets
        sh[32 + lane] = ib - b;
        sh[64 + lane] = ic - c;
        if (lane == 31) {
            sh[96] = ia;
            sh[97] = ib;
            sh[98] = ic;
        }
    }
    __syncthreads();
    Scan3 r;
    r.a = sh[warp] + inc.a - v.a;
    r.b = sh[32 + warp] + inc.b - v.b;
    r.c = sh[64 + warp] + inc.c - v.c;
    total.a = sh[96];
    total.b = sh[97];
    total.c = sh[98];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(MAP_THREADS, 1)
    k_build_mapping(MapDev m, const int32_t *__restrict__ off, const int32_t *__restrict__ ids,
                    const float *__restrict__ alpha, int T, int P, int cap, int nw)
{
    extern __shared__ int32_t hist[];  // [cap][nw]: counts, then cursors
    __shared__ int s_bad;
    __shared__ int s_scan[3 * 32 + 3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        s_bad = (off[0] != 0 || off[T] != P) ? 1 : 0;
        m.hdr[HDR_STATUS] = 0;
    }
    __syncthreads();
    for (int t = tid; t < T; t += MAP_THREADS)
        if (off[t + 1] < off[t])
            s_bad = 1;
    __syncthreads();
    if (s_bad) {
        for (int p = tid; p < P; p += MAP_THREADS)
            m.pos[p] = -1;
        if (tid == 0) {
            m.hdr[HDR_U] = 0;
            m.hdr[HDR_PVALID] = 0;
            m.hdr[HDR_NTILES] = 0;
            m.hdr[HDR_T] = T;
            m.hdr[HDR_STATUS] = LORA_DEV_BAD_OFFSETS;
            m.seg_start[0] = 0;
        }
        return;
    }

    // 1. token of each pair
    for (int t = tid; t < T; t += MAP_THREADS) {
        const int a = off[t], b = off[t + 1];
        for (int p = a; p < b; ++p)
            m.tmp_tok[p] = t;
    }
    for (int i = tid; i < cap * nw; i += MAP_THREADS)
        hist[i] = 0;
    __syncthreads();

    // 2. per-warp histograms over contiguous chunks
    const int chunk = (P + nw - 1) / nw;
    bool bad_id = false;
    if (warp < nw) {
        const int lo = warp * chunk, hi = min(P, lo + chunk);
        for (int base = lo; base < hi; base += 32) {
            const int p = base + lane;
            const bool valid = p < hi;
            const int id = valid ? ids[p] : 0;
            const bool ok = valid && id >= 0 && id < cap;
            bad_id |= valid && !ok;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1 - lane);
            if (ok && lane == __ffs(peers) - 1)
                hist[id * nw + warp] += __popc(peers);
        }
    }
    if (bad_id)
        atomicOr(&m.hdr[HDR_STATUS], LORA_DEV_BAD_ID);
    __syncthreads();

    // 3. scan over bins (each thread owns a contiguous range of bins)
    const int bpt = (cap + MAP_THREADS - 1) / MAP_THREADS;
    const int b0 = min(cap, tid * bpt), b1 = min(cap, b0 + bpt);
    Scan3 mine = {0, 0, 0};
    for (int b = b0; b < b1; ++b) {
        int c = 0;
        for (int w = 0; w < nw; ++w)
            c += hist[b * nw + w];
        mine.a += c;
        if (c > 0) {
            mine.b += 1;
            mine.c += (c + SHRINK_TT - 1) / SHRINK_TT;
        }
    }
    Scan3 total;
    Scan3 base = block_exclusive_scan3(mine, total, s_scan);
    {
        int run = base.a, sidx = base.b, tix = base.c;
        for (int b = b0; b < b1; ++b) {
            int c = 0;
            for (int w = 0; w < nw; ++w)
                c += hist[b * nw + w];
            if (c > 0) {
                m.seg_adapter[sidx] = b;
                m.seg_start[sidx] = run;
                const int ntl = (c + SHRINK_TT - 1) / SHRINK_TT;
                for (int i = 0; i < ntl; ++i)
                    m.tile[tix + i] = make_int4(b, run + i * SHRINK_TT, min(SHRINK_TT, c - i * SHRINK_TT), sidx);
                tix += ntl;
                ++sidx;
            }
            for (int w = 0; w < nw; ++w) {
                const int v = hist[b * nw + w];
                hist[b * nw + w] = run;
                run += v;
            }
        }
    }
    if (tid == 0) {
        m.hdr[HDR_U] = total.b;
        m.hdr[HDR_PVALID] = total.a;
        m.hdr[HDR_NTILES] = total.c;
        m.hdr[HDR_T] = T;
        m.seg_start[total.b] = total.a;
    }
    __syncthreads();

    // 4. stable scatter
    if (warp < nw) {
        const int lo = warp * chunk, hi = min(P, lo + chunk);
        const unsigned lt = (1u << lane) - 1u;
        for (int bse = lo; bse < hi; bse += 32) {
            const int p = bse + lane;
            const bool valid = p < hi;
            const int id = valid ? ids[p] : 0;
            const bool ok = valid && id >= 0 && id < cap;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1 - lane);
            const int cur = ok ? hist[id * nw + warp] : 0;
            if (ok) {
                const int dst = cur + __popc(peers & lt);
                m.tok[dst] = m.tmp_tok[p];
                m.adapter[dst] = id;
                m.alpha[dst] = alpha[p];
                m.src[dst] = p;
                m.pos[p] = dst;
            } else if (valid) {
                m.pos[p] = -1;
            }
            __syncwarp();
            if (ok && lane == __ffs(peers) - 1)
                hist[id * nw + warp] = cur + __popc(peers);
            __syncwarp();
        }
    }
}

}  // namespace

cudaError_t launch_build_mapping(const MapDev &m, const int32_t *offsets, const int32_t *ids,
                                 const float *alpha, int T, int P, int capacity, int max_pairs,
                                 cudaStream_t st)
{
    (void)max_pairs;
    int nw = MAP_HIST_BYTES / (4 * capacity);
    if (nw > 32)
        nw = 32;
    if (nw < 1)
        return cudaErrorInvalidValue;
    const size_t smem = (size_t)capacity * nw * sizeof(int32_t);
    static int attr_done = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_build_mapping, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             MAP_HIST_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    k_build_mapping<<<1, MAP_THREADS, smem, st>>>(m, offsets, ids, alpha, T, P, capacity, nw);
    return cudaGetLastError();
}

}  // namespace tcl
