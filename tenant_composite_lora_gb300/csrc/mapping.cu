// Mapping stage: per-token pair lists (CSR) -> tuples ordered by adapter id.
//
// DyMerge-LoRA summary page, "Core idea" and "Reading map" (paper Sec. 4.3,
// Algorithm 2, Figure 8): the fused kernel first builds tuples for every
// token-LoRA pair of the batch and reorders them by LoRA id, so that one CTA
// processes the tokens of one adapter back to back and each adapter's A and
// B are read once.
//
// Two stages:
//
// k_map_csr (every build; a CTA per 256 tokens) copies the batch into the
// mapping in CSR order:
//   the offsets (toff), and per pair {token, adapter} (pc; adapter -1 when
//   the pair is left out) and alpha (calpha).  It checks the offsets (all
//   pairs are left out when they are malformed), flags ids outside
//   [0, capacity), clears the status word and the fused kernels' counters,
//   and advances the build epoch.  The decode kernels read nothing else:
//   they index pairs in CSR order.
//
// k_map_sort (one CTA; k_sort_count + k_sort_scatter for long batches over
// small pools, below; launched by the paths that read the sorted tuples, before
// their own kernels; it returns at once when the current build is already
// sorted) performs a stable counting sort on the adapter id over the CSR
// copy (the key range is the pool capacity):
//   0. stage pc and calpha in shared memory when they fit (two bulk copies;
//      every later step works on shared memory);
//   1. per-warp histograms of the ids over contiguous chunks of the pairs
//      (shared memory atomics into the warp's own row; layout [warp][bin]);
//   2. block scans over the bins give every warp's first output slot per
//      bin, the segments, the shrink tiles (<= SHRINK_TT pairs of one
//      segment) and the tensor-core shrink tiles (<= MMA_TM pairs of one
//      segment); slots up to the host-known bounds get empty sentinels;
//   3. each warp rescans its chunk and scatters: rank among equal keys =
//      earlier lanes with the same key + the warp's running cursor; the
//      token also goes to its shrink tile's token list;
//   4. when the sorted token and source of every position fit in shared
//      memory, step 3 scatters only there and the sorted arrays are written
//      afterwards position by position, so that every store is coalesced.
// Stability: chunks are in CSR order, warps are ranked by chunk, lanes by
// pair index, so ties keep CSR order -- the tuples come out ordered by
// (adapter, p).  The result does not depend on timing.
#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

struct Scan4 {
    int a, b, c, d;
};

// Block-wide exclusive scan of four ints (blockDim.x threads, a multiple of 32); returns the
// exclusive prefix and writes the block totals.
__device__ Scan4 block_exclusive_scan4(Scan4 v, Scan4 &total, int *sh /* [4 * 32 + 4] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int in[4] = {v.a, v.b, v.c, v.d};
    int inc[4] = {v.a, v.b, v.c, v.d};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int o = __shfl_up_sync(0xffffffffu, inc[j], off);
            if (lane >= off)
                inc[j] += o;
        }
    }
    if (lane == 31)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            sh[32 * j + warp] = inc[j];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int x = lane < (int)(blockDim.x >> 5) ? sh[32 * j + lane] : 0;
            int ix = x;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, ix, off);
                if (lane >= off)
                    ix += o;
            }
            sh[32 * j + lane] = ix - x;
            if (lane == 31)
                sh[128 + j] = ix;
        }
    }
    __syncthreads();
    int r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        r[j] = sh[32 * j + warp] + inc[j] - in[j];
    total = {sh[128], sh[129], sh[130], sh[131]};
    __syncthreads();
    return {r[0], r[1], r[2], r[3]};
}

struct CsrArgs {
    MapDev m;
    const int32_t *off, *ids;
    const float *alpha;
    int T, P, cap;
};

// The CSR stage over a CTA per CSR_TOKENS tokens, a thread per token.
// Before the dependency wait each thread reads its token's offsets and the
// ids and alpha of its first CSR_PR pairs (inputs no kernel of the
// library writes); after it, it writes its token's records.  A CTA that
// finds its tokens' offsets malformed writes no records and flags it; so do
// ids outside the pool.  The CTA that finishes last (a counter in the
// header) writes the status word from the flags of all CTAs, clears both
// words, and -- when some offsets were malformed -- leaves every pair out,
// over the records the other CTAs wrote; a grid of one CTA does all of that
// itself, without the counter.
constexpr int CSR_TOKENS = 256;  // tokens per CTA, one per thread
constexpr int CSR_PR = 8;        // pairs per token read before the wait

__global__ void __launch_bounds__(CSR_TOKENS) k_map_csr(const CsrArgs a)
{
    __shared__ int s_last, s_flags;
    const int tid = threadIdx.x;
    const int T = a.T, P = a.P, cap = a.cap, G = gridDim.x, b = blockIdx.x;
    const int32_t *alb = reinterpret_cast<const int32_t *>(a.alpha);
    const MapDev &m = a.m;
    pdl_launch_dependents();  // the dependents wait for this grid
    const int t = b * CSR_TOKENS + tid;
    int e0 = 0, e1 = 0;
    if (t < T) {
        e0 = __ldg(a.off + t);
        e1 = __ldg(a.off + t + 1);
    }
    // this CTA's share of the check: its tokens' ranges non-decreasing and
    // inside [0, P]; off[0] = 0 and off[T] = P at the ends
    int bad = e1 < e0 || e0 < 0 || e1 > P;
    if (t == 0)
        bad |= e0 != 0;
    if (t == T - 1)
        bad |= e1 != P;
    if (T == 0 && t == 0)  // no token: the offsets are {0} and there is no pair
        bad |= __ldg(a.off) != 0 || P != 0;
    bad = __syncthreads_or(bad);
    int idv[CSR_PR], alv[CSR_PR];
    int pre_bad_id = 0;
#pragma unroll
    for (int i = 0; i < CSR_PR; ++i) {
        const bool in = !bad && e0 + i < e1;
        idv[i] = in ? __ldg(a.ids + e0 + i) : 0;
        alv[i] = in ? __ldg(alb + e0 + i) : 0;
        pre_bad_id |= in && (idv[i] < 0 || idv[i] >= cap);
    }
    // a one-CTA grid whose tokens hold at most CSR_PR pairs each knows its
    // status before the wait (no barrier after it)
    const bool one_pass = G == 1 && !__syncthreads_or(!bad && e1 - e0 > CSR_PR);
    const int pre_status =
        one_pass ? (bad ? LORA_DEV_BAD_OFFSETS : (__syncthreads_or(pre_bad_id) ? LORA_DEV_BAD_ID : 0)) : 0;
    pdl_wait();  // the previous kernel (which may still read this mapping) is done
    if (one_pass && tid == 0)
        m.hdr[HDR_STATUS] = pre_status;
    if (b == 0 && tid == 0) {
        m.hdr[HDR_BAR] = 0;  // fused-kernel counters start over with every mapping
        m.hdr[HDR_BAR_BASE] = 0;
        m.hdr[HDR_EXIT] = 0;
        m.hdr[HDR_EPOCH] = 0;
        m.hdr[HDR_DEXIT] = 0;
        m.hdr[HDR_T] = T;
        atomicAdd(&m.hdr[HDR_BUILD], 1);  // the sorted tuples are stale from here on
    }
    const int q0 = (int)((long long)b * P / G), q1 = (int)((long long)(b + 1) * P / G);
    for (int p = q0 + tid; p < q1; p += CSR_TOKENS)
        m.zcnt[p] = 0;
    int bad_id = 0;
    if (!bad && T == 0 && t == 0)
        m.toff[0] = 0;
    if (!bad && t < T) {
        m.toff[t] = e0;
        if (t == T - 1)
            m.toff[T] = P;
#pragma unroll
        for (int i = 0; i < CSR_PR; ++i)
            if (e0 + i < e1) {
                const bool ok = idv[i] >= 0 && idv[i] < cap;
                bad_id |= !ok;
                m.pc[e0 + i] = make_int2(t, ok ? idv[i] : -1);
                m.calpha[e0 + i] = __int_as_float(alv[i]);
            }
        for (int e = e0 + CSR_PR; e < e1; ++e) {
            const int id = __ldg(a.ids + e);
            const bool ok = id >= 0 && id < cap;
            bad_id |= !ok;
            m.pc[e] = make_int2(t, ok ? id : -1);
            m.calpha[e] = __int_as_float(__ldg(alb + e));
        }
    }
    if (G == 1) {
        // one CTA: it is the last; the status in one store (written above when
        // it was known before the wait), and on malformed offsets every pair
        // left out (it wrote no records)
        if (!one_pass) {
            bad_id = __syncthreads_or(bad_id);
            if (tid == 0)
                m.hdr[HDR_STATUS] = bad ? LORA_DEV_BAD_OFFSETS : (bad_id ? LORA_DEV_BAD_ID : 0);
        }
        if (bad) {
            for (int u = tid; u <= T; u += CSR_TOKENS)
                m.toff[u] = 0;
            for (int p = tid; p < P; p += CSR_TOKENS) {
                m.pc[p] = make_int2(-1, -1);
                m.calpha[p] = 0.f;
            }
        }
        return;
    }
    __threadfence();  // every thread's records before this CTA's count
    bad_id = __syncthreads_or(bad_id);
    if (tid == 0) {
        const int mine = (bad ? LORA_DEV_BAD_OFFSETS : 0) | (bad_id ? LORA_DEV_BAD_ID : 0);
        if (mine)
            atomicOr(&m.hdr[HDR_CSR_FLAGS], mine);
        __threadfence();  // the flags before the count
        const int last = atomicAdd(&m.hdr[HDR_CSR_DONE], 1) == G - 1;
        int flags = 0;
        if (last) {
            __threadfence();
            flags = atomicExch(&m.hdr[HDR_CSR_FLAGS], 0);
            m.hdr[HDR_CSR_DONE] = 0;
            // malformed offsets anywhere: the batch's status is that alone
            m.hdr[HDR_STATUS] = (flags & LORA_DEV_BAD_OFFSETS) ? LORA_DEV_BAD_OFFSETS : flags;
        }
        s_last = last;
        s_flags = flags;
    }
    __syncthreads();
    if (s_last && (s_flags & LORA_DEV_BAD_OFFSETS)) {
        // every pair left out: empty pair ranges, no adapter
        for (int u = tid; u <= T; u += CSR_TOKENS)
            m.toff[u] = 0;
        for (int p = tid; p < P; p += CSR_TOKENS) {
            m.pc[p] = make_int2(-1, -1);
            m.calpha[p] = 0.f;
        }
    }
}

struct SortArgs {
    MapDev m;
    int32_t *hist_g;  // histograms and per-bin arrays in global memory (null: shared memory)
    int T, P, cap, nw, staged, tile_bound, mtile_bound;
    int sorted_smem;  // the scatter lands in shared memory, the sorted arrays are written coalesced after
};

__global__ void __launch_bounds__(MAP_THREADS, 1) k_map_sort(const SortArgs a)
{
    extern __shared__ __align__(16) int32_t sh[];
    __shared__ int s_scan[4 * 32 + 4];
    __shared__ int s_build, s_skip;
    __shared__ __align__(8) uint64_t s_bar;  // the staging copies
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = a.P, cap = a.cap, nw = a.nw;
    const int nthr = blockDim.x;  // 1024, or 256 for short batches
    const MapDev &m = a.m;
    pdl_launch_dependents();  // the dependents wait for this grid
    // pc as words: [2p] token, [2p + 1] adapter (-1: left out); alpha bits
    const int32_t *pcw = reinterpret_cast<const int32_t *>(m.pc), *alb = reinterpret_cast<const int32_t *>(m.calpha);
    // staged: pc words [0, 2 P2), alpha bits [2 P2, 2 P2 + P) (P2 = P rounded up
    // to even: the alpha run starts 16-byte aligned for the bulk copy)
    const int P2 = (P + 1) & ~1, staged_words = 2 * P2 + P;
    int32_t *hist = a.hist_g ? a.hist_g : sh + (a.staged ? staged_words : 0);
    // per bin: first sorted position and first shrink tile of its segment
    int32_t *bin_first = hist + nw * cap, *bin_tile = bin_first + cap;
    // sorted token and source pair per position (with sorted_smem)
    int32_t *s_stok = (a.hist_g ? sh + (a.staged ? staged_words : 0) : bin_tile + cap), *s_ssrc = s_stok + P;
    if (!a.hist_g)
        for (int i = tid; i < nw * cap; i += nthr)
            hist[i] = 0;
    pdl_wait();  // the CSR copy is complete, and no earlier kernel reads the sorted tuples any more
    if (tid == 0) {
        s_build = m.hdr[HDR_BUILD];
        s_skip = m.hdr[HDR_SORTED] == s_build;
    }
    __syncthreads();
    if (s_skip)
        return;  // this build is sorted already
    if (a.staged) {
        // two bulk copies (the 16-byte multiples of pc and alpha) by one
        // thread, the few words beyond them by others, in one round trip
        const uint32_t pc_bytes = 8u * (uint32_t)(P & ~1), al_bytes = 4u * (uint32_t)(P & ~3);
        if (tid == 0) {
            mbar_init(&s_bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&s_bar, pc_bytes + al_bytes);
            if (pc_bytes)
                bulk_g2s(sh, pcw, pc_bytes, &s_bar);
            if (al_bytes)
                bulk_g2s(sh + 2 * P2, alb, al_bytes, &s_bar);
        }
        if (tid < 2 && (P & 1))
            sh[2 * (P - 1) + tid] = pcw[2 * (P - 1) + tid];
        if (tid >= 2 && tid < 2 + (P & 3))
            sh[2 * P2 + (P & ~3) + tid - 2] = alb[(P & ~3) + tid - 2];
        __syncthreads();  // the barrier is initialised before anyone waits on it
        if (!mbar_wait_bounded(&s_bar, 0, m.hdr + HDR_STATUS))
            return;  // status flagged (a copy that never lands)
        pcw = sh;
        alb = sh + 2 * P2;
    }
    if (a.hist_g)
        for (int i = tid; i < nw * cap; i += nthr)
            hist[i] = 0;
    __syncthreads();

    // 1. per-warp histograms
    const int chunk = (P + nw - 1) / nw;
    if (warp < nw) {
        const int lo = warp * chunk, hi = min(P, lo + chunk);
        int32_t *h = hist + warp * cap;
        for (int base = lo; base < hi; base += 32) {
            const int p = base + lane;
            const int id = p < hi ? pcw[2 * p + 1] : -1;
            if (id >= 0)
                atomicAdd(&h[id], 1);  // the warp's own histogram: counts only, order is irrelevant here
        }
    }
    __syncthreads();

    // 2. scan over bins, a CTA's worth of bins per round, bin-ascending
    Scan4 carry = {0, 0, 0, 0};
    for (int base = 0; base < cap; base += nthr) {
        const int b = base + tid;
        int c = 0;
        if (b < cap)
            for (int w = 0; w < nw; ++w)
                c += hist[w * cap + b];
        const Scan4 mine = {c, c > 0 ? 1 : 0, (c + SHRINK_TT - 1) / SHRINK_TT, (c + MMA_TM - 1) / MMA_TM};
        Scan4 tot;
        const Scan4 ex = block_exclusive_scan4(mine, tot, s_scan);
        if (c > 0) {
            int run = carry.a + ex.a;
            const int sidx = carry.b + ex.b, tix = carry.c + ex.c;
            m.seg_adapter[sidx] = b;
            m.seg_start[sidx] = run;
            bin_first[b] = run;
            bin_tile[b] = tix;
            for (int i = 0; i < mine.c; ++i)
                m.tile[tix + i] = make_int4(b, run + i * SHRINK_TT, min(SHRINK_TT, c - i * SHRINK_TT), sidx);
            for (int i = 0, mix = carry.d + ex.d; i < mine.d; ++i)
                m.mtile[mix + i] = make_int4(b, run + i * MMA_TM, min(MMA_TM, c - i * MMA_TM), sidx);
            for (int w = 0; w < nw; ++w) {
                const int v = hist[w * cap + b];
                hist[w * cap + b] = run;
                run += v;
            }
        }
        carry.a += tot.a;
        carry.b += tot.b;
        carry.c += tot.c;
        carry.d += tot.d;
    }
    for (int i = carry.c + tid; i < a.tile_bound; i += nthr)
        m.tile[i] = make_int4(0, 0, 0, -1);  // empty slots up to the host-known bound
    for (int i = carry.d + tid; i < a.mtile_bound; i += nthr)
        m.mtile[i] = make_int4(0, 0, 0, -1);
    if (tid == 0) {
        m.hdr[HDR_U] = carry.b;
        m.hdr[HDR_PVALID] = carry.a;
        m.hdr[HDR_NTILES] = carry.c;
        m.hdr[HDR_NMTILES] = carry.d;
        m.seg_start[carry.b] = carry.a;
    }
    __syncthreads();

    // 3. stable scatter
    if (warp < nw) {
        const int lo = warp * chunk, hi = min(P, lo + chunk);
        int32_t *h = hist + warp * cap;
        const unsigned lt = (1u << lane) - 1u;
        for (int bse = lo; bse < hi; bse += 32) {
            const int p = bse + lane;
            const bool valid = p < hi;
            const int id = valid ? pcw[2 * p + 1] : -1;
            const bool ok = id >= 0;
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1 - lane);
            const int cur = ok ? h[id] : 0;
            if (ok) {
                const int dst = cur + __popc(peers & lt);
                const int t = pcw[2 * p];
                if (a.sorted_smem) {
                    s_stok[dst] = t;
                    s_ssrc[dst] = p;
                } else {
                    m.tok[dst] = t;
                    const int r = dst - bin_first[id];
                    m.tile_tok[(bin_tile[id] + r / SHRINK_TT) * SHRINK_TT + r % SHRINK_TT] = t;
                    m.adapter[dst] = id;
                    reinterpret_cast<int32_t *>(m.alpha)[dst] = alb[p];
                    m.src[dst] = p;
                }
                m.pos[p] = dst;
            } else if (valid) {
                m.pos[p] = -1;
            }
            __syncwarp();
            if (ok && lane == __ffs(peers) - 1)
                h[id] = cur + __popc(peers);
            __syncwarp();
        }
    }
    if (a.sorted_smem) {
        // 4. the sorted arrays, position by position (coalesced stores)
        __syncthreads();
        const int pvalid = carry.a;
        for (int d = tid; d < pvalid; d += nthr) {
            const int p = s_ssrc[d], t = s_stok[d], id = pcw[2 * p + 1];
            m.tok[d] = t;
            m.src[d] = p;
            m.adapter[d] = id;
            reinterpret_cast<int32_t *>(m.alpha)[d] = alb[p];
            const int r = d - bin_first[id];
            m.tile_tok[(bin_tile[id] + r / SHRINK_TT) * SHRINK_TT + r % SHRINK_TT] = t;
        }
    }
    if (tid == 0)
        m.hdr[HDR_SORTED] = s_build;
}

// The sort of a long batch over several CTAs, in two kernels (the second a
// programmatic dependent of the first); the same tuples, bit for bit, as the
// one-CTA sort.  k_sort_count: a CTA per SW_CHUNK pairs (a thread each)
// counts its pairs per adapter and writes the counts; the CTA that finishes
// last (a counter in the header) scans the bins -- segments, shrink tiles,
// tensor-core tiles, the header's counts -- and turns the per-CTA counts into
// every CTA's first sorted position per adapter.  k_sort_scatter: each CTA
// places its pairs -- rank among equal adapters = earlier warps' counts +
// earlier lanes of its own warp (match) + the CTA's first position -- so
// ties keep CSR order.  Both return at once when the build is sorted.
constexpr int SW_CHUNK = 512;     // pairs (threads) per CTA
constexpr int SW_MAX_CTAS = 64;   // up to SW_CHUNK * SW_MAX_CTAS pairs
constexpr int SW_MAX_CAP = 1024;  // pools up to this size

struct SortWideArgs {
    MapDev m;
    int32_t *cnt;             // [G][cap]: per-CTA counts, then per-CTA first positions
    int32_t *bfirst, *btile;  // [cap] each: a bin's first position and first shrink tile
    int P, cap, tile_bound, mtile_bound;
};

__global__ void __launch_bounds__(SW_CHUNK) k_sort_count(const SortWideArgs a)
{
    extern __shared__ __align__(16) int32_t sc[];  // [G][cap]: the last CTA's copy of every CTA's counts
    __shared__ int hist[SW_MAX_CAP];
    __shared__ int s_scan[4 * 32 + 4];
    __shared__ int s_skip, s_last;
    const int tid = threadIdx.x, b = blockIdx.x, G = gridDim.x, cap = a.cap, P = a.P;
    const MapDev &m = a.m;
    pdl_launch_dependents();  // the scatter waits for this grid
    for (int i = tid; i < cap; i += SW_CHUNK)
        hist[i] = 0;
    pdl_wait();  // the CSR copy is complete, and no earlier kernel reads the sorted tuples any more
    if (tid == 0)
        s_skip = m.hdr[HDR_SORTED] == m.hdr[HDR_BUILD];  // no kernel writes either while this grid runs
    __syncthreads();
    if (s_skip) {
        if (b == 0 && tid == 0)
            m.hdr[HDR_SORT_GO] = 0;  // the scatter returns at once
        return;  // this build is sorted already (uniform over the grid)
    }
    const int p = b * SW_CHUNK + tid;
    const int id = p < P ? m.pc[p].y : -1;
    if (id >= 0)
        atomicAdd(&hist[id], 1);
    __syncthreads();
    for (int i = tid; i < cap; i += SW_CHUNK)
        a.cnt[b * cap + i] = hist[i];
    __threadfence();  // the counts before the CTA's arrival
    __syncthreads();
    if (tid == 0)
        s_last = atomicAdd(&m.hdr[HDR_SORT_DONE], 1) == G - 1;
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    // the last CTA: every CTA's counts into shared memory in one round trip,
    // then a scan over bins, a CTA's worth of bins per round, bin-ascending
    for (int i = tid; i < G * cap; i += SW_CHUNK)
        sc[i] = __ldcg(a.cnt + i);
    __syncthreads();
    Scan4 carry = {0, 0, 0, 0};
    for (int base = 0; base < cap; base += SW_CHUNK) {
        const int bin = base + tid;
        int c = 0;
        if (bin < cap)
            for (int g = 0; g < G; ++g)
                c += sc[g * cap + bin];
        const Scan4 mine = {c, c > 0 ? 1 : 0, (c + SHRINK_TT - 1) / SHRINK_TT, (c + MMA_TM - 1) / MMA_TM};
        Scan4 tot;
        const Scan4 ex = block_exclusive_scan4(mine, tot, s_scan);
        if (c > 0) {
            int run = carry.a + ex.a;
            const int sidx = carry.b + ex.b, tix = carry.c + ex.c;
            m.seg_adapter[sidx] = bin;
            m.seg_start[sidx] = run;
            a.bfirst[bin] = run;
            a.btile[bin] = tix;
            for (int i = 0; i < mine.c; ++i)
                m.tile[tix + i] = make_int4(bin, run + i * SHRINK_TT, min(SHRINK_TT, c - i * SHRINK_TT), sidx);
            for (int i = 0, mix = carry.d + ex.d; i < mine.d; ++i)
                m.mtile[mix + i] = make_int4(bin, run + i * MMA_TM, min(MMA_TM, c - i * MMA_TM), sidx);
            for (int g = 0; g < G; ++g) {
                const int v = sc[g * cap + bin];
                sc[g * cap + bin] = run;
                run += v;
            }
        }
        carry.a += tot.a;
        carry.b += tot.b;
        carry.c += tot.c;
        carry.d += tot.d;
    }
    __syncthreads();
    for (int i = tid; i < G * cap; i += SW_CHUNK)
        a.cnt[i] = sc[i];  // every CTA's first position per adapter
    for (int i = carry.c + tid; i < a.tile_bound; i += SW_CHUNK)
        m.tile[i] = make_int4(0, 0, 0, -1);  // empty slots up to the host-known bound
    for (int i = carry.d + tid; i < a.mtile_bound; i += SW_CHUNK)
        m.mtile[i] = make_int4(0, 0, 0, -1);
    if (tid == 0) {
        m.hdr[HDR_U] = carry.b;
        m.hdr[HDR_PVALID] = carry.a;
        m.hdr[HDR_NTILES] = carry.c;
        m.hdr[HDR_NMTILES] = carry.d;
        m.seg_start[carry.b] = carry.a;
        m.hdr[HDR_SORT_DONE] = 0;
        m.hdr[HDR_SORT_GO] = 1;
    }
}

__global__ void __launch_bounds__(SW_CHUNK) k_sort_scatter(const SortWideArgs a)
{
    extern __shared__ __align__(16) int32_t wh[];  // [SW_CHUNK / 32][cap]: each warp's count per adapter
    __shared__ int s_build, s_skip;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x, cap = a.cap, P = a.P;
    const MapDev &m = a.m;
    pdl_launch_dependents();  // the dependents wait for this grid
    for (int i = tid; i < (SW_CHUNK / 32) * cap; i += SW_CHUNK)
        wh[i] = 0;
    pdl_wait();  // the counting grid, its last CTA included, is complete
    if (tid == 0) {
        s_build = m.hdr[HDR_BUILD];
        s_skip = m.hdr[HDR_SORT_GO] == 0;  // set by the counting grid, which is complete
    }
    __syncthreads();
    if (s_skip)
        return;
    const int p = b * SW_CHUNK + tid;
    const bool valid = p < P;
    const int2 pc = valid ? m.pc[p] : make_int2(0, -1);
    const int id = pc.y;
    const bool ok = id >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? id : -1 - lane);
    if (ok && lane == __ffs(peers) - 1)
        wh[warp * cap + id] = __popc(peers);
    __syncthreads();
    if (ok) {
        int dst = __ldcg(a.cnt + b * cap + id) + __popc(peers & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w)
            dst += wh[w * cap + id];
        m.tok[dst] = pc.x;
        m.adapter[dst] = id;
        reinterpret_cast<int32_t *>(m.alpha)[dst] = reinterpret_cast<const int32_t *>(m.calpha)[p];
        m.src[dst] = p;
        m.pos[p] = dst;
        const int r = dst - __ldcg(a.bfirst + id);
        m.tile_tok[(__ldcg(a.btile + id) + r / SHRINK_TT) * SHRINK_TT + r % SHRINK_TT] = pc.x;
    } else if (valid) {
        m.pos[p] = -1;
    }
    if (b == 0 && tid == 0)
        m.hdr[HDR_SORTED] = s_build;  // read by later launches only: this grid decided by HDR_SORT_GO
}

template <class K>
cudaError_t map_attrs(K kernel, int &done)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (done == dev)
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MAP_SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        done = dev;
    return e;
}

template <class Args>
cudaError_t map_launch(void (*kernel)(Args), const Args &a, int threads, size_t smem, cudaStream_t st,
                       unsigned grid = 1)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

int shrink_tile_bound(int P, int capacity)
{
    if (P <= 0)
        return 0;
    const long long b = (long long)(P + SHRINK_TT - 1) / SHRINK_TT + (P < capacity ? P : capacity);
    return (int)(b < P ? b : P);
}

int mma_tile_bound(int P, int capacity)
{
    if (P <= 0)
        return 0;
    const long long b = (long long)(P + MMA_TM - 1) / MMA_TM + (P < capacity ? P : capacity);
    return (int)(b < P ? b : P);
}

int map_wide_sort_words(int capacity)
{
    return capacity <= SW_MAX_CAP ? (SW_MAX_CTAS + 2) * capacity : 0;
}

int map_global_hist_words(int capacity)
{
    // shared memory holds one warp's histogram and the two per-bin arrays
    // (unstaged inputs) up to this capacity
    if (3LL * capacity <= MAP_SMEM_BYTES / 4)
        return 0;
    return (MAP_GHIST_WARPS + 2) * capacity;
}

cudaError_t launch_map_csr(const MapDev &m, const int32_t *offsets, const int32_t *ids, const float *alpha, int T,
                           int P, int capacity, cudaStream_t st)
{
    static thread_local int attr_done = -1;  // per host thread
    const cudaError_t e = map_attrs(k_map_csr, attr_done);
    if (e != cudaSuccess)
        return e;
    const CsrArgs a{m, offsets, ids, alpha, T, P, capacity};
    return map_launch(k_map_csr, a, CSR_TOKENS, 0, st, T > 0 ? (unsigned)((T + CSR_TOKENS - 1) / CSR_TOKENS) : 1u);
}

cudaError_t launch_map_sort(const MapDev &m, int T, int P, int capacity, cudaStream_t st)
{
    const long long sw_ctas = (P + SW_CHUNK - 1) / SW_CHUNK;
    if (m.gsort && P >= 4 * SW_CHUNK && sw_ctas <= SW_MAX_CTAS && capacity <= SW_MAX_CAP &&
        sw_ctas * capacity * 4 <= MAP_SMEM_BYTES) {
        // long batches over small pools: the several-CTA sort
        static thread_local int count_done = -1, scatter_done = -1;  // per host thread
        cudaError_t e = map_attrs(k_sort_count, count_done);
        if (e == cudaSuccess)
            e = map_attrs(k_sort_scatter, scatter_done);
        if (e != cudaSuccess)
            return e;
        const unsigned G = (unsigned)((P + SW_CHUNK - 1) / SW_CHUNK);
        const SortWideArgs a{m, m.gsort, m.gsort + SW_MAX_CTAS * capacity, m.gsort + (SW_MAX_CTAS + 1) * capacity,
                             P, capacity, shrink_tile_bound(P, capacity), mma_tile_bound(P, capacity)};
        e = map_launch(k_sort_count, a, SW_CHUNK, (size_t)G * capacity * 4, st, G);
        if (e == cudaSuccess)
            e = map_launch(k_sort_scatter, a, SW_CHUNK, (size_t)(SW_CHUNK / 32) * capacity * 4, st, G);
        return e;
    }
    const long long budget = MAP_SMEM_BYTES / 4;  // int32 words
    const long long staged_words = 2LL * ((P + 1) & ~1) + P;  // pc (two words per pair, even count) and alpha
    // short batches over small pools: one CTA of 256 threads (cheaper
    // block-wide phases, the bins still one scan round); otherwise 1024
    const int threads = (P <= 512 && capacity <= 256) ? 256 : MAP_THREADS;
    int nw = (P + 63) / 64;
    nw = nw < 1 ? 1 : (nw > threads / 32 ? threads / 32 : nw);
    int staged = 0;
    int32_t *hist_g = nullptr;
    // words: [staged arrays] + nw histograms + two per-bin arrays
    if (map_global_hist_words(capacity) > 0) {
        // a pool too large for shared memory: histograms in global memory
        if (!m.ghist)
            return cudaErrorInvalidValue;
        hist_g = m.ghist;
        if (nw > MAP_GHIST_WARPS)
            nw = MAP_GHIST_WARPS;
        staged = staged_words <= budget ? 1 : 0;
    } else if (staged_words + 3LL * capacity <= budget) {
        staged = 1;
        const long long fit = (budget - staged_words) / capacity - 2;
        if (nw > fit)
            nw = (int)fit;
    } else {
        const long long fit = budget / capacity - 2;
        if (nw > fit)
            nw = (int)fit;
    }
    if (nw < 1)
        return cudaErrorInvalidValue;
    // long batches: the sorted positions' token and source pair also in shared
    // memory when they fit (short ones gain less than the extra phase costs)
    const long long hist_words = hist_g ? 0 : (long long)(nw + 2) * capacity;
    const int sorted_smem = staged && P >= 2048 && staged_words + hist_words + 2LL * P <= budget;
    const size_t smem = 4 * ((staged ? (size_t)staged_words : 0) + (size_t)hist_words + (sorted_smem ? 2 * (size_t)P : 0));
    static thread_local int attr_done = -1;  // per host thread
    const cudaError_t e = map_attrs(k_map_sort, attr_done);
    if (e != cudaSuccess)
        return e;
    const SortArgs a{m, hist_g, T, P, capacity, nw, staged, shrink_tile_bound(P, capacity),
                     mma_tile_bound(P, capacity), sorted_smem};
    return map_launch(k_map_sort, a, threads, smem, st);
}

cudaError_t launch_build_mapping(const MapDev &m, const int32_t *offsets, const int32_t *ids,
                                 const float *alpha, int T, int P, int capacity, int max_pairs,
                                 cudaStream_t st)
{
    (void)max_pairs;
    cudaError_t e = launch_map_csr(m, offsets, ids, alpha, T, P, capacity, st);
    if (e == cudaSuccess)
        e = launch_map_sort(m, T, P, capacity, st);
    return e;
}

}  // namespace tcl
