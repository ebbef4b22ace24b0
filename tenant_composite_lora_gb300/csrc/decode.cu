// Decode path: every batch below the dispatch table's prefill threshold (all
// decode batches, and long batches at small ranks).  Every pair reads its own
// x row and its adapter's factor rows (an adapter shared by several pairs
// comes from L2 after the first).  Two launches chained with programmatic
// dependent launch, every global access a 16-byte coalesced vector:
//
// Pairs are taken in CSR order (the mapping's CSR stage: per pair its token,
// adapter and alpha), so neither kernel needs the adapter-sorted tuples: each
// pair reads its own A rows here, and the sort only pays off where many
// tokens share an adapter segment (the split and tensor-core paths).
//
// 1. Shrink (LoRAForge page, "Approach" (4): direct reduction for short
//    decode batches; DyMerge-LoRA page, "Core idea": the weight alpha folded
//    in).  A CTA owns one pair q and 4 or 8 consecutive rank rows (long
//    batches at large ranks: several such row groups of its pair in turn);
//    its x row is staged once in shared memory (or, in CTAs of 8 rows, read
//    by each warp into registers) and each warp streams one row
//    of A_a (stored transposed, contiguous along d_in) against it, reducing
//    with warp shuffles:  z[q][j] = alpha_q * sum_d x[tok_q][d] * A_a[d][j].
//
// 2. Expand (RowExpand, LoRAForge page, "Approach" (4)): a warp owns one
//    token and 256 output columns (8 per lane); a CTA's warps are
//    consecutive tokens on one column chunk, sharing B rows through L1.
//    Before waiting for the
//    shrink it reads the token's pair list and issues the loads of y and of
//    the first B rows (they do not depend on z; rows are fetched before the
//    rank is known and used only below it); then it adds
//    sum_pairs sum_j z[q][j] * B_a[j][cols] in fp32, 8 or 16 rows in flight
//    at a time, and rounds once to bf16.  The launch picks the instance that
//    keeps the batch's warps in one wave where it can (fewer registers, more
//    CTAs per SM, for long batches; that instance prefetches one pair's rows
//    and reads the next pairs' adapters and ranks before the wait) and a CTA
//    of 8 warps per (token, 256 columns) for few tokens at large ranks.
//
// Both kernels order their loads so that each waits on as few dependent
// round trips to memory as possible: a decode batch moves little data, and
// its time is the chain of latencies.  The shrink is itself a programmatic
// dependent of the mapping kernel (its CTAs are resident when the mapping
// ends) and releases the expand only once its own wait has returned, since
// the expand's prologue reads the mapping and y; the expand lets the next
// kernel in the stream start early (that kernel waits before it writes), and
// every expand warp waits on the shrink before it exits, so that the expand
// completes only after the shrink.
#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int DS_THREADS = 256;  // at most 8 warps: one rank row each

struct DecShrinkArgs {
    const __nv_bfloat16 *x;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int zs;    // z row stride (floats per pair)
    float *z;  // this projection's first z column: z[q * zs + j], q the CSR pair
    int ngroups, gpc;  // row groups per pair, and groups per CTA (k_dec_shrink)
};

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc)
{
    acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc);
    acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
    acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
    acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
    acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
    acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
    acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
    acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
    return acc;
}

// One shrink item: CSR pair q, rank rows [j0, j0 + warps of the CTA), or with
// GROUPS, ngrp such groups one after the other (warp w takes row w of each,
// the x row staged once).  Every thread of the CTA calls it; it returns once
// the CTA's copies have landed.  report: set the status bit of an unusable
// adapter (one item per pair does).
template <bool GROUPS, bool XREG = false>
__device__ __forceinline__ void dec_shrink_item(const DecShrinkArgs &a, uint4 *xs, int q, int j0, int ngrp,
                                                bool report)
{
    if (!GROUPS)
        ngrp = 1;
    // one round trip: the pair's token and adapter, and its alpha
    const int2 pc = a.m.pc[q];
    const float al = a.m.calpha[q];
    const int tk = pc.x, ad = pc.y;
    if (ad < 0)
        return;  // pairs left out of the mapping (and every pair when its offsets were malformed)
    const int r_max = a.pool.r_max;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = j0 + warp;
    // the first row group fetches its rows before the rank is known (they are
    // almost always below it); later groups read the rank first, so rows at or
    // beyond it are never fetched
    int k_early = r_max;
    if (j0 > 0) {
        k_early = effective_rank(a.pool, a.ranks, ad);
        if (k_early <= j0)
            return;  // no row of this group is used (status reported by group 0)
    }
    const bool row = j < k_early;
    const int d_in = a.pool.d_in, nv = d_in / 8;  // 16-byte vectors per row
    if (XREG && nv <= 32 * 16) {
        // (the 8-row CTAs of ranks above 8) each warp reads the x row itself
        // into registers (from L2 after the first warp) beside its A row, so
        // that no block barrier waits for the slowest of the 8 warps' copies
        const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)tk * d_in);
        const uint4 *ar = reinterpret_cast<const uint4 *>(a.pool.At + ((size_t)ad * r_max + (row ? j : 0)) * d_in);
        uint4 av[16], xv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = u * 32 + lane;
            const bool in = row && i < nv;
            av[u] = in ? __ldcs(&ar[i]) : make_uint4(0u, 0u, 0u, 0u);
            xv[u] = in ? __ldg(&xr[i]) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int k = effective_rank(a.pool, a.ranks, ad);
        if (k <= 0 || j0 >= k) {
            if (k < 0 && report && threadIdx.x == 0)
                atomicOr(a.m.hdr + HDR_STATUS, k == -1 ? LORA_DEV_UNREGISTERED : LORA_DEV_BAD_RANK);
            return;
        }
        if (j >= k)
            return;  // this warp's row is at or past the rank (uniform over the warp)
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
            if (u * 32 + lane < nv)
                acc = dot8(av[u], xv[u], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0)
            a.z[(size_t)q * a.zs + j] = al * acc;
        return;
    }
    // second round trip: x row (to shared memory), the A row, the rank
    const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)tk * d_in);
    for (int i = threadIdx.x; i < nv; i += blockDim.x)
        cp_async16(&xs[i], &xr[i]);
    cp_async_commit();
    const uint4 *ar = reinterpret_cast<const uint4 *>(a.pool.At + ((size_t)ad * r_max + (row ? j : 0)) * d_in);
    uint4 av[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int i = u * 32 + lane;
        av[u] = row && i < nv ? __ldcs(&ar[i]) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int k = effective_rank(a.pool, a.ranks, ad);
    if (k <= 0 || j0 >= k) {
        if (k < 0 && report && threadIdx.x == 0)
            atomicOr(a.m.hdr + HDR_STATUS, k == -1 ? LORA_DEV_UNREGISTERED : LORA_DEV_BAD_RANK);
        cp_async_wait_all();
        return;
    }
    cp_async_wait_all();
    __syncthreads();
    const int W = blockDim.x >> 5;
    for (int g = 0; g < ngrp; ++g) {
        const int jw = j + g * W;  // this warp's row of group g
        if (j0 + g * W >= k)
            break;  // uniform: no row of this group is used
        const bool live = jw < k;
        const uint4 *arw = reinterpret_cast<const uint4 *>(a.pool.At + ((size_t)ad * r_max + (live ? jw : 0)) * d_in);
        if (GROUPS && g > 0) {  // the first group's rows were fetched above
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = u * 32 + lane;
                av[u] = live && i < nv ? __ldcs(&arw[i]) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int i = u * 32 + lane;
            if (i < nv)
                acc = dot8(av[u], xs[i], acc);
        }
        // longer rows: further batches of 16 vectors per lane
        for (int base = 32 * 16; base < nv; base += 32 * 16) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = base + u * 32 + lane;
                av[u] = live && i < nv ? __ldcs(&arw[i]) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = base + u * 32 + lane;
                if (i < nv)
                    acc = dot8(av[u], xs[i], acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (live && lane == 0)
            a.z[(size_t)q * a.zs + jw] = al * acc;
    }
}

// XREG: CTAs of 8 rank rows take the x row into each warp's registers
// (measured faster there; slower for the 4-row CTAs of ranks up to 8).
template <bool XREG>
__global__ void __launch_bounds__(DS_THREADS) k_dec_shrink(const DecShrinkArgs a)
{
    extern __shared__ __align__(16) uint4 xs[];  // the pair's x row
    pdl_wait();  // launched as a programmatic dependent of the mapping (or of a previous apply)
    // Only now may the expand launch: it reads the mapping (pair lists, the
    // header) and y before its own wait on this kernel, so everything that
    // precedes this kernel in the stream -- the mapping, and through the
    // mapping's own wait every earlier kernel, a previous expand that wrote y
    // included -- must have completed.  Its prologue still overlaps the work
    // below.
    pdl_launch_dependents();
    dec_shrink_item<false, XREG>(a, xs, blockIdx.x, blockIdx.y * (blockDim.x >> 5), 1, blockIdx.y == 0);
}

// The same over several row groups of its pair per CTA (long batches at large ranks).
__global__ void __launch_bounds__(DS_THREADS) k_dec_shrink_groups(const DecShrinkArgs a)
{
    extern __shared__ __align__(16) uint4 xs[];  // the pair's x row
    pdl_wait();               // as k_dec_shrink
    pdl_launch_dependents();  // as k_dec_shrink
    const int W = blockDim.x >> 5;
    dec_shrink_item<true>(a, xs, blockIdx.x, blockIdx.y * a.gpc * W, min(a.gpc, a.ngroups - (int)blockIdx.y * a.gpc),
                          blockIdx.y == 0);
}

struct DecExpandArgs {
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int T, zs, nc;  // nc: 256-column chunks per row (the last may be partial)
    const float *z; // the shrink's output for this projection: z[q * zs + j], q the CSR pair
};

__device__ __forceinline__ void fma8(float (&acc)[8], float z, uint4 b)
{
    acc[0] = fmaf(z, bf16lo(b.x), acc[0]);
    acc[1] = fmaf(z, bf16hi(b.x), acc[1]);
    acc[2] = fmaf(z, bf16lo(b.y), acc[2]);
    acc[3] = fmaf(z, bf16hi(b.y), acc[3]);
    acc[4] = fmaf(z, bf16lo(b.z), acc[4]);
    acc[5] = fmaf(z, bf16hi(b.z), acc[5]);
    acc[6] = fmaf(z, bf16lo(b.w), acc[6]);
    acc[7] = fmaf(z, bf16hi(b.w), acc[7]);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

constexpr int DE_PP = 3;  // pairs of a token whose B rows are fetched before the dependency wait
constexpr int DE_PR = 8;  // rows fetched per such pair

// Retained rank of adapter ad for this call, 0 when it contributes nothing.
__device__ __forceinline__ int dec_rank(const PoolDev &pool, const int32_t *ranks, int ad)
{
    const int k = effective_rank(pool, ranks, ad);
    return k > 0 ? k : 0;
}

// acc += sum_{j in [jb, k)} z[j] * B row j, R rows in flight at a time (rows
// ascending whatever R: the same sums in the same order).
template <int R>
__device__ __forceinline__ void dec_rows(float (&acc)[8], const __nv_bfloat16 *br, const float *zr, int jb, int k,
                                         int d_out, bool on)
{
    for (int j = jb; j < k; j += R) {
        uint4 bb[R];
        float zz[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const bool v = j + u < k;
            bb[u] = v && on ? __ldg(reinterpret_cast<const uint4 *>(br + (size_t)(j + u) * d_out))
                            : make_uint4(0u, 0u, 0u, 0u);
            zz[u] = v ? __ldcg(zr + j + u) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < R; ++u)
            fma8(acc, zz[u], bb[u]);
    }
}

// One expand item: token t, 256-column chunk c, on one warp.  wait_pair(q)
// is called before the first read of pair q's z (the shrink's output).  NX:
// pairs after the PP prefetched ones whose adapter and rank are also read
// before the wait (then one round trip each after it, for B, instead of
// three) -- for the one-prefetched-pair instance, whose tokens have more.
template <int PP, int R, int NX, class WaitPair>
__device__ __forceinline__ void dec_expand_item(const DecExpandArgs &a, int t, int c, WaitPair wait_pair)
{
    const int lane = threadIdx.x & 31;
    const int d_out = a.pool.d_out, r_max = a.pool.r_max;
    const int col = c * 256 + lane * 8;
    const bool on = col < d_out;  // the last chunk of a row may be partial
    // round trip 1: y, the token's pair range
    __nv_bfloat16 *yp = a.y + (size_t)t * d_out + (on ? col : 0);
    const uint4 yv = on ? *reinterpret_cast<const uint4 *>(yp) : make_uint4(0u, 0u, 0u, 0u);
    const int p0 = a.m.toff[t], p1 = a.m.toff[t + 1];
    if (p1 <= p0)
        return;  // no pair: y stays as it is (every token when the offsets were malformed)
    // round trip 2: the adapters of the first pairs (and of the NX after them)
    int pa[PP], px[NX > 0 ? NX : 1], kx[NX > 0 ? NX : 1];
#pragma unroll
    for (int i = 0; i < PP; ++i)
        pa[i] = p0 + i < p1 ? a.m.pc[p0 + i].y : -1;
#pragma unroll
    for (int i = 0; i < NX; ++i)
        px[i] = p0 + PP + i < p1 ? a.m.pc[p0 + PP + i].y : -1;
    // round trip 3: their first B rows (whatever the rank turns out to be) and ranks
#pragma unroll
    for (int i = 0; i < NX; ++i)
        kx[i] = px[i] >= 0 ? dec_rank(a.pool, a.ranks, px[i]) : 0;
    uint4 bpre[PP][DE_PR];
    int kk[PP];
#pragma unroll
    for (int i = 0; i < PP; ++i) {
        const int ad = pa[i];
        const __nv_bfloat16 *br = a.pool.B + (size_t)(ad < 0 ? 0 : ad) * r_max * d_out + col;
#pragma unroll
        for (int j = 0; j < DE_PR; ++j)
            bpre[i][j] = ad >= 0 && on && j < r_max ? __ldg(reinterpret_cast<const uint4 *>(br + (size_t)j * d_out))
                                                    : make_uint4(0u, 0u, 0u, 0u);
        kk[i] = ad >= 0 ? dec_rank(a.pool, a.ranks, ad) : 0;
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < PP; ++i) {
        const int k = kk[i];
        if (k > 0) {
            wait_pair(p0 + i);
            const float *zr = a.z + (size_t)(p0 + i) * a.zs;
            float zz[DE_PR];
#pragma unroll
            for (int j = 0; j < DE_PR; ++j)
                zz[j] = j < k ? __ldcg(zr + j) : 0.f;
#pragma unroll
            for (int j = 0; j < DE_PR; ++j)
                fma8(acc, zz[j], bpre[i][j]);
            if (k > DE_PR)
                dec_rows<R>(acc, a.pool.B + (size_t)pa[i] * r_max * d_out + col, zr, DE_PR, k, d_out, on);
        }
    }
#pragma unroll
    for (int i = 0; i < NX; ++i) {
        const int p = p0 + PP + i;
        if (p < p1 && kx[i] > 0) {
            wait_pair(p);
            dec_rows<R>(acc, a.pool.B + (size_t)px[i] * r_max * d_out + col, a.z + (size_t)p * a.zs, 0, kx[i], d_out,
                        on);
        }
    }
    for (int p = p0 + PP + NX; p < p1; ++p) {
        const int ad = a.m.pc[p].y;
        if (ad < 0)
            continue;
        const int k = dec_rank(a.pool, a.ranks, ad);
        if (k > 0) {
            wait_pair(p);
            dec_rows<R>(acc, a.pool.B + (size_t)ad * r_max * d_out + col, a.z + (size_t)p * a.zs, 0, k, d_out, on);
        }
    }
    uint4 o;
    o.x = pack2(bf16lo(yv.x) + acc[0], bf16hi(yv.x) + acc[1]);
    o.y = pack2(bf16lo(yv.y) + acc[2], bf16hi(yv.y) + acc[3]);
    o.z = pack2(bf16lo(yv.z) + acc[4], bf16hi(yv.z) + acc[5]);
    o.w = pack2(bf16lo(yv.w) + acc[6], bf16hi(yv.w) + acc[7]);
    if (on)
        *reinterpret_cast<uint4 *>(yp) = o;
}

// PP pairs' rows are fetched before the dependency wait; MINB CTAs per SM
// (two when the batch needs more than one wave of warps, at the price of one
// fewer prefetched pair).  Past the prefetched rows, a pair's rows come RF at
// a time: 16 for ranks above 16 on one CTA per SM (a shorter chain of round
// trips per pair), else 8.
template <int PP, int MINB, int RF>
__global__ void __launch_bounds__(256, MINB) k_dec_expand(const DecExpandArgs a)
{
    pdl_launch_dependents();  // the next kernel in the stream may start its prologue
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (g >= a.T * a.nc)
        return;
    // consecutive warps: consecutive tokens on one column chunk, so the B rows
    // of an adapter several of them use come from L1 after the first
    bool waited = false;
    dec_expand_item<PP, RF, PP == 1 ? 3 : 0>(a, g % a.T, g / a.T, [&](int) {
        if (!waited) {
            pdl_wait();  // z of the shrink
            waited = true;
        }
    });
    if (!waited)
        pdl_wait();  // complete only after the shrink
}

// Few tokens at large ranks: a CTA of 8 warps per (token, 256 columns), warp
// w taking rank rows w, w + 8, ... of every pair (all of a warp's rows of the
// first pairs fetched before the dependency wait), partial sums reduced
// through shared memory.
constexpr int DW_WARPS = 8;
constexpr int DW_PP = 2;                         // pairs whose rows are fetched before the wait
constexpr int DW_PR = LORA_MAX_RANK / DW_WARPS;  // rows per warp and pair

__global__ void __launch_bounds__(32 * DW_WARPS, 1) k_dec_expand_wide(const DecExpandArgs a)
{
    __shared__ float red[DW_WARPS - 1][256];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x % a.T, c = blockIdx.x / a.T;
    const int d_out = a.pool.d_out, r_max = a.pool.r_max;
    const int col = c * 256 + lane * 8;
    const bool on = col < d_out;
    __nv_bfloat16 *yp = a.y + (size_t)t * d_out + (on ? col : 0);
    const uint4 yv = on && warp == 0 ? *reinterpret_cast<const uint4 *>(yp) : make_uint4(0u, 0u, 0u, 0u);
    const int p0 = a.m.toff[t], p1 = a.m.toff[t + 1];
    if (p1 <= p0) {
        pdl_wait();  // no pair (uniform over the CTA); complete only after the shrink
        return;
    }
    int pa[DW_PP];
#pragma unroll
    for (int i = 0; i < DW_PP; ++i)
        pa[i] = p0 + i < p1 ? a.m.pc[p0 + i].y : -1;
    uint4 bpre[DW_PP][DW_PR];
    int kk[DW_PP];
#pragma unroll
    for (int i = 0; i < DW_PP; ++i) {
        const int ad = pa[i];
        const __nv_bfloat16 *br = a.pool.B + (size_t)(ad < 0 ? 0 : ad) * r_max * d_out + col;
#pragma unroll
        for (int u = 0; u < DW_PR; ++u) {
            const int j = warp + DW_WARPS * u;
            bpre[i][u] = ad >= 0 && on && j < r_max ? __ldg(reinterpret_cast<const uint4 *>(br + (size_t)j * d_out))
                                                    : make_uint4(0u, 0u, 0u, 0u);
        }
        kk[i] = ad >= 0 ? dec_rank(a.pool, a.ranks, ad) : 0;
    }
    pdl_wait();  // z of the shrink
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < DW_PP; ++i) {
        const int k = kk[i];
        if (k > 0) {
            const float *zr = a.z + (size_t)(p0 + i) * a.zs;
            float zz[DW_PR];
#pragma unroll
            for (int u = 0; u < DW_PR; ++u) {
                const int j = warp + DW_WARPS * u;
                zz[u] = j < k ? __ldcg(zr + j) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < DW_PR; ++u)
                fma8(acc, zz[u], bpre[i][u]);
        }
    }
    for (int p = p0 + DW_PP; p < p1; ++p) {
        const int ad = a.m.pc[p].y;
        if (ad < 0)
            continue;
        const int k = dec_rank(a.pool, a.ranks, ad);
        if (k <= 0)
            continue;
        const __nv_bfloat16 *br = a.pool.B + (size_t)ad * r_max * d_out + col;
        const float *zr = a.z + (size_t)p * a.zs;
        uint4 bb[DW_PR];
        float zz[DW_PR];
#pragma unroll
        for (int u = 0; u < DW_PR; ++u) {
            const int j = warp + DW_WARPS * u;
            const bool use = j < k;
            bb[u] = use && on ? __ldg(reinterpret_cast<const uint4 *>(br + (size_t)j * d_out)) : make_uint4(0u, 0u, 0u, 0u);
            zz[u] = use ? __ldcg(zr + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < DW_PR; ++u)
            fma8(acc, zz[u], bb[u]);
    }
    if (warp > 0)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            red[warp - 1][lane * 8 + e] = acc[e];
    __syncthreads();
    if (warp == 0) {
        for (int w = 0; w < DW_WARPS - 1; ++w)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] += red[w][lane * 8 + e];
        uint4 o;
        o.x = pack2(bf16lo(yv.x) + acc[0], bf16hi(yv.x) + acc[1]);
        o.y = pack2(bf16lo(yv.y) + acc[2], bf16hi(yv.y) + acc[3]);
        o.z = pack2(bf16lo(yv.z) + acc[4], bf16hi(yv.z) + acc[5]);
        o.w = pack2(bf16lo(yv.w) + acc[6], bf16hi(yv.w) + acc[7]);
        if (on)
            *reinterpret_cast<uint4 *>(yp) = o;
    }
}

// ------------------------------------------------------------ fused (one launch)

struct DecFusedArgs {
    DecShrinkArgs s;
    DecExpandArgs e;
    int ng;  // shrink items per pair: rank rows in groups of 8
    int P;   // pairs of the batch (CSR)
};

// Waits until *cnt >= target, for at most WAIT_LIMIT_NS (then LORA_DEV_TIMEOUT).
__device__ __forceinline__ bool wait_count(const int32_t *cnt, int target, int32_t *status)
{
    return wait_count_bounded(cnt, (unsigned)target, status);
}

// A cooperative launch, every CTA resident: each CTA first runs shrink items
// (pair, 8 rank rows) and counts them per pair, then its warps run expand
// items, each waiting only on the counters of its token's pairs.  The CTAs
// never wait on one another during the shrink phase, so every counter is
// reached.  The launch's epoch (launches since the mapping was built) sets
// the counters' target; the last CTA to exit advances it.
__global__ void __launch_bounds__(256, 1) k_dec_fused(const DecFusedArgs a)
{
    extern __shared__ __align__(16) uint4 xs[];
    pdl_launch_dependents();
    const MapDev &m = a.s.m;
    int32_t *status = m.hdr + HDR_STATUS;
    const int epoch = m.hdr[HDR_EPOCH];
    const int G = gridDim.x;
    for (int it = blockIdx.x; it < a.P * a.ng; it += G) {
        const int q = it / a.ng, g = it % a.ng;
        dec_shrink_item<false>(a.s, xs, q, g * (blockDim.x >> 5), 1, g == 0);
        __syncthreads();  // z rows written, x row consumed
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(m.zcnt + q, 1);
        }
    }
    const int target = (epoch + 1) * a.ng;
    const int nw = blockDim.x >> 5;
    bool ok = true;
    for (int wi = blockIdx.x * nw + (threadIdx.x >> 5); wi < a.e.T * a.e.nc; wi += G * nw)
        dec_expand_item<DE_PP, 8, 0>(a.e, wi % a.e.T, wi / a.e.T, [&](int q) {
            if (ok)
                ok = wait_count(m.zcnt + q, target, status);
        });
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(m.hdr + HDR_DEXIT, 1) == G - 1) {  // the last CTA of this launch
            m.hdr[HDR_DEXIT] = 0;
            __threadfence();
            atomicAdd(m.hdr + HDR_EPOCH, 1);
        }
    }
}

// ------------------------------------------------------------ several projections, one launch each

// The shrink of every projection in one grid: blockIdx.y runs over the
// projections' row groups (prefix gpre), blockIdx.x over the CSR pairs.
__global__ void __launch_bounds__(DS_THREADS) k_dec_shrink_multi(const MultiDecArgs a)
{
    extern __shared__ __align__(16) uint4 xs[];
    pdl_wait();               // as k_dec_shrink
    pdl_launch_dependents();  // the expand reads the mapping and y before its own wait
    const int yb = blockIdx.y;
    int j = 0;
    while (j + 1 < a.n && yb >= a.gpre[j + 1])
        ++j;
    const MultiDecProj &pj = a.p[j];
    const DecShrinkArgs sa{pj.x, pj.pool, pj.ranks, a.m, Z_ROW_FLOATS, a.m.z + pj.zoff};
    dec_shrink_item<false>(sa, xs, blockIdx.x, (yb - a.gpre[j]) * (blockDim.x >> 5), 1, yb == a.gpre[j]);
}

// The expand of every projection in one grid: warp g runs (projection j,
// token, column chunk) with g - wpre[j] = chunk * T + token.
template <int PP, int MINB>
__global__ void __launch_bounds__(256, MINB) k_dec_expand_multi(const MultiDecArgs a)
{
    pdl_launch_dependents();
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (g >= a.wpre[a.n])
        return;
    int j = 0;
    while (j + 1 < a.n && g >= a.wpre[j + 1])
        ++j;
    const MultiDecProj &pj = a.p[j];
    const DecExpandArgs ea{pj.y, pj.pool, pj.ranks, a.m, a.T, Z_ROW_FLOATS, pj.nc, a.m.z + pj.zoff};
    const int gl = g - a.wpre[j];
    bool waited = false;
    dec_expand_item<PP, 8, 0>(ea, gl % a.T, gl / a.T, [&](int) {
        if (!waited) {
            pdl_wait();  // z of the shrink
            waited = true;
        }
    });
    if (!waited)
        pdl_wait();  // complete only after the shrink
}

}  // namespace

// The x row is staged in shared memory: d_in * 2 bytes of at most 200 KB.
constexpr int DS_SMEM_MAX = 200 * 1024;
bool decode_supported(int d_in, int d_out) { return d_in % 8 == 0 && d_out % 8 == 0 && d_in * 2 <= DS_SMEM_MAX; }

cudaError_t launch_decode(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int T, int P, cudaStream_t st)
{
    if (!decode_supported(pool.d_in, pool.d_out))
        return cudaErrorNotSupported;
    static thread_local int attr_dev = -1;  // per host thread: concurrent first calls each set the attribute
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_dec_shrink<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             DS_SMEM_MAX);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_dec_shrink<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM_MAX);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_dec_shrink_groups, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    DecShrinkArgs sa{x, pool, ranks, m, z_stride(pool.r_max), m.z};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // rows per group: 8, or 4 when r_max is small, so that a short batch's A
    // rows spread over more SMs.  A CTA takes g of its pair's groups one after
    // the other: the time goes as g (the CTA's chain) plus the waves of
    // resident CTAs, items / (g * resident), least at g = sqrt(items /
    // resident) -- one group per CTA for decode batches, several for long
    // batches at large ranks (fewer CTAs that stop at the rank, the x row
    // staged once for all of their groups)
    const int rpc = pool.r_max <= 8 ? 4 : 8;
    sa.ngroups = (pool.r_max + rpc - 1) / rpc;
    const long long resident = (long long)sm_count() * (rpc == 8 ? 3 : 6);
    const long long items = (long long)P * sa.ngroups;
    int g = 1;
    while (g < sa.ngroups && (long long)g * g * resident < items)
        ++g;
    sa.gpc = g;
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = dim3(P, (sa.ngroups + sa.gpc - 1) / sa.gpc, 1);
    scfg.blockDim = dim3(32 * rpc, 1, 1);
    scfg.dynamicSmemBytes = (size_t)pool.d_in * 2;
    scfg.stream = st;
    scfg.attrs = attr;
    scfg.numAttrs = 1;
    cudaError_t e = sa.gpc > 1   ? cudaLaunchKernelEx(&scfg, k_dec_shrink_groups, sa)
                    : rpc == 8 ? cudaLaunchKernelEx(&scfg, k_dec_shrink<true>, sa)
                               : cudaLaunchKernelEx(&scfg, k_dec_shrink<false>, sa);
    if (e != cudaSuccess)
        return e;
    const int nc = (pool.d_out + 255) / 256;
    const long long warps = (long long)T * nc;
    DecExpandArgs ea{y, pool, ranks, m, T, z_stride(pool.r_max), nc, m.z};
    if (pool.r_max > 16 && warps <= 2LL * sm_count()) {
        // few (token, chunk) items at large ranks: 8 warps share each item's rows
        cudaLaunchConfig_t wcfg = {};
        wcfg.gridDim = dim3((unsigned)warps, 1, 1);
        wcfg.blockDim = dim3(32 * DW_WARPS, 1, 1);
        wcfg.stream = st;
        wcfg.attrs = attr;
        wcfg.numAttrs = 1;
        return cudaLaunchKernelEx(&wcfg, k_dec_expand_wide, ea);
    }
    int wpc = 8;  // warps per CTA: the most that still gives a CTA per SM
    while (wpc > 1 && (warps + wpc - 1) / wpc < sm_count())
        wpc >>= 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + wpc - 1) / wpc), 1, 1);
    cfg.blockDim = dim3(32 * wpc, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (warps > 16LL * sm_count())  // more than one wave at two 8-warp CTAs per SM: three, one prefetched pair
        return cudaLaunchKernelEx(&cfg, k_dec_expand<1, 3, 8>, ea);
    if (warps > 8LL * sm_count())  // more than one wave at one 8-warp CTA per SM
        return cudaLaunchKernelEx(&cfg, k_dec_expand<2, 2, 8>, ea);
    if (pool.r_max > 16)
        return cudaLaunchKernelEx(&cfg, k_dec_expand<DE_PP, 1, 16>, ea);
    return cudaLaunchKernelEx(&cfg, k_dec_expand<DE_PP, 1, 8>, ea);
}

cudaError_t launch_decode_fused(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                                const MapDev &m, int T, int P, cudaStream_t st)
{
    if (!decode_supported(pool.d_in, pool.d_out))
        return cudaErrorNotSupported;
    // per host thread: the device and its co-residency figure are set together
    static thread_local int attr_dev = -1, resident = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = (size_t)pool.d_in * 2;
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_dec_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        // co-residency of every CTA: one per SM (the launch bound and the
        // largest staging buffer allow one at the least)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, k_dec_fused, 256, DS_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    if (resident < 1)
        return cudaErrorNotSupported;
    const int ng = (pool.r_max + 7) / 8;
    const int nc = (pool.d_out + 255) / 256;
    DecFusedArgs a{{x, pool, ranks, m, z_stride(pool.r_max), m.z}, {y, pool, ranks, m, T, z_stride(pool.r_max), nc, m.z},
                   ng, P};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count(), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_dec_fused, a);
}

cudaError_t launch_decode_multi(const MultiDecArgs &in, int P, cudaStream_t st)
{
    MultiDecArgs a = in;
    if (a.n < 1 || a.n > MULTI_MAX_PROJ)
        return cudaErrorInvalidValue;
    int max_din = 0, max_r = 0, zcols = 0;
    for (int j = 0; j < a.n; ++j) {
        const PoolDev &pj = a.p[j].pool;
        if (!decode_supported(pj.d_in, pj.d_out))
            return cudaErrorNotSupported;
        max_din = pj.d_in > max_din ? pj.d_in : max_din;
        max_r = pj.r_max > max_r ? pj.r_max : max_r;
        a.p[j].zoff = zcols;
        zcols += z_stride(pj.r_max);
    }
    if (zcols > Z_ROW_FLOATS)
        return cudaErrorNotSupported;
    static thread_local int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(k_dec_shrink_multi, cudaFuncAttributeMaxDynamicSharedMemorySize, DS_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    // shrink: one row group per rpc rank rows of each projection
    const int rpc = max_r <= 8 ? 4 : 8;
    a.gpre[0] = 0;
    for (int j = 0; j < a.n; ++j)
        a.gpre[j + 1] = a.gpre[j] + (a.p[j].pool.r_max + rpc - 1) / rpc;
    // expand: T x column chunks of each projection
    a.wpre[0] = 0;
    for (int j = 0; j < a.n; ++j) {
        a.p[j].nc = (a.p[j].pool.d_out + 255) / 256;
        a.wpre[j + 1] = a.wpre[j] + a.T * a.p[j].nc;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t scfg = {};
    scfg.gridDim = dim3(P, a.gpre[a.n], 1);
    scfg.blockDim = dim3(32 * rpc, 1, 1);
    scfg.dynamicSmemBytes = (size_t)max_din * 2;
    scfg.stream = st;
    scfg.attrs = attr;
    scfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&scfg, k_dec_shrink_multi, a);
    if (e != cudaSuccess)
        return e;
    const long long warps = a.wpre[a.n];
    int wpc = 8;
    while (wpc > 1 && (warps + wpc - 1) / wpc < sm_count())
        wpc >>= 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + wpc - 1) / wpc), 1, 1);
    cfg.blockDim = dim3(32 * wpc, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (warps > 8LL * sm_count())
        return cudaLaunchKernelEx(&cfg, k_dec_expand_multi<2, 2>, a);
    return cudaLaunchKernelEx(&cfg, k_dec_expand_multi<DE_PP, 1>, a);
}

}  // namespace tcl
