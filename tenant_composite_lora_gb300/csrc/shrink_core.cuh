// Shrink phase, shared by the split path (k_shrink) and the fused decode
// kernel (k_fused):
//
//   z_q[j] = alpha_q * sum_{d < d_in} x[tok_q, d] * A_{a_q}[d, j]   for j < k_{a_q}
//
// LoRAForge summary page, "Approach" (4) and "Developer view": a rank-aware
// segmented shrink (CSGMV) that reads only the first k rows of the factor.
// DyMerge-LoRA summary page, "Core idea" (paper Sec. 4.3): one CTA processes
// the tokens of one adapter together, so the adapter's A rows are read once
// for all of them; alpha is folded into z (the delta is linear in alpha,
// paper Sec. 3.1 M1).
//
// Work unit = (shrink tile of n <= SHRINK_TT pairs of one adapter, a group of
// retained rows).  The group size depends on n so that the n x rows partial
// sums fill 32 accumulators per thread (n = 1 -> 32 rows, 2 -> 16, 3..4 -> 8,
// 5..8 -> 4 in the wide set; 8 or 4 rows in the narrow set the split kernel
// uses to fit its register budget); a tile's x rows are re-read once per
// group.  Every CTA scans the tile records (rounds of
// SHRINK_ROUND_TILES) and the ranks, counts each tile's units and takes units
// cta, cta + ncta, ... of the resulting list, so live work is spread evenly
// over all CTAs.
//
// The pool stores A transposed (r_max x d_in): a unit's rows are
// 16-byte-aligned contiguous runs.  Each entry (a unit's rows over one d_in
// chunk; whole rows when they fit the entry size, so that the unit's A rows
// are a single copy) streams into a byte ring in shared memory with bulk
// (TMA) copies that complete on the entry's mbarrier; entries are issued as
// long as ring space and barrier slots allow.  (16-byte cp.async copies from
// every thread were measured to cap a CTA near 20 GB/s: each ties up an L1
// miss slot, while the copy engine keeps far more bytes in flight.)
// Each thread owns 16-byte vectors of every staged row, accumulates 32 fp32
// partial dot products, and the CTA reduces them with a warp-shuffle
// reduce-scatter (32 values over 32 lanes in 31 shuffles) and one cross-warp
// pass.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace tcl {

constexpr int SHR_MAXE = SHRINK_MAX_INFLIGHT;
constexpr int SHR_LIST = SHRINK_THREADS;  // units resolved per pass
static_assert(SHRINK_THREADS == 256, "8 warps");
static_assert((SHRINK_TT + 4) * 64 * 2 <= SHRINK_MIN_ENTRY, "a 64-element chunk of a unit with 4 rows fits");

struct ShrinkArgs {
    const __nv_bfloat16 *x;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int zs;          // z row stride (floats)
    int tile_bound;  // tile slots written by the mapping
    int use_tab;     // ranks staged in shared memory
    int ring_bytes;   // size of the entry ring
    int entry_bytes;  // largest entry (a unit's rows over one d_in chunk)
};

// Static shared state of the shrink phase.
struct ShrinkShared {
    uint64_t bar[SHR_MAXE];
    float red[2][8][32];
    int4 unit[SHR_LIST];  // {adapter, q0, n, (j0 << 8) | R}
    int tok[SHR_LIST][SHRINK_TT];
    float alpha[SHR_LIST][SHRINK_TT];  // pair weights of each unit's tile
    short clen[SHR_LIST];
    int wsum[8];
    int capsum[6][8];
    int2 tcache[SHRINK_ROUND_TILES];  // {adapter | n << 16 | k << 20, q0} per tile of the round
    int prefix[SHRINK_ROUND_TILES + 1];
};

// Rows per unit for a tile of n pairs.  WIDE: four shapes (1 x 32, 2 x 16,
// 4 x 8, 8 x 4); otherwise two (4 x 8, 8 x 4), which fit 136 registers.
template <bool WIDE>
__device__ __forceinline__ int shrink_rows_for(int n)
{
    if constexpr (WIDE)
        return n <= 1 ? 32 : (n <= 2 ? 16 : (n <= 4 ? 8 : 4));
    else
        return n <= 4 ? 8 : 4;
}

__device__ __forceinline__ void unpack8(const uint4 w, float f[8])
{
    f[0] = bf16lo(w.x);
    f[1] = bf16hi(w.x);
    f[2] = bf16lo(w.y);
    f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z);
    f[5] = bf16hi(w.z);
    f[6] = bf16lo(w.w);
    f[7] = bf16hi(w.w);
}

// acc[i * RGV + r] += x_i . A_r over this thread's vectors of one entry.
// Few tokens: the token vectors stay in registers and the rows stream by;
// eight tokens: the four row vectors stay in registers and the tokens stream.
template <int TTV, int RGV>
__device__ __forceinline__ void shrink_entry(const __nv_bfloat16 *sA, int clen, int n, int R, float (&acc)[32])
{
    for (int vb = threadIdx.x * 8; vb < clen; vb += SHRINK_THREADS * 8) {
        if constexpr (TTV <= 4) {
            float xv[TTV][8];
#pragma unroll
            for (int i = 0; i < TTV; ++i)
                if (i < n)
                    unpack8(lds128(sA + (R + i) * clen + vb), xv[i]);
#pragma unroll
            for (int r = 0; r < RGV; ++r) {
                if (r < R) {
                    float av[8];
                    unpack8(lds128(sA + r * clen + vb), av);
#pragma unroll
                    for (int i = 0; i < TTV; ++i) {
                        if (i < n) {
                            float s = acc[i * RGV + r];
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                s = fmaf(xv[i][v], av[v], s);
                            acc[i * RGV + r] = s;
                        }
                    }
                }
            }
        } else {
            float av[RGV][8];
#pragma unroll
            for (int r = 0; r < RGV; ++r)
                if (r < R)
                    unpack8(lds128(sA + r * clen + vb), av[r]);
#pragma unroll
            for (int i = 0; i < TTV; ++i) {
                if (i < n) {
                    float xv[8];
                    unpack8(lds128(sA + (R + i) * clen + vb), xv);
#pragma unroll
                    for (int r = 0; r < RGV; ++r) {
                        if (r < R) {
                            float s = acc[i * RGV + r];
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                s = fmaf(xv[v], av[r][v], s);
                            acc[i * RGV + r] = s;
                        }
                    }
                }
            }
        }
    }
}

// Block-wide exclusive scan of s[0..n) in place (n <= SHRINK_ROUND_TILES);
// s[n] receives the total.
__device__ __forceinline__ void shrink_scan(int *s, int n, int *wsum)
{
    constexpr int PER = SHRINK_ROUND_TILES / SHRINK_THREADS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = tid * PER;
    int loc[PER], sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        loc[i] = (b0 + i < n) ? s[b0 + i] : 0;
        sum += loc[i];
    }
    int inc = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off)
            inc += o;
    }
    if (lane == 31)
        wsum[warp] = inc;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        before += (w < warp) ? wsum[w] : 0;
        total += wsum[w];
    }
    int run = before + inc - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        if (b0 + i < n)
            s[b0 + i] = run;
        run += loc[i];
    }
    if (tid == 0)
        s[n] = total;
    __syncthreads();
}

// The whole shrink of this CTA: units cta, cta + ncta, ... of the live list,
// as a small state machine so that a caller can put other work between the
// first copies being issued and their consumption:
//   begin()  barriers, first round's scan, first pass resolved, its copies issued
//   finish() consume that pass, then every further pass and round
// ring: ring_bytes of shared memory; rank_tab: staged ranks (if use_tab).
// finish() returns false if a bounded wait expired (the status word records it).
template <bool WIDE>
struct ShrinkRun {
    const ShrinkArgs &a;
    ShrinkShared &sh;
    unsigned char *ring;
    const int *rank_tab;
    int cta, ncta;
    // round / pass
    int rbase = 0, ntr = 0, total_r = 0, cap_rows = 1, pass = 0, total = 0;
    bool has_pass = false;
    // ring producer (uniform across threads)
    int p_next = 0, p_e = 0, p_ch = 0, head = 0;
    int my_off[SHR_MAXE];
    uint32_t e_base = 0;  // entry sequence number (drives barrier slot and parity)
    int unit_parity = 0;

    __device__ ShrinkRun(const ShrinkArgs &a_, ShrinkShared &sh_, unsigned char *ring_, const int *rank_tab_,
                         int cta_, int ncta_)
        : a(a_), sh(sh_), ring(ring_), rank_tab(rank_tab_), cta(cta_), ncta(ncta_)
    {
    }

    // Units of every tile of the round at rbase.  Rows per unit: the tile
    // shape's maximum, capped by the largest cap in {32, 16, 8, 4, 2, 1} that
    // still gives at least one unit per CTA (small batches spread over all SMs).
    __device__ void scan()
    {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        int32_t *status = a.m.hdr + HDR_STATUS;
        ntr = min(SHRINK_ROUND_TILES, a.tile_bound - rbase);
        int part[6] = {0, 0, 0, 0, 0, 0};
        for (int i = tid; i < ntr; i += SHRINK_THREADS) {
            const int4 t = a.m.tile[rbase + i];  // {adapter, q0, n, segment}; n = 0: empty slot
            int k = 0;
            if (t.z > 0) {
                k = a.use_tab ? rank_tab[t.x] : effective_rank(a.pool, a.ranks, t.x);
                if (k < 0) {
                    atomicOr(status, k == -1 ? LORA_DEV_UNREGISTERED : LORA_DEV_BAD_RANK);
                    k = 0;
                }
                const int rmax = shrink_rows_for<WIDE>(t.z);
#pragma unroll
                for (int ci = 0; ci < 6; ++ci) {
                    const int rows = min(rmax, 32 >> ci);
                    part[ci] += (k + rows - 1) / rows;
                }
            }
            sh.tcache[i] = make_int2(t.x | (t.z << 16) | (k << 20), t.y);
        }
#pragma unroll
        for (int ci = 0; ci < 6; ++ci) {
            const int v = __reduce_add_sync(0xffffffffu, part[ci]);
            if (lane == 0)
                sh.capsum[ci][warp] = v;
        }
        __syncthreads();
        cap_rows = 1;
#pragma unroll
        for (int ci = 5; ci >= 0; --ci) {
            int tot = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                tot += sh.capsum[ci][w];
            if (tot >= ncta)
                cap_rows = 32 >> ci;  // the largest cap that still fills the grid
        }
        for (int i = tid; i < ntr; i += SHRINK_THREADS) {
            const int2 tc = sh.tcache[i];
            const int n = (tc.x >> 16) & 0xf, k = (tc.x >> 20) & 0x7f;
            const int rows = min(shrink_rows_for<WIDE>(n), cap_rows);
            sh.prefix[i] = n > 0 ? (k + rows - 1) / rows : 0;
        }
        __syncthreads();
        shrink_scan(sh.prefix, ntr, sh.wsum);
        total_r = sh.prefix[ntr];
        __syncthreads();  // every thread has read total_r before anything rewrites it
    }

    // Moves to the next pass with work, scanning later rounds as needed.
    __device__ bool next_pass(bool first)
    {
        if (first) {
            rbase = 0;
            scan();
            pass = cta;
        } else {
            pass += ncta * SHR_LIST;
        }
        while (pass >= total_r) {
            rbase += SHRINK_ROUND_TILES;
            if (rbase >= a.tile_bound)
                return false;
            scan();
            pass = cta;
        }
        return true;
    }

    // Resolves this pass's units (unit record, tokens, pair weights, chunking)
    // and counts its entries.
    __device__ void resolve()
    {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        const int d_in = a.pool.d_in;
        const int u = pass + tid * ncta;
        int my_nch = 0;
        if (u < total_r) {
            int lo = 0, hi = ntr;  // last tile with prefix <= u
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sh.prefix[mid] <= u)
                    lo = mid;
                else
                    hi = mid;
            }
            const int2 tc = sh.tcache[lo];
            const int adapter = tc.x & 0xffff, n = (tc.x >> 16) & 0xf, k = (tc.x >> 20) & 0x7f;
            const int rows = min(shrink_rows_for<WIDE>(n), cap_rows);
            const int j0 = (u - sh.prefix[lo]) * rows;
            const int R = min(rows, k - j0);
            sh.unit[tid] = make_int4(adapter, tc.y, n, (j0 << 8) | R);
            const int4 tk0 = reinterpret_cast<const int4 *>(a.m.tile_tok)[2 * (rbase + lo)];
            const int4 tk1 = reinterpret_cast<const int4 *>(a.m.tile_tok)[2 * (rbase + lo) + 1];
            sh.tok[tid][0] = tk0.x;
            sh.tok[tid][1] = tk0.y;
            sh.tok[tid][2] = tk0.z;
            sh.tok[tid][3] = tk0.w;
            sh.tok[tid][4] = tk1.x;
            sh.tok[tid][5] = tk1.y;
            sh.tok[tid][6] = tk1.z;
            sh.tok[tid][7] = tk1.w;
#pragma unroll
            for (int i = 0; i < SHRINK_TT; ++i)
                sh.alpha[tid][i] = i < n ? a.m.alpha[tc.y + i] : 0.f;
            // longest chunk (multiple of 64 elements) whose rows fit one entry
            const int clen = min(d_in, max(64, (a.entry_bytes / (2 * (R + n))) & ~63));
            sh.clen[tid] = (short)clen;
            my_nch = (d_in + clen - 1) / clen;
        }
        const unsigned nb = __reduce_add_sync(0xffffffffu, (unsigned)my_nch);
        if (lane == 0)
            sh.wsum[warp] = (int)nb;
        __syncthreads();
        total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w)
            total += sh.wsum[w];
        p_next = p_e = p_ch = head = 0;
    }

    // Entries (unit, chunk) in order through the byte ring.  Every thread runs
    // the same allocation (uniform state); thread 0 issues the bulk copies.
    __device__ void issue_more(int c_done)
    {
        const int d_in = a.pool.d_in, r_max = a.pool.r_max, RING = a.ring_bytes;
        while (p_next < total && p_next - c_done < SHR_MAXE) {
            const int4 r = sh.unit[p_e];
            const int n = r.z, R = r.w & 0xff, j0 = r.w >> 8;
            const int clen_u = sh.clen[p_e];
            const int c0 = p_ch * clen_u, clen = min(clen_u, d_in - c0);
            const int size = (R + n) * clen * 2;
            int pos;
            if (p_next == c_done) {
                pos = 0;  // ring empty
            } else {
                const int tail = my_off[(e_base + c_done) % SHR_MAXE];
                if (head > tail) {
                    if (head + size <= RING)
                        pos = head;
                    else if (size < tail)
                        pos = 0;
                    else
                        break;
                } else {
                    if (head + size < tail)
                        pos = head;
                    else
                        break;
                }
            }
            const int slot = (e_base + p_next) % SHR_MAXE;
            my_off[slot] = pos;
            if (threadIdx.x == 0) {
                const uint32_t row_bytes = (uint32_t)clen * 2u;
                unsigned char *dst = ring + pos;
                mbar_arrive_expect_tx(&sh.bar[slot], row_bytes * (uint32_t)(R + n));
                const __nv_bfloat16 *Abase = a.pool.At + ((size_t)r.x * r_max + j0) * d_in + c0;
                if (clen == d_in) {  // whole rows: the unit's A rows are one contiguous run
                    bulk_g2s(dst, Abase, row_bytes * (uint32_t)R, &sh.bar[slot]);
                } else {
                    for (int rr = 0; rr < R; ++rr)
                        bulk_g2s(dst + rr * row_bytes, Abase + (size_t)rr * d_in, row_bytes, &sh.bar[slot]);
                }
                for (int i = 0; i < n; ++i)
                    bulk_g2s(dst + (R + i) * row_bytes, a.x + (size_t)sh.tok[p_e][i] * d_in + c0, row_bytes,
                             &sh.bar[slot]);
            }
            head = pos + size;
            ++p_next;
            if (c0 + clen >= d_in) {
                ++p_e;
                p_ch = 0;
            } else {
                ++p_ch;
            }
        }
    }

    // Consumes the current pass's entries (issuing more as space frees up).
    __device__ bool consume()
    {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        const int d_in = a.pool.d_in;
        int32_t *status = a.m.hdr + HDR_STATUS;
        float acc[32];
        float alpha_i = 0.f;
        int c_e = 0, c_ch = 0;  // unit and chunk of entry c
        for (int c = 0; c < total; ++c) {
            const uint32_t g = e_base + c;
            const int slot = g % SHR_MAXE;
            const bool ok = mbar_wait_bounded(&sh.bar[slot], (g / SHR_MAXE) & 1u, status);
            const int e = c_e, ch = c_ch;
            const int4 r = sh.unit[e];
            const int n = r.z, R = r.w & 0xff;
            const int rows = shrink_rows_for<WIDE>(n);  // accumulator shape (R <= rows)
            const int clen_u = sh.clen[e];
            const int clen = min(clen_u, d_in - ch * clen_u);
            const bool last = (ch * clen_u + clen >= d_in);
            if (last) {
                ++c_e;
                c_ch = 0;
            } else {
                ++c_ch;
            }
            if (ch == 0) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    acc[i] = 0.f;
                const int i = lane / rows;  // this lane's pair, needed at the end of the unit
                alpha_i = i < SHRINK_TT ? sh.alpha[e][i] : 0.f;
            }
            const __nv_bfloat16 *sA = reinterpret_cast<const __nv_bfloat16 *>(ring + my_off[slot]);
            if (ok) {
                if constexpr (WIDE) {
                    switch (rows) {
                    case 32:
                        shrink_entry<1, 32>(sA, clen, n, R, acc);
                        break;
                    case 16:
                        shrink_entry<2, 16>(sA, clen, n, R, acc);
                        break;
                    case 8:
                        shrink_entry<4, 8>(sA, clen, n, R, acc);
                        break;
                    default:
                        shrink_entry<8, 4>(sA, clen, n, R, acc);
                        break;
                    }
                } else {
                    if (rows == 8)
                        shrink_entry<4, 8>(sA, clen, n, R, acc);
                    else
                        shrink_entry<8, 4>(sA, clen, n, R, acc);
                }
            }
            if (last) {
                // reduce-scatter: lane l ends with the warp sum of value l
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < off; ++i) {
                        const float send = upper ? acc[i] : acc[i + off];
                        const float keep = upper ? acc[i + off] : acc[i];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                sh.red[unit_parity][warp][lane] = acc[0];
            }
            const int any_bad = __syncthreads_or(!ok);
            if (any_bad)
                return false;
            issue_more(c + 1);
            if (last) {
                if (warp == 0) {
                    float s = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        s += sh.red[unit_parity][w][lane];
                    const int i = lane / rows, rr = lane % rows, j0 = r.w >> 8;
                    if (i < n && rr < R)
                        a.m.z[(size_t)(r.y + i) * a.zs + j0 + rr] = alpha_i * s;
                }
                unit_parity ^= 1;
            }
        }
        e_base += (uint32_t)total;
        __syncthreads();
        return true;
    }

    // Barriers, the first pass resolved and its first copies issued.
    __device__ void begin()
    {
        if (threadIdx.x == 0) {
            for (int s = 0; s < SHR_MAXE; ++s)
                mbar_init(&sh.bar[s], 1);
            fence_mbar_init();
        }
        __syncthreads();
        has_pass = next_pass(true);
        if (has_pass) {
            resolve();
            issue_more(0);
        }
    }

    // Everything else; false if a bounded wait expired.
    __device__ bool finish()
    {
        while (has_pass) {
            if (!consume())
                return false;
            has_pass = next_pass(false);
            if (has_pass) {
                resolve();
                issue_more(0);
            }
        }
        return true;
    }
};

// The whole shrink of this CTA in one call.
template <bool WIDE>
__device__ __forceinline__ bool shrink_phase(const ShrinkArgs &a, ShrinkShared &sh, unsigned char *ring,
                                             const int *rank_tab, int cta, int ncta)
{
    ShrinkRun<WIDE> run(a, sh, ring, rank_tab, cta, ncta);
    run.begin();
    return run.finish();
}

}  // namespace tcl
