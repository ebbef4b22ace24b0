// Shrink: z_q[j] = alpha_q * sum_{d < d_in} x[tok_q, d] * A_{a_q}[d, j]   for j < k_{a_q}
//
// LoRAForge summary page, "Approach" (4) and "Developer view": the shrink
// keeps the retained rank k_m (a rank-aware segmented shrink, CSGMV) so that
// only the first k rows of the factor are read.  DyMerge-LoRA summary page,
// "Core idea" (paper Sec. 4.3): one CTA processes the tokens of one adapter
// together, so the adapter's A is read once for all of them.  The alpha of
// each pair is folded into z here (the delta is linear in alpha, DyMerge-LoRA
// page, "Core idea", paper Sec. 3.1 M1).
//
// Work unit = (segment tile of <= SHRINK_TT pairs of one adapter, group of <=
// SHRINK_RG retained rows); a unit is streamed as one or more entries (d_in
// chunks sized so the unit's rows of a chunk fit SHRINK_ENTRY_BYTES; whole
// rows when they fit, so a unit's A rows are a single copy).  Units are numbered rowgroup-major over the
// host-known tile bound, so a CTA resolves its units with one round trip
// (tile record and its token list, same index) and the retained ranks come
// from a table staged in shared memory.  The pool stores A transposed
// (r_max x d_in): a unit's rows are 16-byte-aligned contiguous runs that all
// threads stream with 16-byte asynchronous copies into a byte ring in shared
// memory, each entry (unit, d_in chunk) completing on its own mbarrier
// (cp.async.mbarrier.arrive); entries are issued as long as ring space and
// barrier slots allow, so every byte a CTA needs is in flight from the start
// when it fits.  (One thread issuing a bulk copy per row was measured to
// serialise on the copy engine: ~0.2 us per copy.)  Each thread owns one
// 16-byte vector of every staged row, accumulates SHRINK_TT x SHRINK_RG fp32
// partial dot products, and the CTA reduces them with a warp-shuffle
// reduce-scatter (32 values over 32 lanes in 31 shuffles) and one cross-warp
// pass.
//
// Persistent grid; griddepcontrol.launch_dependents at entry lets the expand
// kernel that follows start staging B while this one runs.
#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int TT = SHRINK_TT, RG = SHRINK_RG;
constexpr int RING = SHRINK_RING_BYTES, MAXE = SHRINK_MAX_INFLIGHT, EMAX = SHRINK_ENTRY_BYTES;
constexpr int MAX_LIST = SHRINK_THREADS;
static_assert(TT * RG == 32, "one reduced value per lane");
static_assert(EMAX <= RING, "one entry of any shape fits the empty ring");
static_assert((RG + TT) * 64 * 2 <= EMAX, "a 64-element chunk of any unit fits an entry");

struct ShrinkArgs {
    const __nv_bfloat16 *x;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int rg;          // rows per unit, <= RG
    int zs;          // z row stride (floats)
    int tile_bound;  // tile slots written by the mapping
    int use_tab;     // ranks staged in shared memory
};

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

__global__ void __launch_bounds__(SHRINK_THREADS, 2) k_shrink(ShrinkArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *ring = smem_raw;
    int *rank_tab = reinterpret_cast<int *>(smem_raw + RING);
    __shared__ __align__(8) uint64_t bar[MAXE];
    __shared__ float red[2][8][32];
    __shared__ int4 s_unit[MAX_LIST];  // {adapter, q0, n, (j0 << 8) | R}
    __shared__ int s_tok[MAX_LIST][TT];
    __shared__ short s_clen[MAX_LIST];  // d_in chunk of the unit's entries (multiple of 64)
    __shared__ int s_wcount[8];

    pdl_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d_in = a.pool.d_in, r_max = a.pool.r_max;
    int32_t *status = a.m.hdr + HDR_STATUS;
    const int rgm = (r_max + a.rg - 1) / a.rg;
    const long long nunits = (long long)a.tile_bound * rgm;

    if (a.use_tab)
        for (int i = tid; i < a.pool.capacity; i += SHRINK_THREADS)
            rank_tab[i] = effective_rank(a.pool, a.ranks, i);
    if (tid == 0) {
        for (int s = 0; s < MAXE; ++s)
            mbar_init(&bar[s], SHRINK_THREADS);
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t e_base = 0;  // entry sequence number of this pass's first entry
    int unit_parity = 0;
    for (long long pass = blockIdx.x; pass < nunits; pass += (long long)gridDim.x * MAX_LIST) {
        // ---- resolve this pass's units (one round trip) and compact the live ones
        const long long u = pass + (long long)tid * gridDim.x;
        bool live = false;
        int4 rec = make_int4(0, 0, 0, 0);
        int toks[TT];
        if (u < nunits) {
            const int rg = (int)(u / a.tile_bound), tile = (int)(u % a.tile_bound);
            const int4 t = a.m.tile[tile];  // {adapter, q0, n, segment}; n = 0: empty slot
            const int4 tk0 = reinterpret_cast<const int4 *>(a.m.tile_tok)[2 * tile];
            const int4 tk1 = reinterpret_cast<const int4 *>(a.m.tile_tok)[2 * tile + 1];
            toks[0] = tk0.x; toks[1] = tk0.y; toks[2] = tk0.z; toks[3] = tk0.w;
            toks[4] = tk1.x; toks[5] = tk1.y; toks[6] = tk1.z; toks[7] = tk1.w;
            if (t.z > 0) {
                const int k = a.use_tab ? rank_tab[t.x] : effective_rank(a.pool, a.ranks, t.x);
                if (k < 0) {
                    if (rg == 0)
                        atomicOr(status, k == -1 ? LORA_DEV_UNREGISTERED : LORA_DEV_BAD_RANK);
                } else {
                    const int j0 = rg * a.rg;
                    if (j0 < k) {
                        live = true;
                        rec = make_int4(t.x, t.y, t.z, (j0 << 8) | min(a.rg, k - j0));
                    }
                }
            }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, live);
        if (lane == 0)
            s_wcount[warp] = __popc(bal);
        __syncthreads();
        int before = 0, L = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            before += (w < warp) ? s_wcount[w] : 0;
            L += s_wcount[w];
        }
        int my_nch = 0;
        if (live) {
            const int idx = before + __popc(bal & ((1u << lane) - 1u));
            s_unit[idx] = rec;
#pragma unroll
            for (int i = 0; i < TT; ++i)
                s_tok[idx][i] = toks[i];
            // longest chunk (multiple of 64 elements) whose rows fit one entry
            const int rows = (rec.w & 0xff) + rec.z;
            const int clen = min(d_in, (EMAX / (2 * rows)) & ~63);
            s_clen[idx] = (short)clen;
            my_nch = (d_in + clen - 1) / clen;
        }
        __syncthreads();
        // entries of this pass = sum over units of their chunk counts
        const unsigned nb = __reduce_add_sync(0xffffffffu, (unsigned)my_nch);
        if (lane == 0)
            s_wcount[warp] = (int)nb;
        __syncthreads();
        int total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w)
            total += s_wcount[w];

        // ---- entries (unit, chunk) in order through the byte ring.  Every thread
        // runs the same allocation (uniform state) and issues its share of each
        // entry's 16-byte copies; the entry's mbarrier completes when all
        // threads' copies have landed.
        int my_off[MAXE];  // ring offset of the entries in flight, by slot
        int p_next = 0, p_e = 0, p_ch = 0, head = 0;
        auto issue_more = [&](int c_done) {
            while (p_next < total && p_next - c_done < MAXE) {
                const int4 r = s_unit[p_e];
                const int n = r.z, R = r.w & 0xff, j0 = r.w >> 8;
                const int clen_u = s_clen[p_e];
                const int c0 = p_ch * clen_u, clen = min(clen_u, d_in - c0);
                const int size = (R + n) * clen * 2;
                int pos;
                if (p_next == c_done) {
                    pos = 0;  // ring empty
                } else {
                    const int tail = my_off[(e_base + c_done) % MAXE];
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
                const int slot = (e_base + p_next) % MAXE;
                my_off[slot] = pos;
                const int vpr = clen / 8;  // 16-byte vectors per row
                const int nvec = (R + n) * vpr;
                unsigned char *dst = ring + pos;
                const __nv_bfloat16 *Abase = a.pool.At + ((size_t)r.x * r_max + j0) * d_in + c0;
                for (int v = tid; v < nvec; v += SHRINK_THREADS) {
                    const int row = v / vpr, cv = v - row * vpr;
                    const __nv_bfloat16 *src = row < R ? Abase + (size_t)row * d_in + cv * 8
                                                       : a.x + (size_t)s_tok[p_e][row - R] * d_in + c0 + cv * 8;
                    cp_async16(dst + (size_t)v * 16, src);
                }
                cp_async_mbar_arrive(&bar[slot]);
                head = pos + size;
                ++p_next;
                if (c0 + clen >= d_in) {
                    ++p_e;
                    p_ch = 0;
                } else {
                    ++p_ch;
                }
            }
        };
        issue_more(0);

        float acc[TT][RG];
        int c_e = 0, c_ch = 0;  // consumer: unit and chunk of entry c
        for (int c = 0; c < total; ++c) {
            const uint32_t g = e_base + c;
            const int slot = g % MAXE;
            const bool ok = mbar_wait_bounded(&bar[slot], (g / MAXE) & 1u, status);
            const int e = c_e, ch = c_ch;
            const int4 r = s_unit[e];
            const int n = r.z, R = r.w & 0xff;
            const int clen_u = s_clen[e];
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
                for (int i = 0; i < TT; ++i)
#pragma unroll
                    for (int rr = 0; rr < RG; ++rr)
                        acc[i][rr] = 0.f;
            }
            const __nv_bfloat16 *sA = reinterpret_cast<const __nv_bfloat16 *>(ring + my_off[slot]);
            for (int vb = tid * 8; ok && vb < clen; vb += SHRINK_THREADS * 8) {
                float av[RG][8];
#pragma unroll
                for (int rr = 0; rr < RG; ++rr)
                    if (rr < R)
                        unpack8(lds128(sA + rr * clen + vb), av[rr]);
#pragma unroll
                for (int i = 0; i < TT; ++i) {
                    if (i < n) {
                        float xv[8];
                        unpack8(lds128(sA + (R + i) * clen + vb), xv);
#pragma unroll
                        for (int rr = 0; rr < RG; ++rr) {
                            if (rr < R) {
                                float s = acc[i][rr];
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    s = fmaf(xv[v], av[rr][v], s);
                                acc[i][rr] = s;
                            }
                        }
                    }
                }
            }
            if (last) {
                // reduce-scatter: lane l ends with the warp sum of value l = i * RG + r
                float v[32];
#pragma unroll
                for (int i = 0; i < TT; ++i)
#pragma unroll
                    for (int rr = 0; rr < RG; ++rr)
                        v[i * RG + rr] = acc[i][rr];
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int i = 0; i < off; ++i) {
                        const float send = upper ? v[i] : v[i + off];
                        const float keep = upper ? v[i + off] : v[i];
                        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                red[unit_parity][warp][lane] = v[0];
            }
            const int any_bad = __syncthreads_or(!ok);
            if (any_bad)
                return;  // a copy never landed: the status word records it
            issue_more(c + 1);
            if (last) {
                if (warp == 0) {
                    float s = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        s += red[unit_parity][w][lane];
                    const int i = lane / RG, rr = lane % RG, j0 = r.w >> 8;
                    if (i < n && rr < R) {
                        const int q = r.y + i;
                        a.m.z[(size_t)q * a.zs + j0 + rr] = a.m.alpha[q] * s;
                    }
                }
                unit_parity ^= 1;
            }
        }
        e_base += (uint32_t)total;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_shrink(const __nv_bfloat16 *x, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int P, int rg, int grid, cudaStream_t st)
{
    const int use_tab = pool.capacity <= RANK_TAB_MAX ? 1 : 0;
    const size_t smem = (size_t)RING + (use_tab ? (size_t)((pool.capacity + 3) & ~3) * sizeof(int) : 0);
    static int attr_done = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_shrink, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             RING + RANK_TAB_MAX * (int)sizeof(int));
        // the largest shared-memory carveout, so an expand CTA fits beside this one
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_shrink, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    ShrinkArgs a{x, pool, ranks, m, rg, z_stride(pool.r_max), shrink_tile_bound(P, pool.capacity), use_tab};
    k_shrink<<<grid, SHRINK_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace tcl
