// Tensor-core (tcgen05) path for prefill batches, where a segment holds many
// tokens of one adapter and a tile of consecutive tokens touches few
// adapters.  Two kernels chained with programmatic dependent launch:
//
// 1. Segment shrink (the shrink step of the composite delta, with the weight
//    folded in as in the linear-weight definition of the composite adapter):
//    a tile is up to MMA_TM sorted pairs of one adapter a;
//        Z[tile rows, :n_k] = X[tok rows, :] . A_a[:, :n_k]
//    on the tensor cores (M = 128 pair rows, N = 16 * ceil(k / 16),
//    K = d_in), with the K dimension split over a cluster of CK CTAs.  The x
//    rows are gathered with 16-byte asynchronous copies into the 128-byte
//    swizzled K-major operand layout; A (stored transposed, K-major) comes by
//    TMA.  Each CTA's fp32 partial leaves tensor memory for shared memory and
//    the cluster adds them in rank order through distributed shared memory
//    (deterministic), scales by alpha and writes z[q][j], j < k.
//
// 2. Token-tile expand (RowExpand as a dense product): a unit is MMA_TM
//    consecutive tokens x BN output columns; a persistent CTA per SM takes a
//    contiguous run of units (mostly of one token tile).  The tile's adapters, in
//    ascending id order, each give ceil(k / 16) "slots" of 16 rank rows; the
//    A operand holds, per token and slot, the sum of the token's z rows for
//    that adapter (zero elsewhere), split into a bf16 high part and a bf16
//    residual (hi + lo carries ~16 significant bits of the fp32 z), and the
//    B operand is B_a[16c .. 16c + 15, columns] loaded by TMA in the
//    MN-major 128-byte swizzled layout (B is stored row-major, d_out
//    contiguous).  D (128 x BN fp32) accumulates in tensor memory over all
//    slots, in two buffers so that one unit's epilogue (y + D, rounded once
//    to bf16) overlaps the next unit's MMAs.  Warp roles: one streams B by
//    TMA through a ring of stages of ME_SPS chunks (one barrier per stage),
//    one issues the MMAs, eight list the tile's adapters and build the
//    operand (ME_SMAX slots per pass), four run the epilogues of the units
//    the workers queue.  Rank rows at or beyond k of a partial chunk are
//    zeroed in shared memory before use, so padding never reaches the sum.
//
// LoRAForge page, "Approach" (5) (a path fixed per phase and shape) and the
// DyMerge-LoRA page, "Core idea" (tuples reordered by adapter so that one CTA
// runs one adapter's tokens back to back).
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace tcl {

namespace {

// ---------------------------------------------------------------- shrink

constexpr int MS_THREADS = 192;  // warps 0-3: x gather + epilogue; warp 4: MMA; warp 5: A by TMA
constexpr int MS_STAGES = 4;
constexpr int MS_LAG = 3;                        // cp.async groups kept in flight per gather thread, < MS_STAGES
constexpr int MS_X_BYTES = MMA_TM * 128;         // 128 rows x 64 bf16
constexpr int MS_A_BYTES = LORA_MAX_RANK * 128;  // up to 64 rows x 64 bf16
constexpr int MS_SMEM_MAX = 1024 + MS_STAGES * (MS_X_BYTES + MS_A_BYTES);
constexpr int MS_PART_STRIDE = LORA_MAX_RANK + 4;  // fp32 partial row stride (floats)
static_assert(MS_LAG < MS_STAGES, "the gather runs at most MS_STAGES stages ahead of the MMAs");
static_assert(MMA_TM * MS_PART_STRIDE * 4 <= MS_STAGES * (MS_X_BYTES + 16 * 128), "partial fits the stages");

// A stage holds the x rows and A's rows up to the pool's rank rounded to 16
// (a multiple of 2 KB, so every stage starts 1024-aligned); small ranks leave
// room for three CTAs per SM.
inline int ms_stage_bytes(int r_max)
{
    return MS_X_BYTES + ((r_max + 15) & ~15) * 128;
}

struct MmaShrinkArgs {
    const __nv_bfloat16 *x;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int zs;  // z row stride (floats)
    int ck;  // CTAs per cluster (K split)
    int sb;  // bytes per pipeline stage (ms_stage_bytes)
};

__device__ __forceinline__ uint32_t xrow_offset(int row, int ch)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(MS_THREADS, 1)
    k_mma_shrink(const __grid_constant__ CUtensorMap map_at, const MmaShrinkArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t full_x[MS_STAGES], full_a[MS_STAGES], empty[MS_STAGES], done;
    __shared__ uint32_t s_taddr;

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ck = a.ck;
    const uint32_t rank = cluster_ctarank();
    const int4 tile = a.m.mtile[blockIdx.x / ck];  // {adapter, q0, n, segment}
    if (tile.w < 0 || tile.z <= 0)
        return;  // whole cluster: same record
    const int adapter = tile.x, q0 = tile.y, n = tile.z;
    const int k = effective_rank(a.pool, a.ranks, adapter);
    if (k <= 0) {
        if (k < 0 && rank == 0 && tid == 0)
            atomicOr(a.m.hdr + HDR_STATUS, k == -1 ? LORA_DEV_UNREGISTERED : LORA_DEV_BAD_RANK);
        return;  // whole cluster: same adapter
    }
    const int N = (k + 15) & ~15;
    const int d_in = a.pool.d_in;
    const int nkb = d_in / 64;
    const int kb0 = (int)rank * nkb / ck, kb1 = ((int)rank + 1) * nkb / ck;
    const int nk = kb1 - kb0;
    int32_t *status = a.m.hdr + HDR_STATUS;

    if (tid == 0) {
        for (int s = 0; s < MS_STAGES; ++s) {
            mbar_init(&full_x[s], 128);
            mbar_init(&full_a[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    if (warp == 4)
        tmem_alloc(&s_taddr, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = s_taddr;

    if (warp < 4) {
        // ---- x rows of the tile's pairs, gathered into the swizzled K-major layout.
        // Eight lanes share a row (16 bytes each), so one warp instruction moves
        // four whole 128-byte lines; warp w owns rows 32w .. 32w + 31.
        const int sub = lane >> 3, ch = lane & 7;
        const __nv_bfloat16 *xr[8];
        uint32_t dst[8];
        unsigned live = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = warp * 32 + i * 4 + sub;
            const bool valid = row < n;
            xr[i] = a.x + (valid ? (size_t)a.m.tok[q0 + row] * d_in : 0) + ch * 8;
            dst[i] = xrow_offset(row, ch);
            live |= valid ? 1u << i : 0u;
        }
        for (int it = 0; it < nk; ++it) {
            const int s = it % MS_STAGES;
            if (it >= MS_STAGES && !mbar_wait_bounded(&empty[s], ((it / MS_STAGES) - 1) & 1, status))
                break;
            unsigned char *sx = smem + s * a.sb;
            const size_t col = (size_t)(kb0 + it) * 64;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (live & (1u << i))
                    cp_async16(sx + dst[i], xr[i] + col);
            cp_async_commit();
            if (it >= MS_LAG) {
                cp_async_wait_group<MS_LAG>();
                fence_proxy_async_smem();
                mbar_arrive(&full_x[(it - MS_LAG) % MS_STAGES]);
            }
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        for (int it = nk - MS_LAG < 0 ? 0 : nk - MS_LAG; it < nk; ++it)
            mbar_arrive(&full_x[it % MS_STAGES]);
    } else if (warp == 5) {
        // ---- A_a rows [0, N) x 64 columns per stage, by TMA
        if (lane == 0) {
            const int row0 = adapter * a.pool.r_max;
            for (int it = 0; it < nk; ++it) {
                const int s = it % MS_STAGES;
                if (it >= MS_STAGES && !mbar_wait_bounded(&empty[s], ((it / MS_STAGES) - 1) & 1, status))
                    break;
                unsigned char *sa = smem + s * a.sb + MS_X_BYTES;
                mbar_arrive_expect_tx(&full_a[s], (uint32_t)N * 128);
                for (int c = 0; c < N / 16; ++c)
                    tma_load_2d(sa + c * 2048, &map_at, (kb0 + it) * 64, row0 + 16 * c, &full_a[s]);
            }
            // the last loads of every stage have landed before the CTA can exit
            for (int it = nk - MS_STAGES < 0 ? 0 : nk - MS_STAGES; it < nk; ++it)
                mbar_wait_bounded(&full_a[it % MS_STAGES], (it / MS_STAGES) & 1, status);
        }
    } else {
        // ---- warp 4: one thread issues the MMAs
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(MMA_TM, N);
            bool ok = true;
            for (int it = 0; it < nk && ok; ++it) {
                const int s = it % MS_STAGES;
                const uint32_t ph = (it / MS_STAGES) & 1;
                ok = mbar_wait_bounded(&full_x[s], ph, status) && mbar_wait_bounded(&full_a[s], ph, status);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t xs = smem_u32(smem + s * a.sb);
                const uint32_t as = xs + MS_X_BYTES;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(taddr, umma_desc_sw128(xs + kk * 32), umma_desc_sw128(as + kk * 32), idesc,
                              it > 0 || kk > 0);
                umma_commit(&empty[s]);
            }
            umma_commit(&done);
        }
    }

    // ---- epilogue: partial -> shared memory, cluster reduction in rank order
    __syncwarp();
    float *part = reinterpret_cast<float *>(smem);
    if (warp < 4) {
        const bool ok = mbar_wait_bounded(&done, 0, status);
        tc_fence_after();
        for (int c = 0; c < N; c += 16) {
            float v[16];
            tmem_ld16(taddr + ((uint32_t)(warp * 32) << 16) + c, v);
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(part + tid * MS_PART_STRIDE + c + j) =
                    ok ? make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc_fence_before();
    cluster_sync();
    const int rows_per = MMA_TM / ck;
    const int r0 = (int)rank * rows_per;
    const int n4 = N / 4;
    for (int i = tid; i < rows_per * n4; i += MS_THREADS) {
        const int row = r0 + i / n4, j = (i % n4) * 4;
        if (row >= n)
            continue;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < ck; ++r) {
            const float4 v = ld_dsmem_f4(part + row * MS_PART_STRIDE + j, (uint32_t)r);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        const int q = q0 + row;
        const float al = a.m.alpha[q];
        float *zr = a.m.z + (size_t)q * a.zs + j;
        if (j + 4 <= k) {
            *reinterpret_cast<float4 *>(zr) = make_float4(al * s.x, al * s.y, al * s.z, al * s.w);
        } else {
            const float sv[4] = {s.x, s.y, s.z, s.w};
            for (int e = 0; e < 4 && j + e < k; ++e)
                zr[e] = al * sv[e];
        }
    }
    cluster_sync();  // peers finished reading this CTA's partial
    tc_fence_after();
    if (warp == 4)
        tmem_dealloc(taddr, 64);
}

// ---------------------------------------------------------------- expand

constexpr int ME_WORKERS = 256;                        // warps 0-7: lists, A operand, epilogue
constexpr int ME_EPI = 128;                            // warps 10-13: epilogue (one TMEM lane quarter each)
constexpr int ME_THREADS = ME_WORKERS + 64 + ME_EPI;   // warp 8: MMA issue; warp 9: B chunks by TMA
constexpr int ME_JOBS = 4;                             // epilogue jobs queued by the workers
constexpr int ME_SMAX = 12;                            // slots per A-operand build (a multiple of 4)
constexpr int ME_Z_BYTES = MMA_TM * ME_SMAX * 16 * 2;  // one of hi / lo: 128 rows x 16 ME_SMAX bf16
constexpr int ME_B_BYTES = 16 * 256 * 2;               // one chunk: 16 rank rows x up to 256 columns
constexpr int ME_SPS = 4;                              // chunks (slots) per ring stage: one barrier each way
constexpr int ME_STAGES = 3;                           // ring stages of ME_SPS chunks (ME_SMAX chunks in all)
static_assert(ME_SMAX % ME_SPS == 0, "an operand pass fills whole stages");
constexpr int ME_PT_MAX = 512;                         // pairs of a tile cached in shared memory
constexpr int ME_NU_MAX = 512;                         // adapters listed per window

struct MmaExpandArgs {
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int T, zs;
    int n_nt;   // column tiles: d_out / BN
    int units;  // token tiles x column tiles
};

// Dynamic shared memory of the expand kernel (offsets from a 1024-aligned base).
struct MeLayout {
    int zhi, zlo, b, cache, list, lrank, sbase, toff, bitmap, wpre, total;
    __host__ __device__ explicit MeLayout(int capacity)
    {
        const int words = (((capacity + 31) / 32) + 3) & ~3;
        zhi = 0;
        zlo = zhi + ME_Z_BYTES;
        b = zlo + ME_Z_BYTES;
        cache = b + ME_STAGES * ME_SPS * ME_B_BYTES;  // int2 [ME_PT_MAX]: sorted position, adapter (-1: none)
        list = cache + ME_PT_MAX * 8;        // int [ME_NU_MAX]: adapters of the window, ascending
        lrank = list + ME_NU_MAX * 4;        // int [ME_NU_MAX]: their ranks
        sbase = lrank + ME_NU_MAX * 4;       // int [ME_NU_MAX + 1]: first slot of each
        toff = sbase + (ME_NU_MAX + 4) * 4;  // int [MMA_TM + 1]: pair offsets of the tile's tokens
        bitmap = toff + (MMA_TM + 4) * 4;    // uint32 [words]: adapters of the tile with k > 0
        wpre = bitmap + words * 4;           // int [words]: set bits before each word
        total = wpre + words * 4 + 1024;
    }
};

// One unit's epilogue, handed from the workers to the epilogue warps.
struct MeJob {
    int uu, t0, nrows, gi, done;
};

// One A-operand build, handed from the workers to the MMA warp.
struct MeBuild {
    int u0, u1;       // units [u0, u1) take their slots [s0, s1) from this operand
    int s0, s1;       // window slots held (operand column block jj = s - s0)
    int nu;           // adapters in the window lists
    int first, last;  // the build starts / ends each unit's sum
    int gi0;          // running index (in this CTA) of unit u0; accumulator buffer = index % 2
    int done;         // no further builds
};

__device__ __forceinline__ void me_bar() { asm volatile("bar.sync 1, %0;" ::"n"(ME_WORKERS) : "memory"); }

// Exclusive scan of one int over the ME_WORKERS worker threads.
__device__ __forceinline__ int me_scan(int v, int &total, int *sh /* [ME_WORKERS / 32 + 1] */)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off)
            inc += o;
    }
    if (lane == 31)
        sh[warp] = inc;
    me_bar();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < ME_WORKERS / 32; ++w) {
            const int t = sh[w];
            sh[w] = run;
            run += t;
        }
        sh[ME_WORKERS / 32] = run;
    }
    me_bar();
    const int r = sh[warp] + inc - v;
    total = sh[ME_WORKERS / 32];
    me_bar();
    return r;
}

// Slot j of the window -> listed adapter index (last u with sbase[u] <= j).
__device__ __forceinline__ int me_slot_owner(const int *sbase, int nu, int j)
{
    int lo = 0, hi = nu;  // sbase[lo] <= j < sbase[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sbase[mid] <= j)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Token row of the tile owning pair offset i (last row with toff[row] - p0 <= i).
__device__ __forceinline__ int me_pair_row(const int *toff, int nrows, int p0, int i)
{
    int lo = 0, hi = nrows;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (toff[mid] - p0 <= i)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// The B producer warp (lane 0): for each build, streams the B chunks of its
// (unit, slot) sequence through a ring of ME_STAGES stages of ME_SPS chunks
// -- one 3-D TMA box {64 columns, 16 rank rows, BN / 64 column blocks} per
// chunk, which lands in the MN-major swizzled operand layout, and one
// barrier per stage, so that each handshake with the MMA warp covers ME_SPS
// chunks -- refilling a stage as soon as the MMAs that read it complete.
// Per-slot rows are resolved once per build.
template <int BN>
__device__ __forceinline__ void me_producer_warp(const CUtensorMap &map_b, const MmaExpandArgs &a,
                                                 unsigned char *smem, const MeLayout &L, uint64_t *full_b,
                                                 uint64_t *empty_b, uint64_t *lready, uint64_t *lack,
                                                 const MeBuild *s_build, int32_t *status)
{
    if ((threadIdx.x & 31) != 0)
        return;
    unsigned char *sb = smem + L.b;
    const int *list = reinterpret_cast<const int *>(smem + L.list);
    const int *sbase = reinterpret_cast<const int *>(smem + L.sbase);
    const int r_max = a.pool.r_max;
    int g = 0;  // ring sequence
    for (int nb = 0;; ++nb) {
        // a build's slots are listed before its operand is built: its B
        // chunks stream while the workers build
        if (!mbar_wait_bounded(lready, nb & 1, status))
            return;
        const MeBuild bd = s_build[nb & 1];
        mbar_arrive(lack);  // read: the workers may announce the next build
        if (bd.done)
            return;
        const int nsl = bd.s1 - bd.s0;
        int rows[ME_SMAX];
#pragma unroll
        for (int j = 0; j < ME_SMAX; ++j) {
            rows[j] = 0;
            if (j < nsl) {
                const int s = bd.s0 + j, ui = me_slot_owner(sbase, bd.nu, s);
                rows[j] = list[ui] * r_max + 16 * (s - sbase[ui]);
            }
        }
        for (int uu = bd.u0; uu < bd.u1; ++uu) {
            const int z0 = (uu % a.n_nt) * (BN / 64);
#pragma unroll
            for (int j = 0; j < ME_SMAX; j += ME_SPS) {
                if (j < nsl) {
                    const int gs = g++, st = gs % ME_STAGES;
                    if (gs >= ME_STAGES && !mbar_wait_bounded(&empty_b[st], ((gs / ME_STAGES) - 1) & 1, status))
                        return;
                    const int nch = min(ME_SPS, nsl - j);  // chunks of this stage
                    mbar_arrive_expect_tx(&full_b[st], (uint32_t)(nch * 16 * BN * 2));
#pragma unroll
                    for (int h = 0; h < ME_SPS; ++h)
                        if (h < nch)
                            tma_load_3d(sb + (st * ME_SPS + h) * ME_B_BYTES, &map_b, 0, rows[j + h], z0, &full_b[st]);
                }
            }
        }
    }
}

// The MMA warp: waits for each build, then per (unit, slot) for its B chunk,
// masks rank rows >= k of a partial chunk, issues the hi and lo MMAs, frees
// the stage, and commits a unit's accumulator once its last slot is issued.
template <int BN>
__device__ __forceinline__ void me_mma_warp(unsigned char *smem, const MeLayout &L, uint64_t *full_b,
                                            uint64_t *empty_b, uint64_t *zready, uint64_t *zfree,
                                            uint64_t *acc_full, uint64_t *acc_empty, const MeBuild *s_build,
                                            uint32_t taddr, int32_t *status)
{
    const int lane = threadIdx.x & 31;
    unsigned char *sb = smem + L.b;
    const uint32_t zhi = smem_u32(smem + L.zhi), zlo = smem_u32(smem + L.zlo);
    const int *lrank = reinterpret_cast<const int *>(smem + L.lrank);
    const int *sbase = reinterpret_cast<const int *>(smem + L.sbase);
    const uint32_t idesc = umma_idesc_bf16(MMA_TM, BN) | (1u << 16);  // B operand MN-major
    int g = 0;                                                         // ring sequence
    for (int nb = 0;; ++nb) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(zready, nb & 1, status)))
            return;
        const MeBuild bd = s_build[nb & 1];
        if (bd.done)
            return;
        const int nsl = bd.s1 - bd.s0;
        int krs[ME_SMAX];  // rank rows of each slot's chunk (16 = full)
#pragma unroll
        for (int j = 0; j < ME_SMAX; ++j) {
            krs[j] = 16;
            if (j < nsl) {
                const int s = bd.s0 + j, ui = me_slot_owner(sbase, bd.nu, s);
                krs[j] = min(16, lrank[ui] - 16 * (s - sbase[ui]));
            }
        }
        bool ok = true;
        for (int uu = bd.u0; uu < bd.u1 && ok; ++uu) {
            const int gi = bd.gi0 + (uu - bd.u0), b = gi & 1;
            if (bd.first && gi >= 2) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[b], ((gi >> 1) - 1) & 1, status));
                if (!ok)
                    break;
            }
            const uint32_t dt = taddr + (uint32_t)(b * BN);
#pragma unroll
            for (int j = 0; j < ME_SMAX; j += ME_SPS) {
                if (j < nsl && ok) {
                    const int gs = g++, st = gs % ME_STAGES;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full_b[st], (gs / ME_STAGES) & 1, status));
                    if (ok) {
#pragma unroll
                        for (int h = 0; h < ME_SPS; ++h) {
                            const int jj = j + h;
                            if (jj >= nsl)
                                break;
                            unsigned char *bs = sb + (st * ME_SPS + h) * ME_B_BYTES;
                            const int kr = krs[jj];
                            if (kr < 16) {
                                const int nz = (16 - kr) * (BN / 64) * 8;  // 16-byte pieces of rank rows kr..15
                                for (int e = lane; e < nz; e += 32) {
                                    const int piece = e & 7, rest = e >> 3;
                                    const int at = rest % (BN / 64), rr = kr + rest / (BN / 64);
                                    *reinterpret_cast<uint4 *>(bs + at * 2048 + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                                               piece * 16) = make_uint4(0u, 0u, 0u, 0u);
                                }
                                fence_proxy_async_smem();
                            }
                            __syncwarp();
                            if (lane == 0) {
                                tc_fence_after();
                                const uint64_t bdesc = umma_desc_sw128_mn(smem_u32(bs), 2048, 1024);
                                const uint32_t zo = (uint32_t)((jj >> 2) * (MMA_TM * 128) + (jj & 3) * 32);
                                umma_bf16(dt, umma_desc_sw128(zhi + zo), bdesc, idesc, !(bd.first && jj == 0));
                                umma_bf16(dt, umma_desc_sw128(zlo + zo), bdesc, idesc, true);
                            }
                            __syncwarp();
                        }
                        if (lane == 0) {
                            umma_commit(&empty_b[st]);  // the stage is free once its MMAs complete
                            if (bd.last && j + ME_SPS >= nsl)
                                umma_commit(&acc_full[b]);
                        }
                        __syncwarp();
                    }
                }
            }
        }
        if (lane == 0)
            umma_commit(zfree);  // the operand may be rebuilt once these MMAs complete
        __syncwarp();
        if (!ok)
            return;
    }
}

template <int BN>
__global__ void __launch_bounds__(ME_THREADS, 1)
    k_mma_expand(const __grid_constant__ CUtensorMap map_b, const MmaExpandArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const MeLayout L(a.pool.capacity);
    __shared__ uint64_t full_b[ME_STAGES], empty_b[ME_STAGES], zready, zfree, acc_full[2], acc_empty[2];
    __shared__ uint64_t job_full[ME_JOBS], job_empty[ME_JOBS], lready, lack;
    __shared__ MeJob s_jobs[ME_JOBS];
    __shared__ uint32_t s_taddr;
    __shared__ int s_scan[ME_WORKERS / 32 + 1];
    __shared__ MeBuild s_build[2];  // build n in slot n % 2: the next one may be announced early

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *status = a.m.hdr + HDR_STATUS;
    if (a.m.hdr[HDR_PVALID] == 0)
        return;  // nothing valid in this batch (uniform)
    const int G = gridDim.x;
    const int u_begin = (int)((long long)blockIdx.x * a.units / G);
    const int u_end = (int)((long long)(blockIdx.x + 1) * a.units / G);
    if (tid == 0) {
        for (int s = 0; s < ME_STAGES; ++s) {
            mbar_init(&full_b[s], 1);
            mbar_init(&empty_b[s], 1);
        }
        mbar_init(&zready, ME_WORKERS);
        mbar_init(&lready, 1);
        mbar_init(&lack, 1);
        mbar_init(&zfree, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], ME_EPI);
        }
        for (int j = 0; j < ME_JOBS; ++j) {
            mbar_init(&job_full[j], 1);
            mbar_init(&job_empty[j], ME_EPI / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == ME_WORKERS / 32) {
        // z is written by the shrink: wait for it; tensor memory only after that
        // (the shrink's CTAs hold tensor memory until they finish)
        pdl_wait();
        tmem_alloc(&s_taddr, 2 * BN);
        tc_fence_before();
        __syncthreads();  // (A) accumulator address visible
        tc_fence_after();
        const uint32_t taddr = s_taddr;
        me_mma_warp<BN>(smem, L, full_b, empty_b, &zready, &zfree, acc_full, acc_empty, s_build, taddr, status);
        __syncwarp();
        __syncthreads();  // (B) every epilogue has read its accumulator
        tc_fence_after();
        tmem_dealloc(taddr, 2 * BN);
        return;
    }
    if (warp == ME_WORKERS / 32 + 1) {
        __syncthreads();  // (A)
        me_producer_warp<BN>(map_b, a, smem, L, full_b, empty_b, &lready, &lack, s_build, status);
        __syncwarp();
        __syncthreads();  // (B)
        return;
    }
    if (warp >= ME_WORKERS / 32 + 2) {
        // epilogue warps: each unit's y + D, rounded once, in the order the
        // workers queue them; warp w reads accumulator lanes 32 (w % 4).. (its
        // TMEM lane quarter), every column of the unit in two halves
        __syncthreads();  // (A)
        tc_fence_after();
        const uint32_t taddr = s_taddr;
        const int lq = warp & 3, row = lq * 32 + lane;
        const int d_out = a.pool.d_out;
        constexpr int HALF = BN / 2, NV = HALF / 8;
        for (int j = 0;; ++j) {
            const int slot = j % ME_JOBS;
            if (!mbar_wait_bounded(&job_full[slot], (j / ME_JOBS) & 1, status))
                break;
            const MeJob jb = s_jobs[slot];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&job_empty[slot]);  // copied: the slot may be refilled
            if (jb.done)
                break;
            const int b = jb.gi & 1;
            const bool live = row < jb.nrows;
            __nv_bfloat16 *yr = a.y + (size_t)(jb.t0 + (live ? row : 0)) * d_out + (jb.uu % a.n_nt) * BN;
            bool ok = true;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                uint4 yv[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    yv[v] = live ? *reinterpret_cast<const uint4 *>(yr + hf * HALF + 8 * v)
                                 : make_uint4(0u, 0u, 0u, 0u);
                if (hf == 0) {
                    ok = mbar_wait_bounded(&acc_full[b], (jb.gi >> 1) & 1, status);
                    tc_fence_after();
                }
#pragma unroll
                for (int c = 0; c < HALF; c += 16) {
                    float v[16];
                    tmem_ld16(taddr + ((uint32_t)(lq * 32) << 16) + (uint32_t)(b * BN + hf * HALF + c), v);
                    if (live && ok) {
                        uint4 o[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint4 w = yv[c / 8 + hh];
                            const float *d = v + 8 * hh;
                            o[hh] = make_uint4(pack_bf16x2(bf16lo(w.x) + d[0], bf16hi(w.x) + d[1]),
                                               pack_bf16x2(bf16lo(w.y) + d[2], bf16hi(w.y) + d[3]),
                                               pack_bf16x2(bf16lo(w.z) + d[4], bf16hi(w.z) + d[5]),
                                               pack_bf16x2(bf16lo(w.w) + d[6], bf16hi(w.w) + d[7]));
                        }
                        *reinterpret_cast<uint4 *>(yr + hf * HALF + c) = o[0];
                        *reinterpret_cast<uint4 *>(yr + hf * HALF + c + 8) = o[1];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
            if (!ok)
                break;
        }
        __syncwarp();
        __syncthreads();  // (B)
        return;
    }

    // ------------------------------------------------------------ workers
    unsigned char *zhi = smem + L.zhi, *zlo = smem + L.zlo;
    int2 *cache = reinterpret_cast<int2 *>(smem + L.cache);
    int *list = reinterpret_cast<int *>(smem + L.list);
    int *lrank = reinterpret_cast<int *>(smem + L.lrank);
    int *sbase = reinterpret_cast<int *>(smem + L.sbase);
    int *toff = reinterpret_cast<int *>(smem + L.toff);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + L.bitmap);
    int *wpre = reinterpret_cast<int *>(smem + L.wpre);
    const int nwords = (a.pool.capacity + 31) / 32;

    bool synced = false;
    int nb = 0, freed = 0, gi = 0;
    auto wait_free = [&]() {  // every build handed over so far has been consumed
        while (freed < nb) {
            mbar_wait_bounded(&zfree, freed & 1, status);
            ++freed;
        }
    };
    // a build in two steps: announce (its slots, for the B producer) once the
    // lists are in place and the build before the previous one is consumed,
    // then ready (the operand, for the MMA warp) once it is built
    auto announce = [&](int u0, int u1, int s0, int s1, int nu, int first, int last, int done) {
        if (tid == 0) {
            // at most one announcement outstanding: the producer has read the
            // previous one (so a barrier phase is never passed unseen, and the
            // slot reused here was read two builds ago)
            if (nb > 0)
                mbar_wait_bounded(&lack, (nb - 1) & 1, status);
            s_build[nb & 1] = MeBuild{u0, u1, s0, s1, nu, first, last, gi, done};
            mbar_arrive(&lready);
        }
    };
    auto ready = [&]() {
        fence_proxy_async_smem();
        mbar_arrive(&zready);
        ++nb;
    };
    int t0 = 0, nrows = 0, p0 = 0, np = 0, nu_total = 0;

    // lists of window w0: adapters of ordinals [w0, w0 + ME_NU_MAX), ranks, first slots; returns the slot count
    auto build_lists = [&](int w0) -> int {
        for (int wi = tid; wi < nwords; wi += ME_WORKERS) {
            uint32_t word = bitmap[wi];
            int ord = wpre[wi];
            while (word) {
                const int bit = __ffs(word) - 1;
                word &= word - 1u;
                if (ord >= w0 && ord < w0 + ME_NU_MAX)
                    list[ord - w0] = wi * 32 + bit;
                ++ord;
            }
        }
        me_bar();
        const int nu = min(ME_NU_MAX, nu_total - w0);
        int scarry = 0;
        for (int ub = 0; ub < nu; ub += ME_WORKERS) {
            const int u = ub + tid;
            int nch = 0;
            if (u < nu) {
                const int k = effective_rank(a.pool, a.ranks, list[u]);
                lrank[u] = k;
                nch = (k + 15) >> 4;
            }
            int tot;
            const int ex = me_scan(nch, tot, s_scan);
            if (u < nu)
                sbase[u] = scarry + ex;
            scarry += tot;
        }
        if (tid == 0)
            sbase[nu] = scarry;
        me_bar();
        return scarry;
    };

    // A operand for window slots [s0, s1): per token row and slot, the summed z as bf16 hi + lo
    auto build_zsel = [&](int w0, int nu, int s0, int s1) {
        const int nkb = (s1 - s0 + 3) >> 2;  // 64-column blocks in use
        uint4 *zh4 = reinterpret_cast<uint4 *>(zhi), *zl4 = reinterpret_cast<uint4 *>(zlo);
        for (int i = tid; i < nkb * (MMA_TM * 128 / 16); i += ME_WORKERS) {
            zh4[i] = make_uint4(0u, 0u, 0u, 0u);
            zl4[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        me_bar();
        auto pair_at = [&](int i) -> int2 {
            if (i < ME_PT_MAX)
                return cache[i];
            const int q = a.m.pos[p0 + i];
            return make_int2(q, q >= 0 ? a.m.adapter[q] : -1);
        };
        for (int i = tid; i < np; i += ME_WORKERS) {
            const int2 qa = pair_at(i);
            const int ad = qa.y;
            if (ad < 0 || !((bitmap[ad >> 5] >> (ad & 31)) & 1u))
                continue;
            const int u = wpre[ad >> 5] + __popc(bitmap[ad >> 5] & ((1u << (ad & 31)) - 1u)) - w0;
            if (u < 0 || u >= nu)
                continue;
            const int row = me_pair_row(toff, nrows, p0, i);
            const int i_lo = toff[row] - p0, i_hi = toff[row + 1] - p0;
            bool dup = false;  // an earlier pair of the token with the same adapter sums this one
            for (int j = i_lo; j < i && !dup; ++j)
                dup = pair_at(j).y == ad;
            if (dup)
                continue;
            const int k = lrank[u], sb0 = sbase[u];
            for (int c = 0; c < (k + 15) >> 4; ++c) {
                const int s = sb0 + c;
                if (s < s0 || s >= s1)
                    continue;
                const int jj = s - s0, kk = min(16, k - 16 * c);
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    acc[e] = 0.f;
                for (int j = i; j < i_hi; ++j) {
                    const int2 qb = j == i ? qa : pair_at(j);
                    if (qb.y != ad)
                        continue;
                    const float *zr = a.m.z + (size_t)qb.x * a.zs + 16 * c;
#pragma unroll
                    for (int j4 = 0; j4 < 16; j4 += 4) {
                        if (j4 < kk) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(zr + j4));
                            acc[j4] += v.x;
                            acc[j4 + 1] += j4 + 1 < kk ? v.y : 0.f;
                            acc[j4 + 2] += j4 + 2 < kk ? v.z : 0.f;
                            acc[j4 + 3] += j4 + 3 < kk ? v.w : 0.f;
                        }
                    }
                }
                uint32_t h[8], l[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const __nv_bfloat162 hv = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                    h[e] = *reinterpret_cast<const uint32_t *>(&hv);
                    l[e] = pack_bf16x2(acc[2 * e] - __low2float(hv), acc[2 * e + 1] - __high2float(hv));
                }
                const uint32_t o0 = sw128_offset(row, 16 * jj, MMA_TM), o1 = sw128_offset(row, 16 * jj + 8, MMA_TM);
                *reinterpret_cast<uint4 *>(zhi + o0) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(zhi + o1) = make_uint4(h[4], h[5], h[6], h[7]);
                *reinterpret_cast<uint4 *>(zlo + o0) = make_uint4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<uint4 *>(zlo + o1) = make_uint4(l[4], l[5], l[6], l[7]);
            }
        }
    };

    // queues unit uu (running index gi) for the epilogue warps
    int njob = 0;
    auto push_job = [&](int uu, int done) {
        const int slot = njob % ME_JOBS;
        if (tid == 0) {
            if (njob >= ME_JOBS)
                mbar_wait_bounded(&job_empty[slot], ((njob / ME_JOBS) - 1) & 1, status);
            s_jobs[slot] = MeJob{uu, t0, nrows, gi, done};
            mbar_arrive(&job_full[slot]);  // release: the job is visible to the waiting warps
        }
        ++njob;
        if (!done)
            ++gi;
    };

    for (int u = u_begin; u < u_end;) {
        const int tile = u / a.n_nt;
        const int ut_end = min(u_end, (tile + 1) * a.n_nt);
        t0 = tile * MMA_TM;
        nrows = min(MMA_TM, a.T - t0);
        wait_free();  // the lists and the operand are rewritten below
        // ---- the tile's pairs (mapping data: complete before the shrink started)
        for (int i = tid; i <= nrows; i += ME_WORKERS)
            toff[i] = a.m.toff[t0 + i];
        for (int i = tid; i < nwords; i += ME_WORKERS)
            bitmap[i] = 0u;
        me_bar();
        p0 = toff[0];
        np = toff[nrows] - p0;
        for (int i = tid; i < np; i += ME_WORKERS) {
            const int q = a.m.pos[p0 + i];
            int ad = q >= 0 ? a.m.adapter[q] : -1;
            if (ad >= 0 && effective_rank(a.pool, a.ranks, ad) <= 0)
                ad = -1;  // contributes nothing
            if (ad >= 0)
                atomicOr(&bitmap[ad >> 5], 1u << (ad & 31));
            if (i < ME_PT_MAX)
                cache[i] = make_int2(q, ad);
        }
        me_bar();
        nu_total = 0;
        for (int base = 0; base < nwords; base += ME_WORKERS) {
            const int wi = base + tid;
            const int c = wi < nwords ? __popc(bitmap[wi]) : 0;
            int tot;
            const int ex = me_scan(c, tot, s_scan);
            if (wi < nwords)
                wpre[wi] = nu_total + ex;
            nu_total += tot;
        }
        me_bar();
        if (!synced) {
            pdl_wait();  // z of the shrink is complete from here on
            __syncthreads();  // (A)
            tc_fence_after();
            synced = true;
        }
        if (nu_total > 0) {
            const int nwin = (nu_total + ME_NU_MAX - 1) / ME_NU_MAX;
            if (nwin == 1) {
                const int ns = build_lists(0);
                const int nu = nu_total;
                const int npass = (ns + ME_SMAX - 1) / ME_SMAX;
                if (npass == 1) {
                    announce(u, ut_end, 0, ns, nu, 1, 1, 0);
                    build_zsel(0, nu, 0, ns);  // one operand for every column tile of the token tile
                    ready();
                    for (int uu = u; uu < ut_end; ++uu)
                        push_job(uu, 0);
                } else {
                    // several passes: two units at a time (one per accumulator) share each pass
                    for (int uu = u; uu < ut_end; uu += 2) {
                        const int u2 = min(uu + 2, ut_end);
                        for (int p = 0; p < npass; ++p) {
                            const int s0 = p * ME_SMAX, s1 = min(ns, s0 + ME_SMAX);
                            // the pass's B chunks stream while the previous
                            // pass's MMAs finish and this operand is built
                            announce(uu, u2, s0, s1, nu, p == 0, p == npass - 1, 0);
                            wait_free();
                            build_zsel(0, nu, s0, s1);
                            ready();
                        }
                        for (int v = uu; v < u2; ++v)
                            push_job(v, 0);
                    }
                }
            } else {
                for (int uu = u; uu < ut_end; uu += 2) {
                    const int u2 = min(uu + 2, ut_end);
                    for (int w = 0; w < nwin; ++w) {
                        const int w0 = w * ME_NU_MAX;
                        wait_free();
                        const int ns = build_lists(w0);
                        const int nu = min(ME_NU_MAX, nu_total - w0);
                        const int npass = (ns + ME_SMAX - 1) / ME_SMAX;
                        for (int p = 0; p < npass; ++p) {
                            const int s0 = p * ME_SMAX, s1 = min(ns, s0 + ME_SMAX);
                            wait_free();
                            announce(uu, u2, s0, s1, nu, w == 0 && p == 0, w == nwin - 1 && p == npass - 1, 0);
                            build_zsel(w0, nu, s0, s1);
                            ready();
                        }
                    }
                    for (int v = uu; v < u2; ++v)
                        push_job(v, 0);
                }
            }
        }
        u = ut_end;
    }
    if (!synced) {
        pdl_wait();
        __syncthreads();  // (A)
        synced = true;
    }
    wait_free();
    announce(0, 0, 0, 0, 0, 0, 0, 1);
    ready();
    push_job(0, 1);
    tc_fence_before();
    __syncthreads();  // (B)
}

}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    // looked up once per process (a function-local static is initialised
    // exactly once, whatever the number of threads calling)
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// Row-major bf16 matrix [rows][cols], boxes of 16 rows x 64 columns, 128-byte swizzle.
cudaError_t encode_rows(unsigned char *out, const void *base, int cols, long long rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// B as a 3-D tensor {64 columns, rows, d_out / 64 column blocks} (strides: the
// row pitch, then 128 bytes), boxes {64, 16, bn / 64}: one box is a 16-row
// chunk of bn columns, landing column block after column block (2 KB each).
cudaError_t encode_b_blocks(unsigned char *out, const void *base, int d_out, long long rows, int bn)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(d_out / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)d_out * 2, 128};
    const cuuint32_t box[3] = {64, 16, (cuuint32_t)(bn / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Output columns per expand unit.
int expand_bn(int d_out) { return d_out % 256 == 0 ? 256 : (d_out % 128 == 0 ? 128 : 64); }

// Cluster size of the shrink: the K blocks of d_in split over ck CTAs.
int shrink_cluster(int d_in)
{
    const int nkb = d_in / 64;
    int ck = 4;
    while (ck > 1 && ck > nkb)
        ck >>= 1;
    return ck;
}

template <int BN>
cudaError_t launch_expand_bn(__nv_bfloat16 *y, const PoolDev &pool, const CUtensorMap &map_b, const int32_t *ranks,
                             const MapDev &m, int T, cudaStream_t st)
{
    const MeLayout L(pool.capacity);
    static thread_local int attr_dev = -1;  // per host thread
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_mma_expand<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             MeLayout(LORA_MAX_CAPACITY).total);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_mma_expand<BN>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    const int n_nt = pool.d_out / BN;
    const int units = n_nt * ((T + MMA_TM - 1) / MMA_TM);
    MmaExpandArgs a{y, pool, ranks, m, T, z_stride(pool.r_max), n_nt, units};
    const int grid = units < sm_count() ? units : sm_count();  // persistent: one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(ME_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mma_expand<BN>, map_b, a);
}

}  // namespace

bool mma_supported(int d_in, int d_out, int r_max)
{
    return d_in % 64 == 0 && d_out % 64 == 0 && r_max >= 1 && r_max <= LORA_MAX_RANK;
}

cudaError_t mma_encode_maps(const PoolDev &pool, MmaMaps &maps)
{
    maps.ready = false;
    const long long rows = (long long)pool.capacity * pool.r_max;
    cudaError_t e = encode_rows(maps.At, pool.At, pool.d_in, rows);
    if (e == cudaSuccess)
        e = encode_b_blocks(maps.B, pool.B, pool.d_out, rows, expand_bn(pool.d_out));
    maps.ready = e == cudaSuccess;
    return e;
}

cudaError_t launch_mma(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const MmaMaps &maps,
                       const int32_t *ranks, const MapDev &m, int T, int P, cudaStream_t st)
{
    if (!maps.ready || !mma_supported(pool.d_in, pool.d_out, pool.r_max))
        return cudaErrorNotSupported;
    CUtensorMap map_at, map_b;
    memcpy(&map_at, maps.At, sizeof(map_at));
    memcpy(&map_b, maps.B, sizeof(map_b));

    // 1. segment shrink: one cluster of ck CTAs per tile slot (empty slots exit)
    const int ck = shrink_cluster(pool.d_in);
    const int tiles = mma_tile_bound(P, pool.capacity);
    if (tiles > 0) {
        static thread_local int attr_dev = -1;  // per host thread
        int dev = 0;
        cudaGetDevice(&dev);
        if (attr_dev != dev) {
            cudaError_t e = cudaFuncSetAttribute(k_mma_shrink, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   MS_SMEM_MAX);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(k_mma_shrink, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess)
                return e;
            attr_dev = dev;
        }
        const int sb = ms_stage_bytes(pool.r_max);
        MmaShrinkArgs sa{x, pool, ranks, m, z_stride(pool.r_max), ck, sb};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tiles * ck, 1, 1);
        cfg.blockDim = dim3(MS_THREADS, 1, 1);
        cfg.dynamicSmemBytes = 1024 + MS_STAGES * sb;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ck;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, k_mma_shrink, map_at, sa);
        if (e != cudaSuccess)
            return e;
    }

    // 2. token-tile expand, PDL-chained to the shrink
    if (T <= 0)
        return cudaSuccess;
    switch (expand_bn(pool.d_out)) {
    case 256:
        return launch_expand_bn<256>(y, pool, map_b, ranks, m, T, st);
    case 128:
        return launch_expand_bn<128>(y, pool, map_b, ranks, m, T, st);
    default:
        return launch_expand_bn<64>(y, pool, map_b, ranks, m, T, st);
    }
}

}  // namespace tcl
