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
// 2. Token-tile expand (RowExpand as a dense product): a CTA owns MMA_TM
//    consecutive tokens x BN output columns.  Its pairs' adapters, in
//    ascending id order, each give ceil(k / 16) "slots" of 16 rank rows; the
//    A operand holds, per token and slot, the sum of the token's z rows for
//    that adapter (zero elsewhere), split into a bf16 high part and a bf16
//    residual (hi + lo carries ~16 significant bits of the fp32 z), and the
//    B operand is B_a[16c .. 16c + 15, columns] loaded by TMA in the
//    MN-major 128-byte swizzled layout (B is stored row-major, d_out
//    contiguous).  D (128 x BN fp32) accumulates in tensor memory over all
//    slots; the epilogue adds y and rounds once to bf16.  Rank rows at or
//    beyond k of a partial chunk are zeroed in shared memory before use, so
//    padding never reaches the sum.
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
constexpr int MS_LAG = 2;                                // cp.async groups kept in flight per gather thread
constexpr int MS_X_BYTES = MMA_TM * 128;                 // 128 rows x 64 bf16
constexpr int MS_A_BYTES = LORA_MAX_RANK * 128;          // up to 64 rows x 64 bf16
constexpr int MS_STAGE_BYTES = MS_X_BYTES + MS_A_BYTES;  // 24 KB
constexpr int MS_SMEM = 1024 + MS_STAGES * MS_STAGE_BYTES;
constexpr int MS_PART_STRIDE = LORA_MAX_RANK + 4;        // fp32 partial row stride (floats)
static_assert(MMA_TM * MS_PART_STRIDE * 4 <= MS_STAGES * MS_STAGE_BYTES, "partial fits the stages");

struct MmaShrinkArgs {
    const __nv_bfloat16 *x;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int zs;  // z row stride (floats)
    int ck;  // CTAs per cluster (K split)
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
        // ---- x rows of the tile's pairs, gathered into the swizzled K-major layout
        const int row = tid;
        const bool valid = row < n;
        const __nv_bfloat16 *xr = a.x + (valid ? (size_t)a.m.tok[q0 + row] * d_in : 0);
        for (int it = 0; it < nk; ++it) {
            const int s = it % MS_STAGES;
            if (it >= MS_STAGES && !mbar_wait_bounded(&empty[s], ((it / MS_STAGES) - 1) & 1, status))
                break;
            unsigned char *sx = smem + s * MS_STAGE_BYTES;
            if (valid) {
                const __nv_bfloat16 *src = xr + (size_t)(kb0 + it) * 64;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    cp_async16(sx + xrow_offset(row, ch), src + ch * 8);
            }
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
                unsigned char *sa = smem + s * MS_STAGE_BYTES + MS_X_BYTES;
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
                const uint32_t xs = smem_u32(smem + s * MS_STAGE_BYTES);
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

constexpr int ME_THREADS = 256;
constexpr int ME_SP = 8;                            // slots (16 rank rows each) per pass
constexpr int ME_Z_BYTES = MMA_TM * ME_SP * 16 * 2;  // one of hi / lo: 128 rows x 128 bf16
constexpr int ME_STAGES = 4;
constexpr int ME_B_BYTES = 16 * 256 * 2;            // 16 rank rows x up to 256 columns
constexpr int ME_PT_MAX = 512;                      // pairs of a tile cached in shared memory
constexpr int ME_NU_MAX = 512;                      // adapters listed per window

struct MmaExpandArgs {
    __nv_bfloat16 *y;
    PoolDev pool;
    const int32_t *ranks;
    MapDev m;
    int T, zs;
};

// Dynamic shared memory of the expand kernel (offsets from a 1024-aligned base).
struct MeLayout {
    int zhi, zlo, b, cache, list, lrank, sbase, toff, bitmap, total;
    __host__ __device__ explicit MeLayout(int capacity)
    {
        zhi = 0;
        zlo = zhi + ME_Z_BYTES;
        b = zlo + ME_Z_BYTES;
        cache = b + ME_STAGES * ME_B_BYTES;      // int2 [ME_PT_MAX]: sorted position, adapter
        list = cache + ME_PT_MAX * 8;            // int [ME_NU_MAX]: adapters of the window
        lrank = list + ME_NU_MAX * 4;            // int [ME_NU_MAX]: their ranks
        sbase = lrank + ME_NU_MAX * 4;           // int [ME_NU_MAX + 1]: first slot of each
        toff = sbase + (ME_NU_MAX + 4) * 4;      // int [MMA_TM + 1]: pair offsets of the tile's tokens
        bitmap = toff + (MMA_TM + 4) * 4;        // uint32 [ceil(capacity / 32)]
        total = bitmap + ((capacity + 31) / 32) * 4 + 1024;
    }
};

// Block-wide exclusive scan of one int over ME_THREADS threads.
__device__ __forceinline__ int me_scan(int v, int &total, int *sh /* [ME_THREADS / 32 + 1] */)
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
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < ME_THREADS / 32; ++w) {
            const int t = sh[w];
            sh[w] = run;
            run += t;
        }
        sh[ME_THREADS / 32] = run;
    }
    __syncthreads();
    const int r = sh[warp] + inc - v;
    total = sh[ME_THREADS / 32];
    __syncthreads();
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int BN>
__global__ void __launch_bounds__(ME_THREADS, 2)
    k_mma_expand(const __grid_constant__ CUtensorMap map_b, const MmaExpandArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const MeLayout L(a.pool.capacity);
    unsigned char *zhi = smem + L.zhi, *zlo = smem + L.zlo, *sb = smem + L.b;
    int2 *cache = reinterpret_cast<int2 *>(smem + L.cache);
    int *list = reinterpret_cast<int *>(smem + L.list);
    int *lrank = reinterpret_cast<int *>(smem + L.lrank);
    int *sbase = reinterpret_cast<int *>(smem + L.sbase);
    int *toff = reinterpret_cast<int *>(smem + L.toff);
    uint32_t *bitmap = reinterpret_cast<uint32_t *>(smem + L.bitmap);
    __shared__ uint64_t full_b[ME_STAGES], empty_b[ME_STAGES], pass_done;
    __shared__ uint32_t s_taddr;
    __shared__ int s_scan[ME_THREADS / 32 + 1];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, t0 = blockIdx.y * MMA_TM;
    const int nrows = min(MMA_TM, a.T - t0);
    const int d_out = a.pool.d_out, r_max = a.pool.r_max;
    const int nwords = (a.pool.capacity + 31) / 32;
    int32_t *status = a.m.hdr + HDR_STATUS;
    if (a.m.hdr[HDR_PVALID] == 0)
        return;  // nothing valid in this batch (uniform)

    // ---- the tile's pairs (mapping data: complete before the shrink started)
    for (int i = tid; i <= nrows; i += ME_THREADS)
        toff[i] = a.m.toff[t0 + i];
    for (int i = tid; i < nwords; i += ME_THREADS)
        bitmap[i] = 0u;
    if (tid == 0) {
        for (int s = 0; s < ME_STAGES; ++s) {
            mbar_init(&full_b[s], 1);
            mbar_init(&empty_b[s], 1);
        }
        mbar_init(&pass_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int p0 = toff[0], np = toff[nrows] - p0;
    for (int i = tid; i < np; i += ME_THREADS) {
        const int q = a.m.pos[p0 + i];
        int ad = q >= 0 ? a.m.adapter[q] : -1;
        if (ad >= 0 && effective_rank(a.pool, a.ranks, ad) <= 0)
            ad = -1;  // contributes nothing
        if (ad >= 0)
            atomicOr(&bitmap[ad >> 5], 1u << (ad & 31));
        if (i < ME_PT_MAX)
            cache[i] = make_int2(q, ad);
    }
    __syncthreads();
    int nu_total;
    {
        int c = 0;
        for (int i = tid; i < nwords; i += ME_THREADS)
            c += __popc(bitmap[i]);
        me_scan(c, nu_total, s_scan);
    }
    if (nu_total == 0)
        return;  // uniform: y stays as it is

    const uint32_t idesc = umma_idesc_bf16(MMA_TM, BN) | (1u << 16);  // B operand MN-major
    uint32_t taddr = 0;
    int gs_base = 0, gp = 0;
    bool first_mma = true, ok = true;
    for (int w0 = 0; w0 < nu_total; w0 += ME_NU_MAX) {
        // ---- the window's adapters (ascending id), their ranks and first slots
        int carry = 0;
        for (int base = 0; base < nwords; base += ME_THREADS) {
            const int wi = base + tid;
            uint32_t word = wi < nwords ? bitmap[wi] : 0u;
            int tot;
            int ord = carry + me_scan(__popc(word), tot, s_scan);
            while (word) {
                const int b = __ffs(word) - 1;
                word &= word - 1u;
                if (ord >= w0 && ord < w0 + ME_NU_MAX)
                    list[ord - w0] = wi * 32 + b;
                ++ord;
            }
            carry += tot;
        }
        const int nu = min(ME_NU_MAX, nu_total - w0);
        __syncthreads();
        int scarry = 0;
        for (int ub = 0; ub < nu; ub += ME_THREADS) {
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
        __syncthreads();
        const int ns = scarry;

        // ---- B chunks by TMA (warp 0, lane 0): slot j -> stage (gs_base + j) % ME_STAGES
        int issued = 0;
        auto issue_b = [&](int j) -> bool {
            const int gs = gs_base + j, st = gs % ME_STAGES;
            if (gs >= ME_STAGES && !mbar_wait_bounded(&empty_b[st], ((gs / ME_STAGES) - 1) & 1, status))
                return false;
            const int u = me_slot_owner(sbase, nu, j);
            const int row = list[u] * r_max + 16 * (j - sbase[u]);
            mbar_arrive_expect_tx(&full_b[st], 16 * BN * 2);
#pragma unroll
            for (int at = 0; at < BN / 64; ++at)
                tma_load_2d(sb + st * ME_B_BYTES + at * 2048, &map_b, n0 + 64 * at, row, &full_b[st]);
            return true;
        };
        if (warp == 0 && lane == 0)
            while (ok && issued < ns && issued < ME_STAGES)
                ok = issue_b(issued++);
        __syncwarp();

        if (w0 == 0) {
            // z comes from the shrink: wait for it; tensor memory only after that
            // (the shrink's CTAs hold tensor memory until they finish)
            pdl_wait();
            if (warp == 0)
                tmem_alloc(&s_taddr, BN);
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            taddr = s_taddr;
        }

        for (int j0 = 0; j0 < ns; j0 += ME_SP, ++gp) {
            const int npass = min(ME_SP, ns - j0);
            if (gp > 0 && !mbar_wait_bounded(&pass_done, (gp - 1) & 1, status))
                ok = false;
            // ---- A operand: per token row and slot, the summed z, as bf16 hi + lo
            for (int idx = tid; idx < MMA_TM * npass; idx += ME_THREADS) {
                const int row = idx & (MMA_TM - 1), jj = idx / MMA_TM, j = j0 + jj;
                const int u = me_slot_owner(sbase, nu, j);
                const int ad = list[u], c = j - sbase[u];
                const int kk = min(16, lrank[u] - 16 * c);
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    acc[e] = 0.f;
                if (row < nrows) {
                    const int i0 = toff[row] - p0, i1 = toff[row + 1] - p0;
                    for (int i = i0; i < i1; ++i) {
                        int2 qa;
                        if (i < ME_PT_MAX) {
                            qa = cache[i];
                        } else {
                            const int q = a.m.pos[p0 + i];
                            qa = make_int2(q, q >= 0 ? a.m.adapter[q] : -1);
                        }
                        if (qa.y != ad)
                            continue;
                        const float *zr = a.m.z + (size_t)qa.x * a.zs + 16 * c;
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
            fence_proxy_async_smem();
            __syncthreads();

            // ---- warp 0: per slot, wait for its B chunk, mask rank rows >= k, issue hi and lo MMAs
            if (warp == 0) {
                for (int jj = 0; jj < npass && ok; ++jj) {
                    const int j = j0 + jj, gs = gs_base + j, st = gs % ME_STAGES;
                    ok = mbar_wait_bounded(&full_b[st], (gs / ME_STAGES) & 1, status);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (!ok)
                        break;
                    const int u = me_slot_owner(sbase, nu, j);
                    const int kr = lrank[u] - 16 * (j - sbase[u]);
                    unsigned char *bs = sb + st * ME_B_BYTES;
                    if (kr < 16) {
                        const int nz = (16 - kr) * (BN / 64) * 8;  // 16-byte pieces of rows kr..15
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
                        const uint64_t bd = umma_desc_sw128_mn(smem_u32(bs), 2048, 1024);
                        const uint32_t zo = (uint32_t)((jj >> 2) * (MMA_TM * 128) + (jj & 3) * 32);
                        umma_bf16(taddr, umma_desc_sw128(smem_u32(zhi) + zo), bd, idesc, !first_mma);
                        umma_bf16(taddr, umma_desc_sw128(smem_u32(zlo) + zo), bd, idesc, true);
                        first_mma = false;
                        umma_commit(&empty_b[st]);
                        while (ok && issued < ns && issued <= j + ME_STAGES - 1)
                            ok = issue_b(issued++);
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
                if (lane == 0)
                    umma_commit(&pass_done);
                __syncwarp();
            }
        }
        gs_base += ns;
    }

    // ---- epilogue: y (prefetched) + D, rounded once; warp w: lanes 32 (w % 4).., column half w / 4
    constexpr int HALF = BN / 2, NV = HALF / 8;
    const int lq = warp & 3, hf = warp >> 2;
    const int row = lq * 32 + lane;
    const bool live = row < nrows;
    __nv_bfloat16 *yr = a.y + (size_t)(t0 + (live ? row : 0)) * d_out + n0 + hf * HALF;
    uint4 yv[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v)
        yv[v] = live ? *reinterpret_cast<const uint4 *>(yr + 8 * v) : make_uint4(0u, 0u, 0u, 0u);
    ok = mbar_wait_bounded(&pass_done, (gp - 1) & 1, status) && ok;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < HALF; c += 16) {
        float v[16];
        tmem_ld16(taddr + ((uint32_t)(lq * 32) << 16) + hf * HALF + c, v);
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
            *reinterpret_cast<uint4 *>(yr + c) = o[0];
            *reinterpret_cast<uint4 *>(yr + c + 8) = o[1];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(taddr, BN);
}

}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
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
    static int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_mma_expand<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             MeLayout(LORA_MAX_CAPACITY).total);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    MmaExpandArgs a{y, pool, ranks, m, T, z_stride(pool.r_max)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pool.d_out / BN, (T + MMA_TM - 1) / MMA_TM, 1);
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
        e = encode_rows(maps.B, pool.B, pool.d_out, rows);
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
        static int attr_dev = -1;
        int dev = 0;
        cudaGetDevice(&dev);
        if (attr_dev != dev) {
            cudaError_t e = cudaFuncSetAttribute(k_mma_shrink, cudaFuncAttributeMaxDynamicSharedMemorySize, MS_SMEM);
            if (e != cudaSuccess)
                return e;
            attr_dev = dev;
        }
        MmaShrinkArgs sa{x, pool, ranks, m, z_stride(pool.r_max), ck};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(tiles * ck, 1, 1);
        cfg.blockDim = dim3(MS_THREADS, 1, 1);
        cfg.dynamicSmemBytes = MS_SMEM;
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
    if (pool.d_out % 256 == 0)
        return launch_expand_bn<256>(y, pool, map_b, ranks, m, T, st);
    if (pool.d_out % 128 == 0)
        return launch_expand_bn<128>(y, pool, map_b, ranks, m, T, st);
    return launch_expand_bn<64>(y, pool, map_b, ranks, m, T, st);
}

}  // namespace tcl
