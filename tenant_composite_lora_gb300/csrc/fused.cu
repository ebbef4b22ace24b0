// Fused decode kernel: shrink, alpha scale and RowExpand in one launch.
//
// LoRAForge summary page, "Approach" (4) and "Developer view": short decode
// batches get a dedicated kernel (direct reduction per token group) instead of
// the general shrink/expand pair.  DyMerge-LoRA summary page, "Core idea"
// (paper Sec. 4.3): all token-LoRA pairs of the batch are fused in one kernel.
//
// One cooperative launch of one CTA per SM (all resident).  Every CTA:
//   1. stages the rank table and, if it has an expand role (column tile x
//      segment group), the y rows it will finalise;
//   2. starts its share of the shrink (shrink_core.cuh): units resolved and
//      their A / x copies issued; then, while those land, builds its first
//      expand window and stages the B tiles and per-token pair lists (none of
//      it depends on z); then finishes the shrink, writing z to global memory
//      (it stays in L2);
//   3. meets the others at a grid barrier (bounded wait, LORA_DEV_TIMEOUT on
//      expiry) so that every z is visible;
//   4. stages z and accumulates its tile token-major in registers
//      (expand_core.cuh);
//   5. finalises: with one segment group per column tile it adds y and rounds
//      once; with ng > 1 groups it publishes its fp32 tile, meets a second
//      barrier, and reduces rows [r0, r1) over the ng tiles in a fixed order.
// The barrier counters live in the mapping header; the last CTA to leave
// advances the base for the next launch, and building a mapping resets them.
#include "expand_core.cuh"
#include "shrink_core.cuh"

namespace tcl {

namespace {

struct FusedArgs {
    ShrinkArgs s;
    ExpandArgs e;
    int n_exp;       // CTAs with an expand role = column tiles x ng
    float *partial;  // [n_exp][tb][w] fp32 tiles when ng > 1
};

// All CTAs of the (cooperative, fully resident) grid arrive; returns when the
// counter reaches `target` or after WAIT_LIMIT_NS (then sets LORA_DEV_TIMEOUT
// and returns false).  Uniform across the CTA.
__device__ bool grid_barrier(unsigned *count, unsigned target, int32_t *status)
{
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(count, 1u);
        ok = wait_count_bounded(count, target, status);
        __threadfence();
    }
    return __syncthreads_and(ok) != 0;
}

template <int CPT>
__global__ void __launch_bounds__(EXP_THREADS, 1) k_fused(FusedArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ ShrinkShared sh;
    __shared__ ExpandShared es;
    const ExpandArgs &e = a.e;
    const int W = e.w, VPR = W / 8, TPT = W / CPT;
    const ExpLayout L(e.tb, W, e.use_tab ? e.pool.capacity : 0);
    unsigned char *ring = smem_raw + ((L.total + 127) & ~127);
    int *rank_tab = reinterpret_cast<int *>(smem_raw + L.rank);
    __nv_bfloat16 *yin = reinterpret_cast<__nv_bfloat16 *>(smem_raw + L.yin);
    float *acc = reinterpret_cast<float *>(smem_raw + L.B);  // reuses the B area at the end

    const int tid = threadIdx.x, G = gridDim.x;
    int32_t *status = e.m.hdr + HDR_STATUS;
    unsigned *bar_count = reinterpret_cast<unsigned *>(e.m.hdr + HDR_BAR);
    const unsigned base = *reinterpret_cast<volatile unsigned *>(e.m.hdr + HDR_BAR_BASE);
    const int d_out = e.pool.d_out, ng = e.ng, nt = e.T;
    const bool has_exp = (int)blockIdx.x < a.n_exp;
    const int ct = blockIdx.x / ng, g = blockIdx.x % ng, c0 = ct * W;
    const int r0 = has_exp ? (nt * g) / ng : 0, r1 = has_exp ? (nt * (g + 1)) / ng : 0;

    // 1. z-independent staging
    if (e.use_tab)
        for (int i = tid; i < e.pool.capacity; i += EXP_THREADS)
            rank_tab[i] = effective_rank(e.pool, e.ranks, i);
    for (int i = tid; i < (r1 - r0) * VPR; i += EXP_THREADS) {
        const int t = r0 + i / VPR, v = i % VPR;
        cp_async16(&yin[t * W + v * 8], e.y + (size_t)t * d_out + c0 + v * 8);
    }
    cp_async_commit();
    const int U = has_exp ? e.m.hdr[HDR_U] : 0;
    const int s_begin = (int)(((long long)U * g) / ng), s_end = has_exp ? (int)(((long long)U * (g + 1)) / ng) : 0;
    const int my_t = tid / TPT, my_c = (tid % TPT) * CPT;
    float racc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
        racc[c] = 0.f;
    __syncthreads();

    // 2. the shrink's first copies go out first; the expand's z-independent
    // work (window build, B tiles, pair lists) overlaps them; the shrink is
    // finished and the grid meets in the hook that runs before the first z read
    ShrinkRun<true> run(a.s, sh, ring, rank_tab, blockIdx.x, G);
    run.begin();
    bool ok = true;
    expand_accumulate<CPT>(e, smem_raw, es, c0, 0, nt, true, s_begin, s_end, racc, [&] {
        ok = run.finish();
        ok = grid_barrier(bar_count, base + (unsigned)G, status) && ok;
    });

    // 5. finalise
    unsigned nbar = 1;
    if (has_exp && my_t < nt) {
        if constexpr (CPT == 2) {
            *reinterpret_cast<float2 *>(&acc[my_t * W + my_c]) = make_float2(racc[0], racc[1]);
        } else {
#pragma unroll
            for (int c = 0; c < CPT; c += 4)
                *reinterpret_cast<float4 *>(&acc[my_t * W + my_c + c]) =
                    make_float4(racc[c], racc[c + 1], racc[c + 2], racc[c + 3]);
        }
    }
    __syncthreads();
    if (ng > 1) {
        if (has_exp) {
            float *mine = a.partial + (size_t)blockIdx.x * e.tb * W;
            for (int i = tid * 4; i < nt * W; i += EXP_THREADS * 4)
                __stcg(reinterpret_cast<float4 *>(mine + i), *reinterpret_cast<const float4 *>(&acc[i]));
        }
        grid_barrier(bar_count, base + 2u * (unsigned)G, status);
        nbar = 2;
    }
    if (has_exp) {
        for (int i = tid; i < (r1 - r0) * VPR; i += EXP_THREADS) {
            const int t = r0 + i / VPR, v = i % VPR;
            float s[8];
            if (ng > 1) {
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    s[h] = 0.f;
                for (int gg = 0; gg < ng; ++gg) {
                    const float *src = a.partial + ((size_t)(ct * ng + gg) * e.tb + t) * W + v * 8;
                    const float4 p0 = __ldcg(reinterpret_cast<const float4 *>(src));
                    const float4 p1 = __ldcg(reinterpret_cast<const float4 *>(src + 4));
                    s[0] += p0.x; s[1] += p0.y; s[2] += p0.z; s[3] += p0.w;
                    s[4] += p1.x; s[5] += p1.y; s[6] += p1.z; s[7] += p1.w;
                }
            } else {
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    s[h] = acc[t * W + v * 8 + h];
            }
            const uint4 yi = *reinterpret_cast<const uint4 *>(&yin[t * W + v * 8]);
            const uint32_t w[4] = {yi.x, yi.y, yi.z, yi.w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const __nv_bfloat16 lo = __float2bfloat16_rn(bf16lo(w[h]) + s[2 * h]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(bf16hi(w[h]) + s[2 * h + 1]);
                o[h] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
            }
            *reinterpret_cast<uint4 *>(e.y + (size_t)t * d_out + c0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }

    // the last CTA to leave advances the barrier base for the next launch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned old = atomicAdd(reinterpret_cast<unsigned *>(e.m.hdr + HDR_EXIT), 1u);
        if (old == (unsigned)G - 1u) {
            e.m.hdr[HDR_BAR_BASE] = (int)(base + nbar * (unsigned)G);
            e.m.hdr[HDR_EXIT] = 0;
            __threadfence();
        }
    }
    (void)ok;
}

// Largest dynamic shared memory k_fused<CPT> may take on this device.
template <int CPT>
int fused_dynamic_limit()
{
    static thread_local int cached = -1, cached_dev = -1;  // per host thread
    int dev = 0;
    cudaGetDevice(&dev);
    if (cached_dev != dev) {
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, k_fused<CPT>);
        cached = optin - (int)fa.sharedSizeBytes;
        cached_dev = dev;
    }
    return cached;
}

template <int CPT>
cudaError_t launch_fused_cpt(FusedArgs a, int grid, size_t exp_bytes, cudaStream_t st)
{
    const int dyn_max = fused_dynamic_limit<CPT>();
    const long long room = (long long)dyn_max - (long long)exp_bytes;
    const int ring = (int)((room < FUSED_RING_MAX ? room : FUSED_RING_MAX) & ~1023LL);
    if (ring < 2 * SHRINK_MIN_ENTRY)
        return cudaErrorNotSupported;
    a.s.ring_bytes = ring;
    a.s.entry_bytes = ring / 2;
    static thread_local int attr_done = -1;  // per host thread
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_fused<CPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_fused<CPT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(EXP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = exp_bytes + (size_t)ring;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_fused<CPT>, a);
}

}  // namespace

bool fused_supported(int T, int d_out)
{
    return T >= 1 && (long long)T * 32 <= EXP_TILE_ELEMS && d_out % 32 == 0;
}

cudaError_t launch_fused(const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks,
                         const MapDev &m, int T, int P, const ExpandPlan &plan, int grid, cudaStream_t st)
{
    const int use_tab = pool.capacity <= RANK_TAB_MAX ? 1 : 0;
    const size_t exp_bytes = (expand_smem_bytes(plan.tb, plan.w, pool.capacity) + 127) & ~(size_t)127;
    FusedArgs a;
    a.s = ShrinkArgs{x, pool, ranks, m, z_stride(pool.r_max), shrink_tile_bound(P, pool.capacity), use_tab, 0, 0};
    a.e = ExpandArgs{y, pool, ranks, m, T, plan.tb, z_stride(pool.r_max), plan.w, plan.ng, use_tab};
    a.n_exp = (pool.d_out / plan.w) * plan.ng;
    a.partial = m.partial;
    if (a.n_exp > grid || (plan.ng > 1 && a.n_exp > m.partial_ctas) || plan.tb * plan.w > EXP_TILE_ELEMS)
        return cudaErrorNotSupported;
    switch (expand_cpt(plan.tb, plan.w)) {
    case 2:
        return launch_fused_cpt<2>(a, grid, exp_bytes, st);
    case 4:
        return launch_fused_cpt<4>(a, grid, exp_bytes, st);
    case 8:
        return launch_fused_cpt<8>(a, grid, exp_bytes, st);
    case 16:
        return launch_fused_cpt<16>(a, grid, exp_bytes, st);
    case 32:
        return launch_fused_cpt<32>(a, grid, exp_bytes, st);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace tcl
