// Split-path expand kernel (RowExpand), launched with programmatic dependent
// launch after k_shrink.  The phase itself lives in expand_core.cuh.
//
// CTA = (token block [t0, t0 + tb), blockIdx.y) x (W output columns) x
// (segment group g of ng).  The ng CTAs of one column tile form a thread-block
// cluster: each sums the pairs of its share of the segments, then the cluster
// reduces the ng fp32 tiles through distributed shared memory in a fixed
// order, adds y and rounds once to bf16.  No global atomics; the result does
// not depend on timing.
#include "expand_core.cuh"

namespace tcl {

namespace {

// CPT: columns of the tile owned by one thread (2, 4, 8, 16 or 32); the
// tile width W and the threads per token TPT = W / CPT are runtime values.
template <int CPT>
__global__ void __launch_bounds__(EXP_THREADS, 2) k_expand(ExpandArgs a)
{
    static_assert(CPT == 2 || CPT == 4 || CPT == 8 || CPT == 16 || CPT == 32, "columns per thread");
    const int W = a.w;
    const int VPR = W / 8;  // 16-byte vectors per tile row
    const int TPT = W / CPT;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ ExpandShared es;
    const ExpLayout L(a.tb, W, a.use_tab ? a.pool.capacity : 0);
    float *acc = reinterpret_cast<float *>(smem_raw + L.B);  // reuses the B area after the last window
    __nv_bfloat16 *yin = reinterpret_cast<__nv_bfloat16 *>(smem_raw + L.yin);

    const int tid = threadIdx.x;
    const int d_out = a.pool.d_out;
    const int ng = a.ng;
    const int g = ng > 1 ? (int)cluster_ctarank() : 0;
    const int c0 = (blockIdx.x / ng) * W;
    const int t0 = blockIdx.y * a.tb, t1 = min(a.T, t0 + a.tb), nt = t1 - t0;
    const bool full_range = (t0 == 0 && t1 >= a.T);
    const int r0 = (nt * g) / ng, r1 = (nt * (g + 1)) / ng;  // rows of the tile this CTA finalises

    const int U = expand_prologue(a, smem_raw, c0, t0, r0, r1);
    const int my_t = tid / TPT, my_c = (tid % TPT) * CPT;
    float racc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c)
        racc[c] = 0.f;
    const int s_begin = (int)(((long long)U * g) / ng), s_end = (int)(((long long)U * (g + 1)) / ng);
    __syncthreads();

    expand_accumulate<CPT>(a, smem_raw, es, c0, t0, nt, full_range, s_begin, s_end, racc, [] { pdl_wait(); });

    if (my_t < nt) {
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

    // ---- reduce the ng accumulators of the cluster (fixed order), add y, round once
    if (ng > 1)
        cluster_sync();
    for (int i = tid; i < (r1 - r0) * VPR; i += EXP_THREADS) {
        const int t = r0 + i / VPR, v = i % VPR;
        const float *ap = &acc[t * W + v * 8];
        float s[8];
        if (ng > 1) {
            const float4 p0 = ld_dsmem_f4(ap, 0), p1 = ld_dsmem_f4(ap + 4, 0);
            s[0] = p0.x; s[1] = p0.y; s[2] = p0.z; s[3] = p0.w;
            s[4] = p1.x; s[5] = p1.y; s[6] = p1.z; s[7] = p1.w;
            for (int gg = 1; gg < ng; ++gg) {
                const float4 q0 = ld_dsmem_f4(ap, (uint32_t)gg), q1 = ld_dsmem_f4(ap + 4, (uint32_t)gg);
                s[0] += q0.x; s[1] += q0.y; s[2] += q0.z; s[3] += q0.w;
                s[4] += q1.x; s[5] += q1.y; s[6] += q1.z; s[7] += q1.w;
            }
        } else {
#pragma unroll
            for (int h = 0; h < 8; ++h)
                s[h] = ap[h];
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
        *reinterpret_cast<uint4 *>(a.y + (size_t)(t0 + t) * d_out + c0 + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (ng > 1)
        cluster_sync();  // keep this CTA's accumulator alive until the cluster has read it
}

template <int CPT>
cudaError_t launch_cpt(const ExpandArgs &a, dim3 grid, size_t smem, bool pdl, cudaStream_t st)
{
    static thread_local int attr_done = -1;  // per host thread
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_expand<CPT>, cudaFuncAttributeMaxDynamicSharedMemorySize, EXP_SMEM_MAX);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_expand<CPT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(EXP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.ng;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_expand<CPT>, a);
}

}  // namespace

size_t expand_smem_bytes(int tb, int w, int capacity)
{
    return (size_t)ExpLayout(tb, w, capacity <= RANK_TAB_MAX ? capacity : 0).total;
}

// Columns per thread for a tb x w tile over EXP_THREADS threads (power of two,
// 2..32).  Exposed so that host code and tests agree with the kernel.
int expand_cpt(int tb, int w)
{
    int cpt = 2;
    while (cpt < 32 && (long long)tb * w > (long long)cpt * EXP_THREADS)
        cpt *= 2;
    while (w / cpt > EXP_THREADS)
        cpt *= 2;
    return cpt;
}

cudaError_t launch_expand(__nv_bfloat16 *y, const PoolDev &pool, const int32_t *ranks, const MapDev &m, int T,
                          const ExpandPlan &plan, bool pdl, cudaStream_t st)
{
    const int use_tab = pool.capacity <= RANK_TAB_MAX ? 1 : 0;
    ExpandArgs a{y, pool, ranks, m, T, plan.tb, z_stride(pool.r_max), plan.w, plan.ng, use_tab};
    const size_t smem = expand_smem_bytes(plan.tb, plan.w, pool.capacity);
    const dim3 grid((pool.d_out / plan.w) * plan.ng, (T + plan.tb - 1) / plan.tb, 1);
    switch (expand_cpt(plan.tb, plan.w)) {
    case 2:
        return launch_cpt<2>(a, grid, smem, pdl, st);
    case 4:
        return launch_cpt<4>(a, grid, smem, pdl, st);
    case 8:
        return launch_cpt<8>(a, grid, smem, pdl, st);
    case 16:
        return launch_cpt<16>(a, grid, smem, pdl, st);
    case 32:
        return launch_cpt<32>(a, grid, smem, pdl, st);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace tcl
