// Split-path shrink kernel: the shrink phase (shrink_core.cuh) on a
// persistent grid, one CTA per SM beside one expand CTA.
// griddepcontrol.launch_dependents at entry lets the expand kernel that
// follows start its z-independent work (metadata, B tiles, y tile, pair
// lists) while this one runs.
#include "shrink_core.cuh"

namespace tcl {

namespace {

// 136 registers x 256 threads leaves room for an expand CTA on the same SM.
__global__ void __maxnreg__(136) k_shrink(ShrinkArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ ShrinkShared sh;
    unsigned char *ring = smem_raw;
    int *rank_tab = reinterpret_cast<int *>(smem_raw + a.ring_bytes);

    pdl_launch_dependents();
    if (a.use_tab)
        for (int i = threadIdx.x; i < a.pool.capacity; i += SHRINK_THREADS)
            rank_tab[i] = effective_rank(a.pool, a.ranks, i);
    // (shrink_phase synchronises the CTA before it reads rank_tab)
    shrink_phase<false>(a, sh, ring, rank_tab, blockIdx.x, gridDim.x);
}

}  // namespace

cudaError_t launch_shrink(const __nv_bfloat16 *x, const PoolDev &pool, const int32_t *ranks,
                          const MapDev &m, int P, int grid, cudaStream_t st)
{
    const int use_tab = pool.capacity <= RANK_TAB_MAX ? 1 : 0;
    const size_t smem = (size_t)SHRINK_RING_BYTES + (use_tab ? (size_t)((pool.capacity + 3) & ~3) * sizeof(int) : 0);
    static thread_local int attr_done = -1;  // per host thread
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_done != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_shrink, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SHRINK_RING_BYTES + RANK_TAB_MAX * (int)sizeof(int));
        // the largest shared-memory carveout, so an expand CTA fits beside this one
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_shrink, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        attr_done = dev;
    }
    ShrinkArgs a{x, pool, ranks, m, z_stride(pool.r_max), shrink_tile_bound(P, pool.capacity), use_tab,
                 SHRINK_RING_BYTES, SHRINK_RING_BYTES / 2};
    k_shrink<<<grid, SHRINK_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace tcl
