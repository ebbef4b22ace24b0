// The C ABI declared in include/lora.h: objects, argument checks, dispatch.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

struct lora_pool {
    int d_in, d_out, r_max, capacity, device;
    // unique over the process lifetime: a pool created where a destroyed one
    // lived (same host address) is still a different pool
    unsigned long long serial;
    __nv_bfloat16 *At;  // [capacity][r_max][d_in]
    __nv_bfloat16 *B;   // [capacity][r_max][d_out]
    int32_t *reg_rank;  // [capacity]
    tcl::MmaMaps maps;  // TMA descriptors of At and B (tensor-core path)
};

// The arguments of a lora_delta_apply_host call: a repeat of the same ones
// replays a captured graph of the whole step.  The pool enters by its serial
// number, not its address: a graph captured against a destroyed pool holds
// that pool's device pointers and must never replay for a new pool that
// happens to occupy the same host memory.
struct HostStepKey {
    const void *x, *y;
    const int32_t *off, *ids;
    const float *alpha;
    int T, P;
    unsigned long long pool_serial;
    const int32_t *ranks;
    void *stream;
    bool operator==(const HostStepKey &o) const
    {
        return x == o.x && y == o.y && off == o.off && ids == o.ids && alpha == o.alpha && T == o.T && P == o.P &&
               pool_serial == o.pool_serial && ranks == o.ranks && stream == o.stream;
    }
};

// Device addresses of a call's host buffers (null where the GPU cannot
// address one directly); direct = all five exist, so the copy kernels run.
struct HostAliases {
    const void *x, *y, *off, *ids, *alpha;
    bool direct;
    bool operator==(const HostAliases &o) const
    {
        return x == o.x && y == o.y && off == o.off && ids == o.ids && alpha == o.alpha && direct == o.direct;
    }
    bool operator!=(const HostAliases &o) const { return !(*this == o); }
};

struct lora_mapping {
    int max_tokens, max_pairs, capacity, device;
    int T, P;
    bool built;
    // host-side record of the sort stage: builds so far, and the build and
    // stream (by its unique id: a handle may be reused after destruction) of
    // the last sort enqueued eagerly (not into a graph).  graph_builds: a
    // build was enqueued into a caller's graph, whose replays the count
    // cannot see -- the sort launch is then never left out.  self_capture:
    // the host entry point is capturing its own step graph (its replays
    // advance the count).
    long long builds, sorted_builds;
    unsigned long long sorted_stream;
    bool sorted_valid, graph_builds, self_capture;
    tcl::MapDev dev;
    // staging of lora_delta_apply_host
    void *sx, *sy;
    int32_t *soff, *sids;
    float *salpha;
    int s_d_in, s_d_out;
    // its step graph: `seen` is the last eager call's arguments, `exec` the
    // graph captured for `graph_key` with the buffers' addresses `graph_alias`;
    // nocap_key's capture failed (it stays eager)
    HostStepKey seen, graph_key, nocap_key;
    HostAliases graph_alias;
    bool have_seen, have_nocap;
    cudaGraphExec_t exec;
};

namespace tcl {

namespace {

__global__ void k_transpose_bf16(const __nv_bfloat16 *__restrict__ src, __nv_bfloat16 *__restrict__ dst, int rows,
                                 int cols)
{
    // dst[c][r] = src[r][c], 32 x 32 tiles through shared memory
    __shared__ __nv_bfloat16 tile[32][33];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols)
            tile[i][threadIdx.x] = src[(size_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols)
            dst[(size_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

__global__ void k_set_int(int32_t *p, int v) { *p = v; }

// Up to five copies in one launch, 16 bytes per thread-step where both ends
// allow it: the host entry point's transfers between pinned host memory
// (addressed directly by the GPU) and device staging.
struct CopySet {
    const unsigned char *src[5];
    unsigned char *dst[5];
    unsigned long long bytes[5];
    int n;
};

constexpr int CP_UNROLL = 4;  // 16-byte loads each thread keeps in flight

__global__ void __launch_bounds__(256) k_copy_set(const CopySet c)
{
    const unsigned long long nthr = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long span = nthr * CP_UNROLL;  // vectors one round of the grid moves
#pragma unroll
    for (int i = 0; i < 5; ++i) {  // unrolled: the parameter arrays stay unindexed at run time
        if (i >= c.n)
            break;
        const unsigned char *s = c.src[i];
        unsigned char *d = c.dst[i];
        const unsigned long long n = c.bytes[i];
        const bool vec = ((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) & 15u) == 0;
        const unsigned long long nv = vec ? n / 16 : 0;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
        uint4 *d4 = reinterpret_cast<uint4 *>(d);
        // whole rounds: block b's threads own [b * 256 * CP_UNROLL, +256 * CP_UNROLL) of each
        // round, the CP_UNROLL loads of a thread blockDim apart (coalesced per warp)
        const unsigned long long full = nv / span * span;
        for (unsigned long long base = (unsigned long long)blockIdx.x * blockDim.x * CP_UNROLL + threadIdx.x;
             base < full; base += span) {
            uint4 v[CP_UNROLL];
#pragma unroll
            for (int u = 0; u < CP_UNROLL; ++u)
                v[u] = s4[base + (unsigned long long)u * blockDim.x];
#pragma unroll
            for (int u = 0; u < CP_UNROLL; ++u)
                d4[base + (unsigned long long)u * blockDim.x] = v[u];
        }
        for (unsigned long long j = full + tid; j < nv; j += nthr)
            d4[j] = s4[j];
        for (unsigned long long j = nv * 16 + tid; j < n; j += nthr)
            d[j] = s[j];
    }
}

// A decode step's x rows from pinned host memory into the device staging,
// once per step: the shrink reads a token's row once per pair and rank-row
// group, and those repeats stay in device memory instead of crossing the
// host link again.  Launched as a programmatic dependent, it lets the
// mapping stage behind it start at once (that stage stages its own inputs,
// then waits for this grid); it reads the host buffer only after its own
// wait, since the kernel ahead (the previous step's expand) may still be
// writing a y that is this step's x.  Both ends 16-byte aligned, n16 vectors.
constexpr int HI_UNROLL = 2;  // 16-byte loads a thread keeps in flight: 8 KB per CTA

__global__ void __launch_bounds__(256) k_host_in(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                 unsigned long long n16)
{
    pdl_launch_dependents();
    pdl_wait();
    const unsigned long long i0 = (unsigned long long)blockIdx.x * 256 * HI_UNROLL + threadIdx.x;
    uint4 v[HI_UNROLL];
#pragma unroll
    for (int u = 0; u < HI_UNROLL; ++u) {
        const unsigned long long i = i0 + 256ull * u;
        v[u] = i < n16 ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < HI_UNROLL; ++u) {
        const unsigned long long i = i0 + 256ull * u;
        if (i < n16)
            dst[i] = v[u];
    }
}

cudaError_t launch_host_in(const void *src, void *dst, size_t bytes, cudaStream_t st)
{
    const unsigned long long n16 = bytes / 16;
    if (n16 == 0)
        return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((n16 + 256ull * HI_UNROLL - 1) / (256ull * HI_UNROLL)), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_host_in, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
}

// SM count of the current device, cached per host thread (device and count
// together, so a thread never pairs one device with another's count).
struct SmCache {
    int dev = -1, count = 0;
};
thread_local SmCache t_sm;

std::atomic<unsigned long long> g_pool_serial{0};

}  // namespace

cudaError_t launch_transpose_bf16(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int rows, int cols,
                                  cudaStream_t st)
{
    dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
    k_transpose_bf16<<<grid, block, 0, st>>>(src, dst, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_set_int(int32_t *p, int v, cudaStream_t st)
{
    k_set_int<<<1, 1, 0, st>>>(p, v);
    return cudaGetLastError();
}

cudaError_t launch_copy_set(const CopySet &c, cudaStream_t st)
{
    unsigned long long total = 0;
    for (int i = 0; i < c.n; ++i)
        total += c.bytes[i];
    if (total == 0)
        return cudaSuccess;
    unsigned long long blocks = (total / 16 + 256ull * CP_UNROLL - 1) / (256ull * CP_UNROLL);
    const unsigned long long cap = 4ull * sm_count();
    if (blocks > cap)
        blocks = cap;
    k_copy_set<<<(unsigned)(blocks ? blocks : 1), 256, 0, st>>>(c);
    return cudaGetLastError();
}

int sm_count()
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != t_sm.dev) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return 1;  // not cached: asked again on the next call
        t_sm.count = n;
        t_sm.dev = dev;
    }
    return t_sm.count;
}

}  // namespace tcl

using namespace tcl;

namespace {

lora_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess)
        return LORA_OK;
    if (e == cudaErrorMemoryAllocation)
        return LORA_ERR_OUT_OF_MEMORY;
    return LORA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PoolDev pool_dev(const lora_pool *p)
{
    PoolDev d;
    d.At = p->At;
    d.B = p->B;
    d.reg_rank = p->reg_rank;
    d.d_in = p->d_in;
    d.d_out = p->d_out;
    d.r_max = p->r_max;
    d.capacity = p->capacity;
    return d;
}

template <typename T>
cudaError_t dalloc(T **p, size_t count)
{
    return cudaMalloc(reinterpret_cast<void **>(p), (count > 0 ? count : 1) * sizeof(T));
}

// Frees the host entry point's device staging; the step graph (which copies
// into it) goes first, and the recorded shape is cleared until a new staging
// is complete.
void free_staging(lora_mapping *m)
{
    if (m->exec) {
        cudaGraphExecDestroy(m->exec);
        m->exec = nullptr;
    }
    m->have_seen = false;
    void *ptrs[] = {m->sx, m->sy, m->soff, m->sids, m->salpha};
    for (void *p : ptrs)
        if (p)
            cudaFree(p);
    m->sx = m->sy = nullptr;
    m->soff = m->sids = nullptr;
    m->salpha = nullptr;
    m->s_d_in = m->s_d_out = 0;
}

void free_mapping(lora_mapping *m)
{
    if (m->exec)
        cudaGraphExecDestroy(m->exec);
    MapDev &d = m->dev;
    void *ptrs[] = {d.tok,  d.adapter, d.src, d.pos,     d.alpha, d.seg_adapter, d.seg_start,
                    d.tile, d.tile_tok, d.hdr, d.mtile, d.toff,     d.pc, d.calpha, d.zcnt, d.z,
                    d.partial, d.ghist, d.gsort, m->sx, m->sy, m->soff, m->sids, m->salpha};
    for (void *p : ptrs)
        if (p)
            cudaFree(p);
    std::free(m);
}

// Dispatch table (LoRAForge page, "Approach" (5): native path or a special
// kernel, fixed by phase, rank and shape), from a sweep of every path over
// tokens x rank x adapter sharing on this GPU.  The decode kernels (a CTA per
// pair; shared adapters' rows come from L2) are the fastest at every swept
// size of decode-like batches and of most others; the tensor-core path wins
// where long runs of tokens share their adapters (prefill chunks) and the
// rank is large enough to fill its tiles.  The phase is read from the token
// count: at least MMA_FROM tokens of a rank class are taken for a prefill
// batch.  The sharing itself is not known on the host (the pair lists are on
// the device), so it does not enter the choice.  The split path is never the
// fastest on the sweep; it serves shapes that neither of the others takes.
int mma_from_tokens(int r_max)
{
    if (r_max <= 8)
        return MMA_FROM_R8;
    if (r_max <= 16)
        return MMA_FROM_R16;
    return MMA_FROM_R64;
}

int choose_path(int T, int P, int r_max, int d_in, int d_out)
{
    (void)P;
    const bool mma = mma_supported(d_in, d_out, r_max);
    if (mma && T >= mma_from_tokens(r_max))
        return LORA_PATH_MMA;
    if (decode_supported(d_in, d_out))
        return LORA_PATH_DECODE;
    return LORA_PATH_SPLIT;
}

// Expand plan.  Decode batches (T * 32 <= EXP_TILE_ELEMS) take the whole
// batch as one token block and split each column tile's segments over a
// cluster of ng CTAs, choosing (W, ng) for the most CTAs that still fit one
// per SM beside the shrink (ties: the middle width, then wider).  Longer
// batches take 64 columns and the largest token block that gives a CTA per SM.
ExpandPlan choose_expand_plan(int T, int d_out)
{
    const int sms = sm_count();
    ExpandPlan best{0, 0, 0};
    if ((long long)T * 32 <= EXP_TILE_ELEMS) {
        int best_ctas = -1;
        const int order[3] = {64, 128, 32};
        for (int w : order) {
            if (d_out % w || (long long)T * w > EXP_TILE_ELEMS)
                continue;
            const int n_ct = d_out / w;
            if (n_ct > sms)
                continue;
            int ng = 1;
            while (ng < 8 && (long long)n_ct * ng * 2 <= sms)
                ng *= 2;
            if (n_ct * ng > best_ctas) {
                best_ctas = n_ct * ng;
                best = ExpandPlan{T, w, ng};
            }
        }
        if (best_ctas > 0)
            return best;
    }
    best.w = 64;
    best.ng = 1;
    const int n_ct = d_out / 64;
    best.tb = EXP_TILE_ELEMS / 64;
    while (best.tb > 8 && (long long)n_ct * ((T + best.tb - 1) / best.tb) < sms)
        best.tb >>= 1;
    return best;
}

// The adapter-sorted tuples of the mapping's current build (the sort stage
// returns at once when they are there already).
// The sort stage before a path that reads the adapter-sorted tuples.  Its
// kernel checks on the device whether the current build is sorted (so
// graphs and other streams stay correct); on the host, a sort enqueued
// eagerly on this same stream since the last build is already ahead of this
// call in stream order, and the launch is left out.
cudaError_t sort_mapping(const lora_mapping *cm, cudaStream_t st)
{
    lora_mapping *m = const_cast<lora_mapping *>(cm);  // host-side bookkeeping only
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        cs = cudaStreamCaptureStatusActive;  // unknown: launch, record nothing
    }
    unsigned long long sid = 0;
    bool eager = cs == cudaStreamCaptureStatusNone;
    if (eager && cudaStreamGetId(st, &sid) != cudaSuccess) {
        cudaGetLastError();
        eager = false;  // no id: launch, record nothing
    }
    if (eager && !m->graph_builds && m->sorted_valid && m->sorted_stream == sid && m->sorted_builds == m->builds)
        return cudaSuccess;
    const cudaError_t e = launch_map_sort(m->dev, m->T, m->P, m->capacity, st);
    if (e == cudaSuccess && eager) {
        m->sorted_valid = true;
        m->sorted_stream = sid;
        m->sorted_builds = m->builds;
    }
    return e;
}

lora_status run_fused(const void *x, void *y, const lora_pool *pool, const int32_t *ranks, const lora_mapping *m,
                      cudaStream_t st)
{
    if (decode_supported(pool->d_in, pool->d_out)) {
        const cudaError_t e = launch_decode_fused(static_cast<const __nv_bfloat16 *>(x),
                                                  static_cast<__nv_bfloat16 *>(y), pool_dev(pool), ranks, m->dev,
                                                  m->T, m->P, st);
        if (e != cudaErrorNotSupported)
            return from_cuda(e);
    }
    if (!fused_supported(m->T, pool->d_out))
        return LORA_ERR_NOT_SUPPORTED;
    const ExpandPlan plan = choose_expand_plan(m->T, pool->d_out);
    cudaError_t e = sort_mapping(m, st);
    if (e != cudaSuccess)
        return from_cuda(e);
    e = launch_fused(static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(y),
                                       pool_dev(pool), ranks, m->dev, m->T, m->P, plan, sm_count(), st);
    if (e == cudaErrorNotSupported)
        return LORA_ERR_NOT_SUPPORTED;  // the shape does not fit this kernel
    return from_cuda(e);
}

lora_status run_mma(const void *x, void *y, const lora_pool *pool, const int32_t *ranks, const lora_mapping *m,
                    cudaStream_t st)
{
    if (!pool->maps.ready || !mma_supported(pool->d_in, pool->d_out, pool->r_max))
        return LORA_ERR_NOT_SUPPORTED;
    cudaError_t e = sort_mapping(m, st);
    if (e != cudaSuccess)
        return from_cuda(e);
    e = launch_mma(static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(y),
                                     pool_dev(pool), pool->maps, ranks, m->dev, m->T, m->P, st);
    if (e == cudaErrorNotSupported)
        return LORA_ERR_NOT_SUPPORTED;
    return from_cuda(e);
}

lora_status run_decode(const void *x, void *y, const lora_pool *pool, const int32_t *ranks,
                       const lora_mapping *m, cudaStream_t st)
{
    const cudaError_t e = launch_decode(static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(y),
                                        pool_dev(pool), ranks, m->dev, m->T, m->P, st);
    if (e == cudaErrorNotSupported)
        return LORA_ERR_NOT_SUPPORTED;
    return from_cuda(e);
}

lora_status run_split(const void *x, void *y, const lora_pool *pool, const int32_t *ranks, const lora_mapping *m,
                      cudaStream_t st)
{
    const PoolDev pd = pool_dev(pool);
    const int grid = sm_count();
    cudaError_t e = sort_mapping(m, st);
    if (e == cudaSuccess)
        e = launch_shrink(static_cast<const __nv_bfloat16 *>(x), pd, ranks, m->dev, m->P, grid, st);
    if (e != cudaSuccess)
        return from_cuda(e);
    const ExpandPlan plan = choose_expand_plan(m->T, pool->d_out);
    e = launch_expand(static_cast<__nv_bfloat16 *>(y), pd, ranks, m->dev, m->T, plan, /*pdl=*/true, st);
    return from_cuda(e);
}

}  // namespace

extern "C" {

const char *lora_status_string(lora_status s)
{
    switch (s) {
    case LORA_OK:
        return "ok";
    case LORA_ERR_INVALID_ARG:
        return "invalid argument";
    case LORA_ERR_OUT_OF_MEMORY:
        return "out of device memory";
    case LORA_ERR_CUDA:
        return "CUDA error";
    case LORA_ERR_BAD_ADAPTER:
        return "bad adapter slot or rank";
    case LORA_ERR_NOT_SUPPORTED:
        return "not supported by this implementation";
    }
    return "unknown status";
}

const char *lora_version(void) { return "tclora 0.1 (sm_103a)"; }

int lora_dispatch_choose(int T, int P, int r_max, int d_in, int d_out)
{
    return choose_path(T, P, r_max, d_in, d_out);
}

lora_status lora_pool_create(int d_in, int d_out, int r_max, int capacity, lora_pool **out)
{
    if (!out)
        return LORA_ERR_INVALID_ARG;
    *out = nullptr;
    if (d_in <= 0 || d_out <= 0 || r_max <= 0 || capacity <= 0)
        return LORA_ERR_INVALID_ARG;
    if (d_in % LORA_DIM_MULTIPLE || d_out % LORA_DIM_MULTIPLE || r_max > LORA_MAX_RANK ||
        capacity > LORA_MAX_CAPACITY)
        return LORA_ERR_NOT_SUPPORTED;
    lora_pool *p = static_cast<lora_pool *>(std::calloc(1, sizeof(lora_pool)));
    if (!p)
        return LORA_ERR_OUT_OF_MEMORY;
    p->d_in = d_in;
    p->d_out = d_out;
    p->r_max = r_max;
    p->capacity = capacity;
    p->serial = ++g_pool_serial;
    cudaGetDevice(&p->device);
    const size_t na = (size_t)capacity * r_max * d_in, nb = (size_t)capacity * r_max * d_out;
    cudaError_t e = dalloc(&p->At, na);
    if (e == cudaSuccess)
        e = dalloc(&p->B, nb);
    if (e == cudaSuccess)
        e = dalloc(&p->reg_rank, (size_t)capacity);
    if (e == cudaSuccess)
        e = cudaMemset(p->At, 0, na * sizeof(__nv_bfloat16));
    if (e == cudaSuccess)
        e = cudaMemset(p->B, 0, nb * sizeof(__nv_bfloat16));
    if (e == cudaSuccess)
        e = cudaMemset(p->reg_rank, 0xff, (size_t)capacity * sizeof(int32_t));  // -1: unregistered
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        mma_encode_maps(pool_dev(p), p->maps);  // without it the tensor-core path reports NOT_SUPPORTED
    if (e != cudaSuccess) {
        if (p->At)
            cudaFree(p->At);
        if (p->B)
            cudaFree(p->B);
        if (p->reg_rank)
            cudaFree(p->reg_rank);
        std::free(p);
        return from_cuda(e);
    }
    *out = p;
    return LORA_OK;
}

lora_status lora_pool_register(lora_pool *pool, int slot, const void *A_dev, const void *B_dev, int k,
                               lora_stream_t stream)
{
    if (!pool || !A_dev || !B_dev || slot < 0 || slot >= pool->capacity || k < 0 || k > pool->r_max)
        return LORA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t off_a = (size_t)slot * pool->r_max * pool->d_in;
    const size_t off_b = (size_t)slot * pool->r_max * pool->d_out;
    cudaError_t e = launch_transpose_bf16(static_cast<const __nv_bfloat16 *>(A_dev), pool->At + off_a, pool->d_in,
                                          pool->r_max, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(pool->B + off_b, B_dev, (size_t)pool->r_max * pool->d_out * sizeof(__nv_bfloat16),
                            cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess)
        e = launch_set_int(pool->reg_rank + slot, k, st);
    return from_cuda(e);
}

lora_status lora_pool_unregister(lora_pool *pool, int slot, lora_stream_t stream)
{
    if (!pool || slot < 0 || slot >= pool->capacity)
        return LORA_ERR_INVALID_ARG;
    return from_cuda(launch_set_int(pool->reg_rank + slot, -1, static_cast<cudaStream_t>(stream)));
}

lora_status lora_pool_destroy(lora_pool *pool)
{
    if (!pool)
        return LORA_OK;
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(pool->At);
    cudaFree(pool->B);
    cudaFree(pool->reg_rank);
    std::free(pool);
    return from_cuda(e);
}

lora_status lora_mapping_create(int max_tokens, int max_pairs, int capacity, lora_mapping **out)
{
    if (!out)
        return LORA_ERR_INVALID_ARG;
    *out = nullptr;
    if (max_tokens < 0 || max_pairs < 0 || capacity <= 0)
        return LORA_ERR_INVALID_ARG;
    if (max_tokens > LORA_MAX_TOKENS || max_pairs > LORA_MAX_PAIRS || capacity > LORA_MAX_CAPACITY)
        return LORA_ERR_NOT_SUPPORTED;
    lora_mapping *m = static_cast<lora_mapping *>(std::calloc(1, sizeof(lora_mapping)));
    if (!m)
        return LORA_ERR_OUT_OF_MEMORY;
    m->max_tokens = max_tokens;
    m->max_pairs = max_pairs;
    m->capacity = capacity;
    cudaGetDevice(&m->device);
    MapDev &d = m->dev;
    const size_t P = (size_t)max_pairs;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = dalloc(&d.tok, P);
    if (e == cudaSuccess) e = dalloc(&d.adapter, P);
    if (e == cudaSuccess) e = dalloc(&d.src, P);
    if (e == cudaSuccess) e = dalloc(&d.pos, P);
    if (e == cudaSuccess) e = dalloc(&d.alpha, P);
    if (e == cudaSuccess) e = dalloc(&d.seg_adapter, (size_t)capacity);
    if (e == cudaSuccess) e = dalloc(&d.seg_start, (size_t)capacity + 1);
    if (e == cudaSuccess) e = dalloc(&d.tile, P);
    if (e == cudaSuccess) e = dalloc(&d.tile_tok, P * SHRINK_TT);
    if (e == cudaSuccess) e = dalloc(&d.hdr, (size_t)HDR_WORDS);
    if (e == cudaSuccess) e = dalloc(&d.mtile, (size_t)mma_tile_bound(max_pairs, capacity));
    if (e == cudaSuccess) e = dalloc(&d.toff, (size_t)max_tokens + 1);
    if (e == cudaSuccess) e = dalloc(&d.pc, P);
    if (e == cudaSuccess) e = dalloc(&d.calpha, P);
    if (e == cudaSuccess) e = dalloc(&d.zcnt, P);
    if (e == cudaSuccess) e = dalloc(&d.z, P * Z_ROW_FLOATS);
    d.partial_ctas = sm_count();
    if (e == cudaSuccess) e = dalloc(&d.partial, (size_t)d.partial_ctas * EXP_TILE_ELEMS);
    if (e == cudaSuccess && map_global_hist_words(capacity) > 0)
        e = dalloc(&d.ghist, (size_t)map_global_hist_words(capacity));
    if (e == cudaSuccess && map_wide_sort_words(capacity) > 0)
        e = dalloc(&d.gsort, (size_t)map_wide_sort_words(capacity));
    if (e == cudaSuccess) e = cudaMemset(d.hdr, 0, HDR_WORDS * sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(d.seg_start, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_mapping(m);
        return from_cuda(e);
    }
    *out = m;
    return LORA_OK;
}

lora_status lora_build_mapping(lora_mapping *m, const int32_t *offsets_dev, const int32_t *ids_dev,
                               const float *alpha_dev, int T, int P, lora_stream_t stream)
{
    if (!m || !offsets_dev || T < 0 || P < 0 || T > m->max_tokens || P > m->max_pairs)
        return LORA_ERR_INVALID_ARG;
    if (P > 0 && (!ids_dev || !alpha_dev))
        return LORA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!m->self_capture) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
            cudaGetLastError();
            cs = cudaStreamCaptureStatusActive;  // unknown: as if captured
        }
        if (cs != cudaStreamCaptureStatusNone)
            m->graph_builds = true;
    }
    // the CSR stage only: the paths that read the adapter-sorted tuples sort
    // them first (once per build)
    cudaError_t e = launch_map_csr(m->dev, offsets_dev, ids_dev, alpha_dev, T, P, m->capacity, st);
    if (e != cudaSuccess)
        return from_cuda(e);
    m->T = T;
    m->P = P;
    m->built = true;
    ++m->builds;  // a later sorted path sorts this build
    return LORA_OK;
}

lora_status lora_delta_apply_path(const void *x_dev, void *y_dev, const lora_pool *pool, const int32_t *ranks_dev,
                                  const lora_mapping *m, int path, lora_stream_t stream)
{
    if (!x_dev || !y_dev || !pool || !m || !m->built || x_dev == y_dev)
        return LORA_ERR_INVALID_ARG;
    if (m->capacity != pool->capacity)
        return LORA_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(y_dev))
        return LORA_ERR_INVALID_ARG;
    if (m->T == 0 || m->P == 0)
        return LORA_OK;  // no pair: y is already the result
    if (path == LORA_PATH_AUTO)
        path = choose_path(m->T, m->P, pool->r_max, pool->d_in, pool->d_out);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (path) {
    case LORA_PATH_SPLIT:
        return run_split(x_dev, y_dev, pool, ranks_dev, m, st);
    case LORA_PATH_FUSED:
        return run_fused(x_dev, y_dev, pool, ranks_dev, m, st);
    case LORA_PATH_MMA:
        return run_mma(x_dev, y_dev, pool, ranks_dev, m, st);
    case LORA_PATH_DECODE:
        return run_decode(x_dev, y_dev, pool, ranks_dev, m, st);
    default:
        return LORA_ERR_NOT_SUPPORTED;
    }
}

lora_status lora_delta_apply(const void *x_dev, void *y_dev, const lora_pool *pool, const int32_t *ranks_dev,
                             const lora_mapping *m, lora_stream_t stream)
{
    return lora_delta_apply_path(x_dev, y_dev, pool, ranks_dev, m, LORA_PATH_AUTO, stream);
}

size_t lora_ablation_workspace_bytes(int variant, int T, int P, int d_in, int d_out, int r_max)
{
    if (T < 0 || P < 0 || d_in <= 0 || d_out <= 0 || r_max <= 0)
        return 0;
    return ablation_workspace_bytes(variant, T, P, d_in, d_out, r_max);
}

lora_status lora_delta_apply_ablation(const void *x_dev, void *y_dev, const lora_pool *pool,
                                      const int32_t *ranks_dev, const lora_mapping *m, int variant,
                                      void *workspace_dev, size_t workspace_bytes, lora_stream_t stream)
{
    if (!x_dev || !y_dev || !pool || !m || !m->built || x_dev == y_dev || m->capacity != pool->capacity)
        return LORA_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(y_dev))
        return LORA_ERR_INVALID_ARG;
    if (variant != LORA_ABLATION_NAIVE && variant != LORA_ABLATION_COPY_SGMV && variant != LORA_ABLATION_PREMERGE)
        return LORA_ERR_NOT_SUPPORTED;
    const size_t need = ablation_workspace_bytes(variant, m->T, m->P, pool->d_in, pool->d_out, pool->r_max);
    if (need > 0 && (!workspace_dev || workspace_bytes < need || !aligned16(workspace_dev)))
        return LORA_ERR_INVALID_ARG;
    if (m->T == 0 || m->P == 0)
        return LORA_OK;
    return from_cuda(run_ablation(variant, static_cast<const __nv_bfloat16 *>(x_dev), static_cast<__nv_bfloat16 *>(y_dev),
                                  pool_dev(pool), ranks_dev, m->dev, m->T, m->P, workspace_dev,
                                  static_cast<cudaStream_t>(stream)));
}

size_t lora_recompress_workspace_bytes(int M, int d_in, int r)
{
    if (M < 1 || r < 1 || r > LORA_MAX_RANK || d_in < r)
        return 0;
    return recompress_workspace_bytes(M, d_in, r);
}

lora_status lora_recompress(const void *A_dev, const void *B_dev, int M, int d_in, int d_out, int r, float *F_dev,
                            float *T_dev, float *sigma_dev, void *workspace_dev, size_t workspace_bytes,
                            lora_stream_t stream)
{
    if (!A_dev || !B_dev || !F_dev || !T_dev || !sigma_dev || !workspace_dev || M < 0 || d_in < 1 || d_out < 1)
        return LORA_ERR_INVALID_ARG;
    if (r < 1 || r > LORA_MAX_RANK || d_in < r)
        return LORA_ERR_NOT_SUPPORTED;
    if (M == 0)
        return LORA_OK;
    if (workspace_bytes < recompress_workspace_bytes(M, d_in, r) || !aligned16(workspace_dev))
        return LORA_ERR_INVALID_ARG;
    const cudaError_t e =
        launch_recompress(static_cast<const __nv_bfloat16 *>(A_dev), static_cast<const __nv_bfloat16 *>(B_dev), M,
                          d_in, d_out, r, F_dev, T_dev, sigma_dev, workspace_dev, static_cast<cudaStream_t>(stream));
    return e == cudaErrorNotSupported ? LORA_ERR_NOT_SUPPORTED : from_cuda(e);
}

lora_status lora_rank_allocate(const float *sigma_host, int M, int r_stride, const int32_t *rank_host,
                               const int32_t *cost_host, int policy, int d, int floor_k, int32_t *k_host)
{
    if (!sigma_host || !rank_host || !cost_host || !k_host || M < 0 || r_stride < 1 || d < 1 || floor_k < 0)
        return LORA_ERR_INVALID_ARG;
    if (policy != LORA_RANK_UNIFORM && policy != LORA_RANK_SPECTRAL)
        return LORA_ERR_NOT_SUPPORTED;
    for (int m = 0; m < M; ++m)
        if (cost_host[m] < 1 || rank_host[m] < 0)
            return LORA_ERR_INVALID_ARG;
    rank_allocate(sigma_host, M, r_stride, rank_host, cost_host, policy, d, floor_k, k_host);
    return LORA_OK;
}

lora_status lora_delta_apply_multi(const lora_projection *projs, int n_proj, const lora_mapping *m,
                                   lora_stream_t stream)
{
    if (!projs || !m || !m->built || n_proj < 1)
        return LORA_ERR_INVALID_ARG;
    if (n_proj > LORA_MAX_PROJECTIONS)
        return LORA_ERR_NOT_SUPPORTED;
    int zcols = 0;
    bool decode_ok = true;
    for (int j = 0; j < n_proj; ++j) {
        const lora_projection &p = projs[j];
        if (!p.x_dev || !p.y_dev || !p.pool || p.x_dev == p.y_dev || p.pool->capacity != m->capacity)
            return LORA_ERR_INVALID_ARG;
        if (!aligned16(p.x_dev) || !aligned16(p.y_dev))
            return LORA_ERR_INVALID_ARG;
        for (int i = 0; i < j; ++i)
            if (projs[i].y_dev == p.y_dev || projs[i].x_dev == p.y_dev || p.x_dev == projs[i].y_dev)
                return LORA_ERR_INVALID_ARG;  // one projection's output is another's input or output
        zcols += z_stride(p.pool->r_max);
        decode_ok = decode_ok && choose_path(m->T, m->P, p.pool->r_max, p.pool->d_in, p.pool->d_out) ==
                                     LORA_PATH_DECODE;
    }
    if (m->T == 0 || m->P == 0)
        return LORA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (decode_ok && zcols <= Z_ROW_FLOATS) {
        MultiDecArgs a{};
        a.n = n_proj;
        a.m = m->dev;
        a.T = m->T;
        for (int j = 0; j < n_proj; ++j) {
            a.p[j].x = static_cast<const __nv_bfloat16 *>(projs[j].x_dev);
            a.p[j].y = static_cast<__nv_bfloat16 *>(projs[j].y_dev);
            a.p[j].pool = pool_dev(projs[j].pool);
            a.p[j].ranks = projs[j].ranks_dev;
        }
        const cudaError_t e = launch_decode_multi(a, m->P, st);
        if (e != cudaErrorNotSupported)
            return from_cuda(e);
    }
    // batches the dispatch table sends elsewhere for some projection (or
    // shapes the decode kernels do not take): one apply per projection, each
    // on the path the dispatch table picks
    for (int j = 0; j < n_proj; ++j) {
        const lora_status s =
            lora_delta_apply(projs[j].x_dev, projs[j].y_dev, projs[j].pool, projs[j].ranks_dev, m, stream);
        if (s != LORA_OK)
            return s;
    }
    return LORA_OK;
}

}  // extern "C"

namespace {

// The device address of a host buffer when the GPU can address it directly
// (pinned memory), else nullptr.
const void *device_alias(const void *host)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

HostAliases host_aliases(const void *x_host, const void *y_host, const int32_t *offsets_host, const int32_t *ids_host,
                         const float *alpha_host, int P)
{
    HostAliases a{};
    a.x = device_alias(x_host);
    a.y = device_alias(y_host);
    a.off = device_alias(offsets_host);
    a.ids = P > 0 ? device_alias(ids_host) : a.off;
    a.alpha = P > 0 ? device_alias(alpha_host) : a.off;
    a.direct = a.x && a.y && a.off && a.ids && a.alpha;
    return a;
}

// One step of lora_delta_apply_host, enqueued on the stream: the inputs in,
// the mapping, the apply, y back.  With pinned buffers the transfers are two
// copy kernels reading and writing host memory directly (one launch in, one
// out); otherwise one cudaMemcpyAsync per buffer.
lora_status host_step(const void *x_host, void *y_host, const int32_t *offsets_host, const int32_t *ids_host,
                      const float *alpha_host, int T, int P, const lora_pool *pool, const int32_t *ranks_dev,
                      lora_mapping *m, lora_stream_t stream, const HostAliases &al)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t xb = (size_t)T * pool->d_in * sizeof(__nv_bfloat16);
    const size_t yb = (size_t)T * pool->d_out * sizeof(__nv_bfloat16);
    const size_t ob = (size_t)(T + 1) * sizeof(int32_t), pb = (size_t)P * sizeof(int32_t);
    const void *ax = al.x, *ay = al.y, *ao = al.off, *ai = al.ids, *aa = al.alpha;
    cudaError_t e = cudaSuccess;
    const bool direct = al.direct;
    if (direct && aligned16(ax) && aligned16(ay) && ax != ay && xb % 16 == 0 &&
        choose_path(T, P, pool->r_max, pool->d_in, pool->d_out) == LORA_PATH_DECODE) {
        // decode batches: x crosses the host link once, into the device
        // staging, by one copy kernel that the mapping's CSR stage overlaps;
        // the CSR stage reads the pair lists and the expand reads and writes
        // y straight from and to the pinned host buffers (each byte crosses
        // once): no copy launch after the step
        e = launch_host_in(ax, m->sx, xb, st);
        if (e != cudaSuccess)
            return from_cuda(e);
        lora_status s = lora_build_mapping(m, static_cast<const int32_t *>(ao), static_cast<const int32_t *>(ai),
                                           static_cast<const float *>(aa), T, P, stream);
        if (s == LORA_OK)
            s = lora_delta_apply(m->sx, const_cast<void *>(ay), pool, ranks_dev, m, stream);
        return s;
    }
    if (direct) {
        CopySet in{};
        const void *srcs[5] = {ao, ai, aa, ax, ay};
        void *dsts[5] = {m->soff, m->sids, m->salpha, m->sx, m->sy};
        const size_t sizes[5] = {ob, P > 0 ? pb : 0, P > 0 ? pb : 0, xb, yb};
        for (int i = 0; i < 5; ++i) {
            in.src[in.n] = static_cast<const unsigned char *>(srcs[i]);
            in.dst[in.n] = static_cast<unsigned char *>(dsts[i]);
            in.bytes[in.n] = sizes[i];
            ++in.n;
        }
        e = launch_copy_set(in, st);
    } else {
        e = cudaMemcpyAsync(m->soff, offsets_host, ob, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && P > 0)
            e = cudaMemcpyAsync(m->sids, ids_host, pb, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && P > 0)
            e = cudaMemcpyAsync(m->salpha, alpha_host, pb, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && xb)
            e = cudaMemcpyAsync(m->sx, x_host, xb, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && yb)
            e = cudaMemcpyAsync(m->sy, y_host, yb, cudaMemcpyHostToDevice, st);
    }
    if (e != cudaSuccess)
        return from_cuda(e);
    lora_status s = lora_build_mapping(m, m->soff, m->sids, m->salpha, T, P, stream);
    if (s != LORA_OK)
        return s;
    s = lora_delta_apply(m->sx, m->sy, pool, ranks_dev, m, stream);
    if (s != LORA_OK)
        return s;
    if (yb) {
        if (direct) {
            CopySet out{};
            out.src[0] = static_cast<const unsigned char *>(m->sy);
            out.dst[0] = static_cast<unsigned char *>(const_cast<void *>(ay));
            out.bytes[0] = yb;
            out.n = 1;
            e = launch_copy_set(out, st);
        } else {
            e = cudaMemcpyAsync(y_host, m->sy, yb, cudaMemcpyDeviceToHost, st);
        }
    }
    return from_cuda(e);
}

}  // namespace

extern "C" {

lora_status lora_delta_apply_host(const void *x_host, void *y_host, const int32_t *offsets_host,
                                  const int32_t *ids_host, const float *alpha_host, int T, int P,
                                  const lora_pool *pool, const int32_t *ranks_dev, lora_mapping *m,
                                  lora_stream_t stream)
{
    if (!x_host || !y_host || !offsets_host || !pool || !m || T < 0 || P < 0 || T > m->max_tokens ||
        P > m->max_pairs || m->capacity != pool->capacity)
        return LORA_ERR_INVALID_ARG;
    if (P > 0 && (!ids_host || !alpha_host))
        return LORA_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    if (!m->sx || m->s_d_in != pool->d_in || m->s_d_out != pool->d_out) {
        e = cudaDeviceSynchronize();  // earlier steps may still use the old staging
        free_staging(m);
        const size_t mt = (size_t)(m->max_tokens > 0 ? m->max_tokens : 1);
        if (e == cudaSuccess) e = cudaMalloc(&m->sx, mt * pool->d_in * sizeof(__nv_bfloat16));
        if (e == cudaSuccess) e = cudaMalloc(&m->sy, mt * pool->d_out * sizeof(__nv_bfloat16));
        if (e == cudaSuccess) e = dalloc(&m->soff, mt + 1);
        if (e == cudaSuccess) e = dalloc(&m->sids, (size_t)m->max_pairs);
        if (e == cudaSuccess) e = dalloc(&m->salpha, (size_t)m->max_pairs);
        if (e != cudaSuccess) {
            free_staging(m);  // nothing half-built is kept
            return from_cuda(e);
        }
        m->s_d_in = pool->d_in;
        m->s_d_out = pool->d_out;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const HostStepKey key{x_host, y_host, offsets_host, ids_host, alpha_host, T, P, pool->serial, ranks_dev, stream};
    // where the GPU can address each buffer, looked up on every call: the
    // graph replays only while that is what it was captured with (a buffer
    // freed and another one allocated at its address, pinned or not, is
    // caught here)
    const HostAliases al = host_aliases(x_host, y_host, offsets_host, ids_host, alpha_host, P);
    if (m->exec && m->graph_key == key) {
        if (m->graph_alias == al) {
            m->T = T;  // the host-side state lora_build_mapping would leave
            m->P = P;
            m->built = true;
            ++m->builds;
            return from_cuda(cudaGraphLaunch(m->exec, st));
        }
        cudaGraphExecDestroy(m->exec);
        m->exec = nullptr;
        m->have_seen = false;  // run eagerly now, capture again on the next repeat
    }
    // A repeat of the previous eager call (whose run did every lazy set-up) is
    // captured; graphs need a stream of the caller's own that is not capturing.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const bool capturable = st != nullptr && st != cudaStreamPerThread &&
                            cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone;
    if (capturable && m->have_seen && m->seen == key && !(m->have_nocap && m->nocap_key == key)) {
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;
        lora_status s = from_cuda(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
        if (s == LORA_OK) {
            m->self_capture = true;
            s = host_step(x_host, y_host, offsets_host, ids_host, alpha_host, T, P, pool, ranks_dev, m, stream, al);
            m->self_capture = false;
            const cudaError_t e2 = cudaStreamEndCapture(st, &graph);
            if (s == LORA_OK && e2 == cudaSuccess && graph)
                s = from_cuda(cudaGraphInstantiate(&exec, graph, 0));
            else if (s == LORA_OK)
                s = from_cuda(e2 != cudaSuccess ? e2 : cudaErrorStreamCaptureInvalidated);
            if (graph)
                cudaGraphDestroy(graph);
        }
        if (s == LORA_OK && exec) {
            if (m->exec)
                cudaGraphExecDestroy(m->exec);
            m->exec = exec;
            m->graph_key = key;
            m->graph_alias = al;
            return from_cuda(cudaGraphLaunch(exec, st));
        }
        cudaGetLastError();  // capture failed: this key runs eagerly from now on
        m->nocap_key = key;
        m->have_nocap = true;
    }
    m->seen = key;
    m->have_seen = true;
    return host_step(x_host, y_host, offsets_host, ids_host, alpha_host, T, P, pool, ranks_dev, m, stream, al);
}

lora_status lora_mapping_status(const lora_mapping *m, lora_stream_t stream, int *device_error)
{
    if (!m || !device_error)
        return LORA_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&v, m->dev.hdr + HDR_STATUS, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    *device_error = v;
    return from_cuda(e);
}

lora_status lora_mapping_export(const lora_mapping *m, lora_stream_t stream, int32_t *tok, int32_t *adapter,
                                float *alpha, int32_t *src, int32_t *pos, int32_t *seg_adapter, int32_t *seg_start,
                                int32_t *counts)
{
    if (!m)
        return LORA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = m->built ? sort_mapping(m, st) : cudaSuccess;
    int32_t hdr[HDR_WORDS];
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(hdr, m->dev.hdr, sizeof hdr, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return from_cuda(e);
    const size_t U = (size_t)hdr[HDR_U], Pv = (size_t)hdr[HDR_PVALID], P = (size_t)(m->built ? m->P : 0);
    struct {
        void *dst;
        const void *src;
        size_t bytes;
    } cp[] = {
        {tok, m->dev.tok, Pv * 4},          {adapter, m->dev.adapter, Pv * 4}, {alpha, m->dev.alpha, Pv * 4},
        {src, m->dev.src, Pv * 4},          {pos, m->dev.pos, P * 4},          {seg_adapter, m->dev.seg_adapter, U * 4},
        {seg_start, m->dev.seg_start, (U + 1) * 4},
    };
    for (auto &c : cp)
        if (c.dst && c.bytes && e == cudaSuccess)
            e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (counts) {
        counts[0] = hdr[HDR_U];
        counts[1] = hdr[HDR_PVALID];
        counts[2] = hdr[HDR_STATUS];
    }
    return from_cuda(e);
}

lora_status lora_mapping_destroy(lora_mapping *m)
{
    if (!m)
        return LORA_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_mapping(m);
    return from_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation variant
namespace {

// The fixed scratch of lora_delta_apply_noalloc (one per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[LORA_NOALLOC_SCRATCH_BYTES];

struct NoallocLayout {
    size_t tok, adapter, src, pos, alpha, seg_adapter, seg_start, tile, tile_tok, hdr, mtile, toff, pc, calpha,
        zcnt, z, ghist;
    size_t total;
};

NoallocLayout noalloc_layout(int T, int P, int capacity, int r_max)
{
    NoallocLayout L;
    size_t off = 0;
    auto take = [&off](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~static_cast<size_t>(255);
        return o;
    };
    const size_t p = P > 0 ? (size_t)P : 1;
    const size_t tiles = (size_t)(P > 0 ? shrink_tile_bound(P, capacity) : 1);
    const size_t mtiles = (size_t)(P > 0 ? mma_tile_bound(P, capacity) : 1);
    L.tok = take(4 * p);
    L.adapter = take(4 * p);
    L.src = take(4 * p);
    L.pos = take(4 * p);
    L.alpha = take(4 * p);
    L.seg_adapter = take(4 * (size_t)capacity);
    L.seg_start = take(4 * ((size_t)capacity + 1));
    L.tile = take(16 * tiles);
    L.tile_tok = take(4 * tiles * SHRINK_TT);
    L.hdr = take(4 * (size_t)HDR_WORDS);
    L.mtile = take(16 * mtiles);
    L.toff = take(4 * ((size_t)T + 1));
    L.pc = take(8 * p);
    L.calpha = take(4 * p);
    L.zcnt = take(4 * p);
    L.z = take(4 * p * (size_t)z_stride(r_max));
    L.ghist = take(4 * (size_t)map_global_hist_words(capacity));
    L.total = off;
    return L;
}

// Device address of the scratch on the current device, looked up once per
// device (under a lock: concurrent first calls from several host threads
// see either no entry or the finished one).
unsigned char *noalloc_base()
{
    constexpr int MAX_DEVICES = 64;
    static unsigned char *base[MAX_DEVICES] = {};
    static std::mutex lock;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return nullptr;
    std::lock_guard<std::mutex> g(lock);
    if (!base[dev]) {
        unsigned char *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        base[dev] = ptr;
    }
    return base[dev];
}

}  // namespace

extern "C" lora_status lora_delta_apply_noalloc(const void *x_dev, void *y_dev, const lora_pool *pool,
                                                const int32_t *ranks_dev, const int32_t *offsets_dev,
                                                const int32_t *ids_dev, const float *alpha_dev, int T, int P,
                                                int32_t *status_dev, lora_stream_t stream)
{
    if (!x_dev || !y_dev || !pool || !offsets_dev || x_dev == y_dev || T < 0 || P < 0)
        return LORA_ERR_INVALID_ARG;
    if (P > 0 && (!ids_dev || !alpha_dev))
        return LORA_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(y_dev))
        return LORA_ERR_INVALID_ARG;
    if (T > LORA_MAX_TOKENS || P > LORA_MAX_PAIRS)
        return LORA_ERR_NOT_SUPPORTED;
    const NoallocLayout L = noalloc_layout(T, P, pool->capacity, pool->r_max);
    if (L.total > (size_t)LORA_NOALLOC_SCRATCH_BYTES)
        return LORA_ERR_NOT_SUPPORTED;  // batch too large for the fixed scratch
    unsigned char *base = noalloc_base();
    if (!base)
        return LORA_ERR_CUDA;
    MapDev d = {};
    d.tok = reinterpret_cast<int32_t *>(base + L.tok);
    d.adapter = reinterpret_cast<int32_t *>(base + L.adapter);
    d.src = reinterpret_cast<int32_t *>(base + L.src);
    d.pos = reinterpret_cast<int32_t *>(base + L.pos);
    d.alpha = reinterpret_cast<float *>(base + L.alpha);
    d.seg_adapter = reinterpret_cast<int32_t *>(base + L.seg_adapter);
    d.seg_start = reinterpret_cast<int32_t *>(base + L.seg_start);
    d.tile = reinterpret_cast<int4 *>(base + L.tile);
    d.tile_tok = reinterpret_cast<int32_t *>(base + L.tile_tok);
    d.hdr = reinterpret_cast<int32_t *>(base + L.hdr);
    d.mtile = reinterpret_cast<int4 *>(base + L.mtile);
    d.toff = reinterpret_cast<int32_t *>(base + L.toff);
    d.pc = reinterpret_cast<int2 *>(base + L.pc);
    d.calpha = reinterpret_cast<float *>(base + L.calpha);
    d.zcnt = reinterpret_cast<int32_t *>(base + L.zcnt);
    d.z = reinterpret_cast<float *>(base + L.z);
    d.ghist = map_global_hist_words(pool->capacity) > 0 ? reinterpret_cast<int32_t *>(base + L.ghist) : nullptr;
    d.partial = nullptr;  // used by the fused kernel only
    d.partial_ctas = 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(d.hdr, 0, HDR_WORDS * sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = launch_build_mapping(d, offsets_dev, ids_dev, alpha_dev, T, P, pool->capacity, P, st);
    if (e == cudaSuccess && T > 0 && P > 0) {
        const PoolDev pd = pool_dev(pool);
        e = launch_shrink(static_cast<const __nv_bfloat16 *>(x_dev), pd, ranks_dev, d, P, sm_count(), st);
        if (e == cudaSuccess)
            e = launch_expand(static_cast<__nv_bfloat16 *>(y_dev), pd, ranks_dev, d, T,
                              choose_expand_plan(T, pool->d_out), /*pdl=*/true, st);
    }
    if (e == cudaSuccess && status_dev)
        e = cudaMemcpyAsync(status_dev, d.hdr + HDR_STATUS, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    return from_cuda(e);
}
