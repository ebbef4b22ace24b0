// The pages' kernel ablation, reproduced on this device: three ways of
// computing the same composite delta that the fused path replaces
// (DyMerge-LoRA page, "How far to trust it": the fused multi-LoRA kernel
// against Copy+SGMV and a naive for-loop, paper Sec. 5.4-5.5, Figs. 14 and
// 16; pre-merging the composite weight, Figs. 3-4).  They are baselines to
// time against, written plainly: no fusion across their steps.
//
//  * Naive loop: the host reads the batch's adapter segments back and, for
//    each adapter, launches a shrink over that adapter's pairs and an expand
//    that adds their rows into an fp32 copy of y; a last launch rounds y.
//  * Copy + SGMV: gather x into adapter-sorted order (one row per pair),
//    segment shrink and expand over the gathered rows into a per-pair fp32
//    output, then add each token's pair rows back into y (one rounding).
//  * Pre-merge: per token, the merged weight dW_t = sum alpha A[:, :k] B[:k, :]
//    (fp32, d_in x d_out), then y_t += x_t dW_t.
//
// Every variant accumulates in fp32 and rounds y once.
#include <cstdlib>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int AB_THREADS = 256;

__device__ __forceinline__ float ab_dot8(uint4 a, uint4 b, float acc)
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

// z[q][j] = alpha_q * sum_d xrow_q[d] A_a[d][j] for j < k, a warp per (q, j).
// xrow_q is x[tok[q]] (naive) or xs[q] (the gathered copy).  Pairs [q0, q1).
__global__ void k_ab_shrink(const __nv_bfloat16 *x, const __nv_bfloat16 *xs, PoolDev pool, const int32_t *ranks,
                            MapDev m, int q0, int q1, float *z, int zs)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int q = q0 + warp / pool.r_max, j = warp % pool.r_max;
    if (q >= q1)
        return;
    const int a = m.adapter[q];
    const int k = effective_rank(pool, ranks, a);
    if (j >= (k > 0 ? k : 0))
        return;
    const int nv = pool.d_in / 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(xs ? xs + (size_t)q * pool.d_in : x + (size_t)m.tok[q] * pool.d_in);
    const uint4 *ar = reinterpret_cast<const uint4 *>(pool.At + ((size_t)a * pool.r_max + j) * pool.d_in);
    float acc = 0.f;
    for (int i = lane; i < nv; i += 32)
        acc = ab_dot8(ar[i], xr[i], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        z[(size_t)q * zs + j] = m.alpha[q] * acc;
}

// Naive expand of one adapter's pairs: yacc[tok_q][c] += sum_j z[q][j] B[j][c].
// A thread per (pair, column); pairs of one adapter belong to different
// tokens unless a token lists the adapter twice, so the add is atomic.
__global__ void k_ab_naive_expand(PoolDev pool, const int32_t *ranks, MapDev m, int q0, int q1, const float *z, int zs,
                                  float *yacc)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int q = q0 + (int)(i / pool.d_out), c = (int)(i % pool.d_out);
    if (q >= q1)
        return;
    const int a = m.adapter[q];
    const int k = effective_rank(pool, ranks, a);
    float acc = 0.f;
    for (int j = 0; j < k; ++j)
        acc = fmaf(z[(size_t)q * zs + j], __bfloat162float(pool.B[((size_t)a * pool.r_max + j) * pool.d_out + c]), acc);
    atomicAdd(yacc + (size_t)m.tok[q] * pool.d_out + c, acc);
}

__global__ void k_ab_to_f32(const __nv_bfloat16 *y, float *yacc, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        yacc[i] = __bfloat162float(y[i]);
}

__global__ void k_ab_to_bf16(const float *yacc, __nv_bfloat16 *y, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        y[i] = __float2bfloat16_rn(yacc[i]);
}

// Copy: xs[q] = x[tok[q]] (16-byte vectors).
__global__ void k_ab_gather(const __nv_bfloat16 *x, MapDev m, int pvalid, int d_in, __nv_bfloat16 *xs)
{
    const int nv = d_in / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)pvalid * nv;
         i += (long long)gridDim.x * blockDim.x) {
        const int q = (int)(i / nv), v = (int)(i % nv);
        reinterpret_cast<uint4 *>(xs + (size_t)q * d_in)[v] =
            reinterpret_cast<const uint4 *>(x + (size_t)m.tok[q] * d_in)[v];
    }
}

// SGMV expand: ys[q][c] = sum_j z[q][j] B_a[j][c] (fp32, one row per pair).
__global__ void k_ab_sgmv_expand(PoolDev pool, const int32_t *ranks, MapDev m, int pvalid, const float *z, int zs,
                                 float *ys)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)pvalid * pool.d_out;
         i += (long long)gridDim.x * blockDim.x) {
        const int q = (int)(i / pool.d_out), c = (int)(i % pool.d_out);
        const int a = m.adapter[q];
        const int k = effective_rank(pool, ranks, a);
        float acc = 0.f;
        for (int j = 0; j < k; ++j)
            acc = fmaf(z[(size_t)q * zs + j], __bfloat162float(pool.B[((size_t)a * pool.r_max + j) * pool.d_out + c]),
                       acc);
        ys[i] = acc;
    }
}

// Copy back: y[t][c] = bf16(y[t][c] + sum over t's pairs (CSR order) of ys[pos][c]).
__global__ void k_ab_scatter(__nv_bfloat16 *y, MapDev m, int T, int d_out, const float *ys)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)T * d_out;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / d_out), c = (int)(i % d_out);
        float acc = __bfloat162float(y[i]);
        for (int p = m.toff[t]; p < m.toff[t + 1]; ++p) {
            const int q = m.pos[p];
            if (q >= 0)
                acc += ys[(size_t)q * d_out + c];
        }
        y[i] = __float2bfloat16_rn(acc);
    }
}

// Pre-merge: dW_t[i][c] = sum over t's pairs of alpha sum_{j<k} A[i][j] B[j][c]
// (fp32).  A 16 x 256 tile of dW_t per CTA, a thread per column
// vector of 16 rows.
__global__ void k_ab_merge(PoolDev pool, const int32_t *ranks, MapDev m, int T, float *dw)
{
    const int t = blockIdx.z;
    const int i0 = blockIdx.y * 16, c = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T || c >= pool.d_out)
        return;
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        acc[r] = 0.f;
    for (int p = m.toff[t]; p < m.toff[t + 1]; ++p) {
        const int2 v = m.pc[p];  // {token, adapter}
        if (v.y < 0)
            continue;
        const int k = effective_rank(pool, ranks, v.y);
        const float al = m.calpha[p];
        for (int j = 0; j < k; ++j) {
            const float b = al * __bfloat162float(pool.B[((size_t)v.y * pool.r_max + j) * pool.d_out + c]);
            const __nv_bfloat16 *ac = pool.At + ((size_t)v.y * pool.r_max + j) * pool.d_in + i0;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (i0 + r < pool.d_in)
                    acc[r] = fmaf(__bfloat162float(ac[r]), b, acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 16; ++r)
        if (i0 + r < pool.d_in)
            dw[((size_t)t * pool.d_in + i0 + r) * pool.d_out + c] = acc[r];
}

// y_t[c] = bf16(y_t[c] + sum_i x_t[i] dW_t[i][c]), a thread per (t, column).
__global__ void k_ab_premerge_apply(const __nv_bfloat16 *x, __nv_bfloat16 *y, int T, int d_in, int d_out,
                                    const float *dw)
{
    const int t = blockIdx.y, c = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T || c >= d_out)
        return;
    float acc = 0.f;
    const float *w = dw + (size_t)t * d_in * d_out + c;
    const __nv_bfloat16 *xr = x + (size_t)t * d_in;
    for (int i = 0; i < d_in; ++i)
        acc = fmaf(__bfloat162float(xr[i]), w[(size_t)i * d_out], acc);
    y[(size_t)t * d_out + c] = __float2bfloat16_rn(__bfloat162float(y[(size_t)t * d_out + c]) + acc);
}

unsigned grid_for(long long n)
{
    long long g = (n + AB_THREADS - 1) / AB_THREADS;
    const long long cap = 8LL * sm_count();
    return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

size_t ablation_workspace_bytes(int variant, int T, int P, int d_in, int d_out, int r_max)
{
    const size_t zs = (size_t)z_stride(r_max);
    switch (variant) {
    case LORA_ABLATION_NAIVE:
        return round256((size_t)P * zs * 4) + round256((size_t)T * d_out * 4);
    case LORA_ABLATION_COPY_SGMV:
        return round256((size_t)P * d_in * 2) + round256((size_t)P * zs * 4) + round256((size_t)P * d_out * 4);
    case LORA_ABLATION_PREMERGE:
        return round256((size_t)T * d_in * d_out * 4);
    default:
        return 0;
    }
}

cudaError_t run_ablation(int variant, const __nv_bfloat16 *x, __nv_bfloat16 *y, const PoolDev &pool,
                         const int32_t *ranks, const MapDev &m, int T, int P, void *ws, cudaStream_t st)
{
    unsigned char *w = static_cast<unsigned char *>(ws);
    const int zs = z_stride(pool.r_max);
    if (variant == LORA_ABLATION_PREMERGE) {
        float *dw = reinterpret_cast<float *>(w);
        const dim3 mg((pool.d_out + AB_THREADS - 1) / AB_THREADS, (pool.d_in + 15) / 16, T);
        k_ab_merge<<<mg, AB_THREADS, 0, st>>>(pool, ranks, m, T, dw);
        const dim3 ag((pool.d_out + AB_THREADS - 1) / AB_THREADS, T);
        k_ab_premerge_apply<<<ag, AB_THREADS, 0, st>>>(x, y, T, pool.d_in, pool.d_out, dw);
        return cudaGetLastError();
    }
    // both other variants work on the adapter-sorted tuples; they need the
    // number of valid pairs, and the naive loop its segments, on the host:
    // read them back (this synchronises the stream)
    cudaError_t e = launch_map_sort(m, T, P, pool.capacity, st);
    if (e != cudaSuccess)
        return e;
    int32_t hdr[HDR_WORDS];
    e = cudaMemcpyAsync(hdr, m.hdr, sizeof hdr, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    const int U = hdr[HDR_U], pvalid = hdr[HDR_PVALID];
    if (pvalid <= 0)
        return cudaSuccess;
    const unsigned shrink_threads = 128;
    if (variant == LORA_ABLATION_NAIVE) {
        std::vector<int32_t> seg(U + 1);
        e = cudaMemcpyAsync(seg.data(), m.seg_start, (U + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
        if (e != cudaSuccess)
            return e;
        float *z = reinterpret_cast<float *>(w);
        float *yacc = reinterpret_cast<float *>(w + round256((size_t)P * zs * 4));
        const long long ny = (long long)T * pool.d_out;
        k_ab_to_f32<<<grid_for(ny), AB_THREADS, 0, st>>>(y, yacc, ny);
        for (int u = 0; u < U; ++u) {  // one adapter per iteration
            const int q0 = seg[u], q1 = seg[u + 1];
            const long long warps = (long long)(q1 - q0) * pool.r_max;
            k_ab_shrink<<<(unsigned)((warps * 32 + shrink_threads - 1) / shrink_threads), shrink_threads, 0, st>>>(
                x, nullptr, pool, ranks, m, q0, q1, z, zs);
            const long long n = (long long)(q1 - q0) * pool.d_out;
            k_ab_naive_expand<<<(unsigned)((n + AB_THREADS - 1) / AB_THREADS), AB_THREADS, 0, st>>>(pool, ranks, m, q0,
                                                                                                     q1, z, zs, yacc);
        }
        k_ab_to_bf16<<<grid_for(ny), AB_THREADS, 0, st>>>(yacc, y, ny);
        return cudaGetLastError();
    }
    // Copy + SGMV
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(w);
    float *z = reinterpret_cast<float *>(w + round256((size_t)P * pool.d_in * 2));
    float *ys = reinterpret_cast<float *>(w + round256((size_t)P * pool.d_in * 2) + round256((size_t)P * zs * 4));
    k_ab_gather<<<grid_for((long long)pvalid * pool.d_in / 8), AB_THREADS, 0, st>>>(x, m, pvalid, pool.d_in, xs);
    const long long warps = (long long)pvalid * pool.r_max;
    k_ab_shrink<<<(unsigned)((warps * 32 + shrink_threads - 1) / shrink_threads), shrink_threads, 0, st>>>(
        nullptr, xs, pool, ranks, m, 0, pvalid, z, zs);
    k_ab_sgmv_expand<<<grid_for((long long)pvalid * pool.d_out), AB_THREADS, 0, st>>>(pool, ranks, m, pvalid, z, zs,
                                                                                      ys);
    k_ab_scatter<<<grid_for((long long)T * pool.d_out), AB_THREADS, 0, st>>>(y, m, T, pool.d_out, ys);
    return cudaGetLastError();
}

}  // namespace tcl
