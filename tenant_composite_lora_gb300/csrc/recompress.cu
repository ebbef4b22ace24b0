// Batched LoRA recompression on the device (FlashTSQR factor construction)
// and retained-rank allocation (LoRAForge summary page, "Key contributions"
// and "Approach" (2)-(3)).
//
// For M modules of one shape, dW_m = A_m B_m (A: d_in x r, B: r x d_out, bf16):
//  1. tall-skinny QR of every A_m without forming Q: each A_m is cut into P
//     row tiles, the M P leaf QRs (Householder, fp32, shared memory) run as
//     independent CTAs, then the triangular factors are merged pairwise, one
//     launch per level, until one R_m is left (diagonal made non-negative);
//  2. H = R_m B_m streamed over column chunks, G_m = H H^T and B_m H^T;
//  3. G_m = U diag(lambda) U^T by cyclic Jacobi (parallel round-robin
//     rotations), sorted descending; sigma = sqrt(lambda); directions with
//     lambda <= LIVE_REL * lambda_0 are dead;
//  4. balanced factors F = Q U diag(sqrt sigma) and T = diag(1/sqrt sigma) U^T H,
//     formed without Q as F = A M1 with M1 = B H^T U diag(sigma^-3/2) and
//     T = M2 B with M2 = diag(sigma^-1/2) U^T R: F T = A B, F^T F = T T^T =
//     diag(sigma), and the first k directions give the rank-k truncated SVD.
// The rank policies (uniform retention, spectral budget) run on the host.
#include <algorithm>
#include <cmath>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int RC_THREADS = 256;
constexpr int RC_MAX_R = 64;
constexpr float RC_LIVE_REL = 1e-6f;  // on lambda = sigma^2
constexpr int RC_SWEEPS = 16;

__device__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        s += red[w];
    return s;
}

// Householder QR of a column-major h x r tile (col c at t + c * ld), h >= r;
// the upper triangle of the first r rows becomes R.  All threads call it.
__device__ void householder_qr(float *t, int ld, int h, int r, float *red, float *wv)
{
    for (int j = 0; j < r; ++j) {
        float *x = t + j * ld;
        float s = 0.f;
        for (int i = j + threadIdx.x; i < h; i += blockDim.x)
            s += x[i] * x[i];
        s = block_sum(s, red);
        const float alpha = x[j], norm = sqrtf(s);
        __syncthreads();
        if (norm == 0.f)
            continue;  // a zero column: R[j][j] = 0, nothing to reflect
        const float beta = alpha >= 0.f ? -norm : norm;
        const float vj = alpha - beta;
        const float vv = s - alpha * alpha + vj * vj;  // v . v
        // w_c = v . col_c over rows >= j, a warp per column
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int c = j + 1 + warp; c < r; c += blockDim.x >> 5) {
            const float *y = t + c * ld;
            float d = lane == 0 ? vj * y[j] : 0.f;
            for (int i = j + 1 + lane; i < h; i += 32)
                d += x[i] * y[i];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                d += __shfl_xor_sync(0xffffffffu, d, off);
            if (lane == 0)
                wv[c] = d;
        }
        __syncthreads();
        const float tau = 2.f / vv;
        const int nc = r - j - 1, nr = h - j;
        for (int e = threadIdx.x; e < nc * nr; e += blockDim.x) {
            const int c = j + 1 + e / nr, i = j + e % nr;
            const float vi = i == j ? vj : x[i];
            t[c * ld + i] -= tau * wv[c] * vi;
        }
        __syncthreads();
        if (threadIdx.x == 0)
            x[j] = beta;
        __syncthreads();
    }
}

// Leaf QRs: CTA (p, m) factors rows [p h, (p + 1) h) of A_m (bf16 row-major
// d_in x r) and writes its R (row-major r x r, zeros below the diagonal).
__global__ void __launch_bounds__(RC_THREADS) k_tsqr_leaf(const __nv_bfloat16 *A, int d_in, int r, int P, float *rbuf)
{
    extern __shared__ float sm[];
    __shared__ float red[RC_THREADS / 32], wv[RC_MAX_R];
    const int p = blockIdx.x, m = blockIdx.y, h = d_in / P;
    const int ld = h + 1;
    const __nv_bfloat16 *a = A + ((size_t)m * d_in + (size_t)p * h) * r;
    for (int e = threadIdx.x; e < h * r; e += blockDim.x)
        sm[(e % r) * ld + e / r] = __bfloat162float(a[e]);
    __syncthreads();
    householder_qr(sm, ld, h, r, red, wv);
    float *out = rbuf + ((size_t)m * P + p) * r * r;
    for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
        const int i = e / r, c = e % r;
        out[e] = c >= i ? sm[c * ld + i] : 0.f;
    }
}

// One merge level: R at p and p + stride (p a multiple of 2 stride) stacked
// (2r x r) and factored; the result replaces R at p.  The last level makes
// the diagonal non-negative.
__global__ void __launch_bounds__(RC_THREADS) k_tsqr_merge(int r, int P, int stride, int last, float *rbuf)
{
    extern __shared__ float sm[];
    __shared__ float red[RC_THREADS / 32], wv[RC_MAX_R];
    const int p = blockIdx.x * 2 * stride, m = blockIdx.y;
    const int ld = 2 * r + 1;
    float *r0 = rbuf + ((size_t)m * P + p) * r * r, *r1 = rbuf + ((size_t)m * P + p + stride) * r * r;
    for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
        const int i = e / r, c = e % r;
        sm[c * ld + i] = r0[e];
        sm[c * ld + r + i] = r1[e];
    }
    __syncthreads();
    householder_qr(sm, ld, 2 * r, r, red, wv);
    for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
        const int i = e / r, c = e % r;
        float v = c >= i ? sm[c * ld + i] : 0.f;
        if (last && sm[i * ld + i] < 0.f)
            v = -v;
        r0[e] = v;
    }
}

// Per module: H = R B streamed over column chunks of B (H is never stored
// whole), G = H H^T and Y = B H^T accumulated chunk by chunk, then the
// Jacobi eigen-decomposition of G, sigma, M1 = Y U diag(sigma^-3/2) (= S R^T
// U diag(sigma^-3/2) with S = B B^T, formed without S: R S R^T from a
// separately rounded S loses the cancellation between A's and B's mixing)
// and M2 = diag(sigma^-1/2) U^T R.  Shared memory: 5 r x r and 2 r x RC_CW
// fp32 matrices.
constexpr int RC_CW = 64;  // columns of B per chunk

__global__ void __launch_bounds__(RC_THREADS) k_spectrum(const __nv_bfloat16 *Bm, int d_out, int r, int P,
                                                         const float *rbuf, float *sigma_out, float *m1_out,
                                                         float *m2_out)
{
    extern __shared__ float sm[];
    __shared__ float lam[RC_MAX_R], cs[RC_MAX_R / 2][2];
    __shared__ int perm[RC_MAX_R], pairs[RC_MAX_R / 2][2];
    __shared__ float red[RC_THREADS / 32];
    const int m = blockIdx.x, rr = r * r;
    float *R = sm, *Y = sm + rr, *G = sm + 2 * rr, *U = sm + 3 * rr, *W = sm + 4 * rr;
    float *Bc = sm + 5 * rr, *Hc = Bc + r * RC_CW;
    const float *rin = rbuf + (size_t)m * P * rr;  // the merged R sits at tile 0
    for (int e = threadIdx.x; e < rr; e += blockDim.x) {
        R[e] = rin[e];
        G[e] = 0.f;
        Y[e] = 0.f;
        U[e] = (e / r == e % r) ? 1.f : 0.f;
    }
    const __nv_bfloat16 *B = Bm + (size_t)m * r * d_out;
    for (int c0 = 0; c0 < d_out; c0 += RC_CW) {
        const int cw = min(RC_CW, d_out - c0);
        __syncthreads();  // the previous chunk is consumed (and R, G, Y initialised)
        for (int e = threadIdx.x; e < r * RC_CW; e += blockDim.x) {
            const int i = e / RC_CW, cc = e % RC_CW;
            Bc[e] = cc < cw ? __bfloat162float(B[(size_t)i * d_out + c0 + cc]) : 0.f;
        }
        __syncthreads();
        // Hc = R Bc (R upper triangular)
        for (int e = threadIdx.x; e < r * RC_CW; e += blockDim.x) {
            const int i = e / RC_CW, cc = e % RC_CW;
            float h = 0.f;
            for (int q = i; q < r; ++q)
                h = fmaf(R[i * r + q], Bc[q * RC_CW + cc], h);
            Hc[e] = h;
        }
        __syncthreads();
        // G += Hc Hc^T, Y += Bc Hc^T
        for (int e = threadIdx.x; e < rr; e += blockDim.x) {
            const int i = e / r, j = e % r;
            float g = 0.f, y = 0.f;
            for (int cc = 0; cc < RC_CW; ++cc) {
                const float hj = Hc[j * RC_CW + cc];
                g = fmaf(Hc[i * RC_CW + cc], hj, g);
                y = fmaf(Bc[i * RC_CW + cc], hj, y);
            }
            G[e] += g;
            Y[e] += y;
        }
    }
    __syncthreads();
    // symmetrise (the two triangles of R S R^T are rounded separately)
    for (int e = threadIdx.x; e < rr; e += blockDim.x) {
        const int i = e / r, j = e % r;
        if (j > i) {
            const float v = 0.5f * (G[i * r + j] + G[j * r + i]);
            G[i * r + j] = v;
            G[j * r + i] = v;
        }
    }
    __syncthreads();
    // cyclic Jacobi, round-robin: n = r rounded up to even players, n - 1
    // rounds of n / 2 disjoint pairs per sweep (a dummy player when r is odd)
    const int n = (r + 1) & ~1;
    for (int sweep = 0; sweep < RC_SWEEPS; ++sweep) {
        float off = 0.f, tot = 0.f;
        for (int e = threadIdx.x; e < rr; e += blockDim.x) {
            const float g = G[e] * G[e];
            tot += g;
            if (e / r != e % r)
                off += g;
        }
        off = block_sum(off, red);
        tot = block_sum(tot, red);
        if (off <= 1e-12f * tot || tot == 0.f)  // off-diagonal at fp32's noise floor
            break;
        for (int round = 0; round < n - 1; ++round) {
            if (threadIdx.x < n / 2) {
                const int k = threadIdx.x;
                // player positions: 0 fixed, others rotate
                auto player = [&](int pos) { return pos == 0 ? 0 : 1 + (pos - 1 + round) % (n - 1); };
                int a = player(k), b = player(n - 1 - k);
                if (a > b) {
                    const int tmp = a;
                    a = b;
                    b = tmp;
                }
                pairs[k][0] = a;
                pairs[k][1] = b;
                float c = 1.f, s = 0.f;
                if (b < r) {
                    const float app = G[a * r + a], aqq = G[b * r + b], apq = G[a * r + b];
                    if (fabsf(apq) > 1e-30f) {
                        const float tau = (aqq - app) / (2.f * apq);
                        const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
                        // correctly rounded square root and division: c^2 + s^2 = 1 to
                        // an ulp, so thousands of rotations keep G's norm
                        c = 1.f / sqrtf(1.f + t * t);
                        s = t * c;
                    }
                }
                cs[k][0] = c;
                cs[k][1] = s;
            }
            __syncthreads();
            // columns: G <- G J, U <- U J (each pair rotates its two columns)
            for (int e = threadIdx.x; e < (n / 2) * r; e += blockDim.x) {
                const int k = e / r, i = e % r;
                const int a = pairs[k][0], b = pairs[k][1];
                if (b >= r)
                    continue;
                const float c = cs[k][0], s = cs[k][1];
                const float ga = G[i * r + a], gb = G[i * r + b];
                G[i * r + a] = c * ga - s * gb;
                G[i * r + b] = s * ga + c * gb;
                const float ua = U[i * r + a], ub = U[i * r + b];
                U[i * r + a] = c * ua - s * ub;
                U[i * r + b] = s * ua + c * ub;
            }
            __syncthreads();
            // rows: G <- J^T G
            for (int e = threadIdx.x; e < (n / 2) * r; e += blockDim.x) {
                const int k = e / r, j = e % r;
                const int a = pairs[k][0], b = pairs[k][1];
                if (b >= r)
                    continue;
                const float c = cs[k][0], s = cs[k][1];
                const float ga = G[a * r + j], gb = G[b * r + j];
                G[a * r + j] = c * ga - s * gb;
                G[b * r + j] = s * ga + c * gb;
            }
            __syncthreads();
        }
    }
    // sort descending (rank of each eigenvalue; equal values by index)
    if (threadIdx.x < r) {
        const int j = threadIdx.x;
        const float v = G[j * r + j];
        int rank = 0;
        for (int i = 0; i < r; ++i) {
            const float w = G[i * r + i];
            rank += (w > v) || (w == v && i < j);
        }
        perm[rank] = j;
    }
    __syncthreads();
    if (threadIdx.x < r)
        lam[threadIdx.x] = fmaxf(G[perm[threadIdx.x] * r + perm[threadIdx.x]], 0.f);
    __syncthreads();
    const float lam0 = lam[0];
    // W = U sorted (columns), sigma
    for (int e = threadIdx.x; e < rr; e += blockDim.x) {
        const int i = e / r, j = e % r;
        W[e] = U[i * r + perm[j]];
    }
    __syncthreads();
    if (threadIdx.x < r) {
        const int j = threadIdx.x;
        const bool live = lam[j] > RC_LIVE_REL * lam0 && lam0 > 0.f;
        sigma_out[(size_t)m * r + j] = live ? sqrtf(lam[j]) : 0.f;
    }
    // M1 = Y W diag(sigma^-3/2) (Y = B H^T = S R^T), M2 = diag(sigma^-1/2) W^T R
    float *m1 = m1_out + (size_t)m * rr, *m2 = m2_out + (size_t)m * rr;
    for (int e = threadIdx.x; e < rr; e += blockDim.x) {
        const int i = e / r, j = e % r;
        const bool lj = lam[j] > RC_LIVE_REL * lam0 && lam0 > 0.f;
        const bool li = lam[i] > RC_LIVE_REL * lam0 && lam0 > 0.f;
        float s1 = 0.f, s2 = 0.f;
        for (int q = 0; q < r; ++q) {
            s1 = fmaf(Y[i * r + q], W[q * r + j], s1);
            s2 = fmaf(W[q * r + i], R[q * r + j], s2);
        }
        const float sj = sqrtf(lam[j]), si = sqrtf(lam[i]);
        m1[e] = lj ? s1 / (sj * sqrtf(sj)) : 0.f;
        m2[e] = li ? s2 / sqrtf(si) : 0.f;
    }
}

// F = A M1: CTA (row block of 64, m), a thread per (row, column).
__global__ void __launch_bounds__(RC_THREADS) k_factor_f(const __nv_bfloat16 *A, int d_in, int r, const float *m1,
                                                         float *F)
{
    __shared__ float mm[RC_MAX_R * RC_MAX_R];
    const int m = blockIdx.y, row0 = blockIdx.x * 64;
    for (int e = threadIdx.x; e < r * r; e += blockDim.x)
        mm[e] = m1[(size_t)m * r * r + e];
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * r; e += blockDim.x) {
        const int i = row0 + e / r, j = e % r;
        if (i >= d_in)
            continue;
        const __nv_bfloat16 *a = A + ((size_t)m * d_in + i) * r;
        float s = 0.f;
        for (int q = 0; q < r; ++q)
            s = fmaf(__bfloat162float(a[q]), mm[q * r + j], s);
        F[((size_t)m * d_in + i) * r + j] = s;
    }
}

// T = M2 B: CTA (column block of 256, m), a thread per column.
__global__ void __launch_bounds__(RC_THREADS) k_factor_t(const __nv_bfloat16 *B, int d_out, int r, const float *m2,
                                                         float *Tout)
{
    __shared__ float mm[RC_MAX_R * RC_MAX_R];
    const int m = blockIdx.y, c = blockIdx.x * blockDim.x + threadIdx.x;
    for (int e = threadIdx.x; e < r * r; e += blockDim.x)
        mm[e] = m2[(size_t)m * r * r + e];
    __syncthreads();
    if (c >= d_out)
        return;
    const __nv_bfloat16 *b = B + (size_t)m * r * d_out + c;
    float bc[RC_MAX_R];
    for (int q = 0; q < r; ++q)
        bc[q] = __bfloat162float(b[(size_t)q * d_out]);
    for (int i = 0; i < r; ++i) {
        float s = 0.f;
        for (int q = 0; q < r; ++q)
            s = fmaf(mm[i * r + q], bc[q], s);
        Tout[((size_t)m * r + i) * d_out + c] = s;
    }
}

// Row tiles of the leaf QRs: the largest power of two P with d_in / P an
// integer of at least max(r, 128) rows (the launcher refuses tiles that do
// not fit shared memory).
int leaf_tiles(int d_in, int r)
{
    int P = 1;
    while (d_in % (2 * P) == 0 && d_in / (2 * P) >= (r > 128 ? r : 128))
        P *= 2;
    return P;
}

}  // namespace

size_t recompress_workspace_bytes(int M, int d_in, int r)
{
    const size_t rr = (size_t)r * r;
    return ((size_t)M * leaf_tiles(d_in, r) * rr + 2 * (size_t)M * rr) * sizeof(float);
}

cudaError_t launch_recompress(const __nv_bfloat16 *A, const __nv_bfloat16 *B, int M, int d_in, int d_out, int r,
                              float *F, float *Tout, float *sigma, void *ws, cudaStream_t st)
{
    const int P = leaf_tiles(d_in, r), h = d_in / P;
    if ((size_t)(h + 1) * r * 4 > 160 * 1024)
        return cudaErrorNotSupported;
    float *rbuf = static_cast<float *>(ws);
    float *m1 = rbuf + (size_t)M * P * r * r, *m2 = m1 + (size_t)M * r * r;
    static thread_local int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_tsqr_leaf, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_tsqr_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_spectrum, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (5 * RC_MAX_R * RC_MAX_R + 2 * RC_MAX_R * RC_CW) * 4);
        if (e != cudaSuccess)
            return e;
        attr_dev = dev;
    }
    k_tsqr_leaf<<<dim3(P, M), RC_THREADS, (size_t)(h + 1) * r * 4, st>>>(A, d_in, r, P, rbuf);
    for (int stride = 1; stride < P; stride *= 2)
        k_tsqr_merge<<<dim3(P / (2 * stride), M), RC_THREADS, (size_t)(2 * r + 1) * r * 4, st>>>(
            r, P, stride, 2 * stride >= P ? 1 : 0, rbuf);
    // (with a single tile the leaf's R keeps Householder's diagonal signs:
    // G = R S R^T becomes D G D for a sign matrix D, U becomes D U, and M1 and
    // M2 -- hence F and T -- do not change)
    k_spectrum<<<M, RC_THREADS, ((size_t)5 * r * r + 2 * (size_t)r * RC_CW) * 4, st>>>(B, d_out, r, P, rbuf, sigma, m1,
                                                                                     m2);
    k_factor_f<<<dim3((d_in + 63) / 64, M), RC_THREADS, 0, st>>>(A, d_in, r, m1, F);
    k_factor_t<<<dim3((d_out + RC_THREADS - 1) / RC_THREADS, M), RC_THREADS, 0, st>>>(B, d_out, r, m2, Tout);
    return cudaGetLastError();
}

// LoRAForge-U and -S (host): see lora.h.
int rank_allocate(const float *sigma, int M, int r_stride, const int32_t *rank, const int32_t *cost, int policy,
                  int d, int floor_k, int32_t *k_out)
{
    std::vector<int> live(M), uni(M);
    long long budget = 0;
    for (int m = 0; m < M; ++m) {
        int n = 0;
        for (int j = 0; j < r_stride; ++j)
            n += sigma[(size_t)m * r_stride + j] > 0.f;
        live[m] = n;
        const int u = std::max(1, rank[m] / d);
        uni[m] = std::min(u, n);
        budget += (long long)uni[m] * cost[m];
    }
    if (policy == LORA_RANK_UNIFORM) {
        for (int m = 0; m < M; ++m)
            k_out[m] = uni[m];
        return 0;
    }
    long long spent = 0;
    for (int m = 0; m < M; ++m) {
        k_out[m] = std::min(floor_k, live[m]);
        spent += (long long)k_out[m] * cost[m];
    }
    struct Cand {
        double eta;
        int m, j;
    };
    std::vector<Cand> cand;
    for (int m = 0; m < M; ++m)
        for (int j = k_out[m]; j < live[m]; ++j) {
            const double s = sigma[(size_t)m * r_stride + j];
            cand.push_back({s * s / cost[m], m, j});
        }
    std::stable_sort(cand.begin(), cand.end(), [](const Cand &a, const Cand &b) {
        if (a.eta != b.eta)
            return a.eta > b.eta;
        if (a.m != b.m)
            return a.m < b.m;
        return a.j < b.j;
    });
    for (const Cand &c : cand)
        if (c.j == k_out[c.m] && spent + cost[c.m] <= budget) {
            ++k_out[c.m];
            spent += cost[c.m];
        }
    return 0;
}

}  // namespace tcl
