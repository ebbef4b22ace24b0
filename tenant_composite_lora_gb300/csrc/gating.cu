// MoE-LoRA gating on the device: the step that produces the per-token pair
// lists the mapping consumes (DyMerge-LoRA page, MoE-LoRA scenario and code
// release notes, paper Sec. 5.3 and Appendix A: each token weights its
// request's adapters by a gate; candidate lists are padded and masked, the
// top-k kept and their softmax weights renormalised).
//
//  * k_gate_logits: logits[t][e] = x_t . Wg[req_t][e] -- a warp per
//    (token, candidate), 16-byte loads, fp32 accumulation, shuffle reduce.
//  * k_gate_topk: a thread per token; the top_k valid candidates by logit
//    (largest first, equal logits by the lower candidate index) and
//    alpha_i = exp(l_i - l_max) / sum_kept exp(l_j - l_max), written as the
//    token's top_k CSR pairs (offsets[t] = t * top_k); a token short of
//    valid candidates repeats its best one with alpha 0, a token with none
//    emits id -1 (left out by the mapping).
#include "internal.h"
#include "ptx.cuh"

namespace tcl {

namespace {

constexpr int GT_MAX_E = 64;
constexpr int GT_MAX_K = 8;

__global__ void k_gate_logits(const __nv_bfloat16 *x, const __nv_bfloat16 *wg, const int32_t *req, int T, int E,
                              int d_in, float *logits)
{
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= (long long)T * E)
        return;
    const int t = (int)(warp / E), e = (int)(warp % E);
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (size_t)t * d_in);
    const uint4 *wr = reinterpret_cast<const uint4 *>(wg + ((size_t)req[t] * E + e) * d_in);
    float acc = 0.f;
    for (int i = lane; i < d_in / 8; i += 32) {
        const uint4 a = xr[i], b = __ldg(&wr[i]);
        acc = fmaf(bf16lo(a.x), bf16lo(b.x), acc);
        acc = fmaf(bf16hi(a.x), bf16hi(b.x), acc);
        acc = fmaf(bf16lo(a.y), bf16lo(b.y), acc);
        acc = fmaf(bf16hi(a.y), bf16hi(b.y), acc);
        acc = fmaf(bf16lo(a.z), bf16lo(b.z), acc);
        acc = fmaf(bf16hi(a.z), bf16hi(b.z), acc);
        acc = fmaf(bf16lo(a.w), bf16lo(b.w), acc);
        acc = fmaf(bf16hi(a.w), bf16hi(b.w), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0)
        logits[(size_t)t * E + e] = acc;
}

__global__ void k_gate_topk(const float *logits, const int32_t *cand, int T, int E, int top_k, int32_t *offsets,
                            int32_t *ids, float *alpha)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t == 0)
        offsets[0] = 0;
    if (t >= T)
        return;
    offsets[t + 1] = (t + 1) * top_k;
    const float *l = logits + (size_t)t * E;
    const int32_t *c = cand + (size_t)t * E;
    unsigned long long taken = 0ull;  // E <= 64
    int sel[GT_MAX_K];
    int n = 0;
    for (int i = 0; i < top_k; ++i) {
        int best = -1;
        float bl = 0.f;
        for (int e = 0; e < E; ++e) {
            if (c[e] < 0 || ((taken >> e) & 1ull))
                continue;
            const float v = l[e];
            if (best < 0 || v > bl) {  // strict: the lower index keeps a tie
                best = e;
                bl = v;
            }
        }
        if (best < 0)
            break;
        taken |= 1ull << best;
        sel[n++] = best;
    }
    int32_t *id = ids + (size_t)t * top_k;
    float *al = alpha + (size_t)t * top_k;
    if (n == 0) {
        for (int i = 0; i < top_k; ++i) {
            id[i] = -1;
            al[i] = 0.f;
        }
        return;
    }
    const float mx = l[sel[0]];
    float w[GT_MAX_K], den = 0.f;
    for (int i = 0; i < n; ++i) {
        w[i] = expf(l[sel[i]] - mx);
        den += w[i];
    }
    for (int i = 0; i < top_k; ++i) {
        if (i < n) {
            id[i] = c[sel[i]];
            al[i] = w[i] / den;
        } else {
            id[i] = c[sel[0]];
            al[i] = 0.f;
        }
    }
}

}  // namespace

}  // namespace tcl

using namespace tcl;

extern "C" {

lora_status lora_gate_logits(const void *x_dev, const void *wg_dev, const int32_t *req_dev, int T, int E, int d_in,
                             float *logits_dev, lora_stream_t stream)
{
    if (!x_dev || !wg_dev || !req_dev || !logits_dev || T < 0 || E < 1 || d_in < 8 || d_in % 8)
        return LORA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(wg_dev)) & 15u)
        return LORA_ERR_INVALID_ARG;
    if (T == 0)
        return LORA_OK;
    const long long threads = (long long)T * E * 32;
    k_gate_logits<<<(unsigned)((threads + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(x_dev), static_cast<const __nv_bfloat16 *>(wg_dev), req_dev, T, E, d_in,
        logits_dev);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

lora_status lora_gate_topk(const float *logits_dev, const int32_t *cand_dev, int T, int E, int top_k,
                           int32_t *offsets_dev, int32_t *ids_dev, float *alpha_dev, lora_stream_t stream)
{
    if (!logits_dev || !cand_dev || !offsets_dev || !ids_dev || !alpha_dev || T < 0)
        return LORA_ERR_INVALID_ARG;
    if (E < 1 || E > GT_MAX_E || top_k < 1 || top_k > GT_MAX_K || top_k > E)
        return LORA_ERR_NOT_SUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // at least one thread: it writes offsets[0] even for an empty batch
    k_gate_topk<<<(T + 256) / 256, 256, 0, st>>>(logits_dev, cand_dev, T, E, top_k, offsets_dev, ids_dev, alpha_dev);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // extern "C"
