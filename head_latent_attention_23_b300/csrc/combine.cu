// Merge of split-KV partial results.
//
// Each partial is a normalised output o_s over a token range with its
// log-sum-exp lse_s.  The full result over the union of the ranges is
//   LSE = log sum_s exp(lse_s),   o = sum_s exp(lse_s - LSE) * o_s,
// which is exact because exp(lse_s) is the softmax denominator of range s.
// Empty ranges carry lse = -inf and weigh nothing.  One CTA per (sequence,
// head), threads over the latent width; HBM-bound, no tensor-core work.
#include "common.cuh"
#include "kernels.h"

namespace mla {

template <typename T, bool kPlanned>
__global__ void __launch_bounds__(128) combine_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, int n_splits,
    int batch, int heads, int DL, T* __restrict__ o_lat, float* __restrict__ lse,
    const int32_t* __restrict__ seq_lens, int cap, int W) {
    extern __shared__ int pre[];   // planned: [batch + 1]
    __shared__ float wts[1024];
    __shared__ int slots[1024];
    __shared__ int n_sl;
    __shared__ float sh_lse;
    const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;

    if (kPlanned) {
        tile_prefix(seq_lens, batch, cap, pre, nullptr);
        if (tid == 0) {
            const int64_t total = pre[batch];
            int cnt = 0;
            if (pre[b + 1] > pre[b]) {
                // workers whose tile range meets [pre[b], pre[b+1])
                int g = (int)((int64_t)pre[b] * W / total);
                while (g > 0 && plan_lo(g, total, W) > pre[b]) --g;
                while (g + 1 < W && plan_lo(g + 1, total, W) <= pre[b]) ++g;
                for (; g < W && plan_lo(g, total, W) < pre[b + 1]; ++g) {
                    if (plan_lo(g + 1, total, W) <= pre[b]) continue;
                    if (plan_lo(g, total, W) >= plan_lo(g + 1, total, W)) continue;
                    if (cnt < 1024) slots[cnt++] = g + b;
                }
            }
            n_sl = cnt;
        }
    } else {
        if (tid == 0) {
            int cnt = 0;
            for (int s = 0; s < n_splits && cnt < 1024; ++s) slots[cnt++] = s;
            n_sl = cnt;
        }
    }
    __syncthreads();
    const int ns = n_sl;
    auto lse_at = [&](int s) -> float {
        return kPlanned ? lse_part[(size_t)slots[s] * heads + h]
                        : lse_part[((size_t)slots[s] * batch + b) * heads + h];
    };
    auto o_at = [&](int s) -> const float* {
        return kPlanned ? o_part + ((size_t)slots[s] * heads + h) * DL
                        : o_part + (((size_t)slots[s] * batch + b) * heads + h) * DL;
    };
    if (tid == 0) {
        float m = -INFINITY;
        for (int s = 0; s < ns; ++s) m = fmaxf(m, lse_at(s));
        float sum = 0.f;
        for (int s = 0; s < ns; ++s) {
            float l = lse_at(s);
            float w = (l == -INFINITY) ? 0.f : expf(l - m);
            wts[s] = w;
            sum += w;
        }
        float inv = sum > 0.f ? 1.f / sum : 0.f;
        for (int s = 0; s < ns; ++s) wts[s] *= inv;
        sh_lse = sum > 0.f ? m + logf(sum) : -INFINITY;
    }
    __syncthreads();
    T* out = o_lat + ((size_t)b * heads + h) * DL;
    for (int j = tid; j < DL; j += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s) {
            float w = wts[s];
            if (w != 0.f) acc = fmaf(w, o_at(s)[j], acc);
        }
        out[j] = from_f<T>(acc);
    }
    if (lse && tid == 0) lse[(size_t)b * heads + h] = sh_lse;
}

cudaError_t launch_combine_planned(const DecodeArgs& a, int dtype, cudaStream_t st) {
    dim3 grid(a.batch, a.heads);
    size_t sm = sizeof(int) * (size_t)(a.batch + 1);
    int cap = a.max_blocks * a.block_size;
    if (dtype == MLA_DTYPE_BF16)
        combine_kernel<__nv_bfloat16, true><<<grid, 128, sm, st>>>(
            a.o_part, a.lse_part, 0, a.batch, a.heads, a.d_latent, (__nv_bfloat16*)a.o_lat,
            a.lse, a.seq_lens, cap, a.workers);
    else
        combine_kernel<float, true><<<grid, 128, sm, st>>>(
            a.o_part, a.lse_part, 0, a.batch, a.heads, a.d_latent, (float*)a.o_lat, a.lse,
            a.seq_lens, cap, a.workers);
    return cudaGetLastError();
}

cudaError_t launch_combine_dense(const float* o_part, const float* lse_part, int n_splits,
                                 int batch, int heads, int d_latent, void* o_lat, float* lse,
                                 int dtype, cudaStream_t st) {
    dim3 grid(batch, heads);
    if (dtype == MLA_DTYPE_BF16)
        combine_kernel<__nv_bfloat16, false><<<grid, 128, 0, st>>>(
            o_part, lse_part, n_splits, batch, heads, d_latent, (__nv_bfloat16*)o_lat, lse,
            nullptr, 0, 1);
    else
        combine_kernel<float, false><<<grid, 128, 0, st>>>(
            o_part, lse_part, n_splits, batch, heads, d_latent, (float*)o_lat, lse, nullptr, 0,
            1);
    return cudaGetLastError();
}

}  // namespace mla
