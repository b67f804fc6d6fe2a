// Merge of split-KV partial results.
//
// Each partial is a normalised output o_s over a token range with its
// log-sum-exp lse_s.  The full result over the union of the ranges is
//   LSE = log sum_s exp(lse_s),   o = sum_s exp(lse_s - LSE) * o_s,
// which is exact because exp(lse_s) is the softmax denominator of range s.
// Empty ranges carry lse = -inf and weigh nothing.
//
// One warp per (sequence, head), eight heads per CTA: the lanes compute the
// weights of up to 32 partials at a time with shuffles, then stream the
// partial rows with 16-byte loads (HBM/L2-bound, no tensor-core work).  The
// planned variant is launched as a programmatic dependent of the decode
// kernel: its set-up overlaps the decode tail and it waits for the partials
// with griddepcontrol.wait.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kWarps = 8;        // one head per warp
constexpr int kMaxSlots = 512;
constexpr int kEarly = 6;        // planned merges of up to 6 partials load every row at once

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
    *(float4*)dst = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b,
                                                      float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *(uint2*)dst = v;
}

template <typename T, bool kPlanned>
__global__ void __launch_bounds__(kWarps * 32, 2) combine_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, int n_splits,
    int batch, int heads, int DL, T* __restrict__ o_lat, float* __restrict__ lse,
    const int4* __restrict__ seq_slots, int W) {
    __shared__ int slots[kMaxSlots];
    __shared__ float wts[kWarps][kMaxSlots];
    __shared__ int n_sl;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y * kWarps + warp;

    if (kPlanned) {
        pdl_wait();
        // the decode kernel published this sequence's workers [g0, g1]; a worker
        // with an empty range (only when there are fewer tiles than workers)
        // wrote no partial and is skipped
        const int4 info = seq_slots[b];
        const int g0 = info.x, cnt = info.y - info.x + 1;
        const int64_t total = (int64_t)(uint32_t)info.z | ((int64_t)info.w << 32);
        for (int s = tid; s < cnt && s < kMaxSlots; s += blockDim.x) {
            const int g = g0 + s;
            slots[s] = plan_lo(g, total, W) < plan_lo(g + 1, total, W) ? g + b : -1;
        }
        if (tid == 0) n_sl = cnt < 0 ? 0 : (cnt < kMaxSlots ? cnt : kMaxSlots);
    } else {
        for (int s = tid; s < n_splits && s < kMaxSlots; s += blockDim.x) slots[s] = s;
        if (tid == 0) n_sl = n_splits < kMaxSlots ? n_splits : kMaxSlots;
    }
    __syncthreads();
    if (h >= heads) return;
    const int ns = n_sl;
    // slot -1: a worker without tokens (weight 0, never read)
    auto lse_at = [&](int s) -> float {
        if (slots[s] < 0) return -INFINITY;
        return kPlanned ? lse_part[(size_t)slots[s] * heads + h]
                        : lse_part[((size_t)slots[s] * batch + b) * heads + h];
    };
    auto row_at = [&](int s) -> const float* {
        if (slots[s] < 0) return nullptr;
        return kPlanned ? o_part + ((size_t)slots[s] * heads + h) * DL
                        : o_part + (((size_t)slots[s] * batch + b) * heads + h) * DL;
    };

    // A planned slot always holds a partial the decode kernel wrote, so with at
    // most kEarly slots every row load is issued before the weights are known:
    // the rows and the log-sum-exps then arrive in one memory round trip.
    const bool early = kPlanned && ns <= kEarly && (DL & 3) == 0 && DL <= 512;
    const int nq = (DL + 127) / 128;
    float4 v8[kEarly][4];
    if (early) {
#pragma unroll
        for (int i = 0; i < kEarly; ++i) {
            const float* row = i < ns ? row_at(i) : nullptr;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * lane + 128 * q;
                v8[i][q] = (row && q < nq && j < DL) ? *(const float4*)(row + j)
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }

    // weights: max and sum over the slots, 32 at a time
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32) m = fmaxf(m, lse_at(s));
    m = warp_max(m);
    float sum = 0.f;
    for (int s = lane; s < ns; s += 32) {
        const float l = lse_at(s);
        const float w = (l == -INFINITY) ? 0.f : expf(l - m);
        wts[warp][s] = w;
        sum += w;
    }
    sum = warp_sum(sum);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    __syncwarp();

    T* out = o_lat + ((size_t)b * heads + h) * DL;
    if (early) {
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kEarly; ++i) {
            const float w = i < ns ? wts[warp][i] * inv : 0.f;   // 0 for slot -1
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[q].x = fmaf(w, v8[i][q].x, acc[q].x);
                acc[q].y = fmaf(w, v8[i][q].y, acc[q].y);
                acc[q].z = fmaf(w, v8[i][q].z, acc[q].z);
                acc[q].w = fmaf(w, v8[i][q].w, acc[q].w);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 4 * lane + 128 * q;
            if (q < nq && j < DL) store4<T>(out + j, acc[q].x, acc[q].y, acc[q].z, acc[q].w);
        }
    } else if ((DL & 3) == 0 && DL <= 512) {
        // lane: columns 4 * lane + 128 * q, q < DL / 128 (at most 4 float4).
        // Four partials at a time, every load of a batch issued before the
        // first multiply, so a warp waits for memory once per batch.
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < ns; s0 += 4) {
            float4 v[4][4];
            float w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int si = s0 + i;
                w[i] = si < ns ? wts[warp][si] * inv : 0.f;
                const float* row = si < ns ? row_at(si) : nullptr;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = 4 * lane + 128 * q;
                    v[i][q] = (row && w[i] != 0.f && q < nq && j < DL)
                                  ? *(const float4*)(row + j)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[q].x = fmaf(w[i], v[i][q].x, acc[q].x);
                    acc[q].y = fmaf(w[i], v[i][q].y, acc[q].y);
                    acc[q].z = fmaf(w[i], v[i][q].z, acc[q].z);
                    acc[q].w = fmaf(w[i], v[i][q].w, acc[q].w);
                }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = 4 * lane + 128 * q;
            if (q < nq && j < DL) store4<T>(out + j, acc[q].x, acc[q].y, acc[q].z, acc[q].w);
        }
    } else {
        for (int j = lane; j < DL; j += 32) {
            float acc = 0.f;
            for (int s = 0; s < ns; ++s) {
                const float w = wts[warp][s] * inv;
                if (w != 0.f) acc = fmaf(w, row_at(s)[j], acc);   // w == 0 for slot -1
            }
            out[j] = from_f<T>(acc);
        }
    }
    if (lse && lane == 0) lse[(size_t)b * heads + h] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

template <typename T, bool kPlanned>
cudaError_t launch(const float* o_part, const float* lse_part, int n_splits, int batch,
                   int heads, int DL, void* o_lat, float* lse, const int4* seq_slots, int W,
                   bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(batch, (heads + kWarps - 1) / kWarps);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel<T, kPlanned>, o_part, lse_part, n_splits,
                              batch, heads, DL, (T*)o_lat, lse, seq_slots, W);
}

}  // namespace

cudaError_t launch_combine_planned(const DecodeArgs& a, int dtype, cudaStream_t st) {
    if (dtype == MLA_DTYPE_BF16)
        return launch<__nv_bfloat16, true>(a.o_part, a.lse_part, 0, a.batch, a.heads,
                                           a.d_latent, a.o_lat, a.lse, a.seq_slots, a.workers,
                                           true, st);
    return launch<float, true>(a.o_part, a.lse_part, 0, a.batch, a.heads, a.d_latent, a.o_lat,
                               a.lse, a.seq_slots, a.workers, true, st);
}

cudaError_t launch_combine_dense(const float* o_part, const float* lse_part, int n_splits,
                                 int batch, int heads, int d_latent, void* o_lat, float* lse,
                                 int dtype, cudaStream_t st) {
    if (n_splits > kMaxSlots) return cudaErrorInvalidValue;
    if (dtype == MLA_DTYPE_BF16)
        return launch<__nv_bfloat16, false>(o_part, lse_part, n_splits, batch, heads, d_latent,
                                            o_lat, lse, nullptr, 1, false, st);
    return launch<float, false>(o_part, lse_part, n_splits, batch, heads, d_latent, o_lat, lse,
                                nullptr, 1, false, st);
}

}  // namespace mla
