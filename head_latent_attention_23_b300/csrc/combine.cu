// Merge of split-KV partial results.
//
// Each partial is a normalised output o_s over a token range with its
// log-sum-exp lse_s.  The full result over the union of the ranges is
//   LSE = log sum_s exp(lse_s),   o = sum_s exp(lse_s - LSE) * o_s,
// which is exact because exp(lse_s) is the softmax denominator of range s.
// Empty ranges carry lse = -inf and weigh nothing.
//
// One warp per (sequence, head), four heads per CTA: the lanes compute the
// weights of up to 32 partials at a time with shuffles, then stream the
// partial rows with 16-byte loads (HBM/L2-bound, no tensor-core work).  The
// planned variant is launched as a programmatic dependent of the decode
// kernel: its set-up overlaps the decode tail and it waits for the partials
// with griddepcontrol.wait.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int kWarps = 4;
constexpr int kMaxSlots = 1024;

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
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, int n_splits,
    int batch, int heads, int DL, T* __restrict__ o_lat, float* __restrict__ lse,
    const int32_t* __restrict__ seq_lens, int cap, int W, int tile) {
    __shared__ int slots[kMaxSlots];
    __shared__ float wts[kWarps][kMaxSlots];
    __shared__ int red[2][kWarps];
    __shared__ int n_sl;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y * kWarps + warp;

    if (kPlanned) {
        pdl_wait();
        // tiles of the sequences before b, and in all sequences
        int before = 0, all = 0, mine = 0;
        for (int j = tid; j < batch; j += blockDim.x) {
            int n = seq_lens[j];
            n = (n < 1) ? 0 : (n > cap ? cap : n);
            const int t = (n + tile - 1) / tile;
            all += t;
            if (j < b) before += t;
            if (j == b) mine = t;
        }
        before = __reduce_add_sync(0xffffffffu, before);
        all = __reduce_add_sync(0xffffffffu, all);
        mine = __reduce_add_sync(0xffffffffu, mine);
        if (lane == 0) {
            red[0][warp] = before;
            red[1][warp] = all;
        }
        __shared__ int sh_mine[kWarps];
        if (lane == 0) sh_mine[warp] = mine;
        __syncthreads();
        if (tid == 0) {
            int64_t p0 = 0, total = 0;
            int t_b = 0;
            for (int w = 0; w < kWarps; ++w) {
                p0 += red[0][w];
                total += red[1][w];
                t_b += sh_mine[w];
            }
            const int64_t p1 = p0 + t_b;
            int cnt = 0;
            if (p1 > p0) {
                // workers whose tile range [plan_lo(g), plan_lo(g+1)) meets [p0, p1)
                int g = (int)(p0 * W / total);
                while (g > 0 && plan_lo(g, total, W) > p0) --g;
                while (g + 1 < W && plan_lo(g + 1, total, W) <= p0) ++g;
                for (; g < W && plan_lo(g, total, W) < p1; ++g) {
                    const int64_t glo = plan_lo(g, total, W), ghi = plan_lo(g + 1, total, W);
                    if (ghi <= p0 || glo >= ghi) continue;
                    if (cnt < kMaxSlots) slots[cnt++] = g + b;
                }
            }
            n_sl = cnt;
        }
    } else {
        for (int s = tid; s < n_splits && s < kMaxSlots; s += blockDim.x) slots[s] = s;
        if (tid == 0) n_sl = n_splits < kMaxSlots ? n_splits : kMaxSlots;
    }
    __syncthreads();
    if (h >= heads) return;
    const int ns = n_sl;
    auto lse_at = [&](int s) -> float {
        return kPlanned ? lse_part[(size_t)slots[s] * heads + h]
                        : lse_part[((size_t)slots[s] * batch + b) * heads + h];
    };
    auto row_at = [&](int s) -> const float* {
        return kPlanned ? o_part + ((size_t)slots[s] * heads + h) * DL
                        : o_part + (((size_t)slots[s] * batch + b) * heads + h) * DL;
    };

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
    if ((DL & 3) == 0 && DL <= 512) {
        // lane: columns 4 * lane + 128 * q, q < DL / 128 (at most 4 float4).
        // Eight partials at a time, every load of a batch issued before the
        // first multiply, so a warp waits for memory once per batch.
        const int nq = (DL + 127) / 128;
        float4 acc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < ns; s0 += 8) {
            float4 v[8][4];
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
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
            for (int i = 0; i < 8; ++i)
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
                if (w != 0.f) acc = fmaf(w, row_at(s)[j], acc);
            }
            out[j] = from_f<T>(acc);
        }
    }
    if (lse && lane == 0) lse[(size_t)b * heads + h] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

template <typename T, bool kPlanned>
cudaError_t launch(const float* o_part, const float* lse_part, int n_splits, int batch,
                   int heads, int DL, void* o_lat, float* lse, const int32_t* seq_lens, int cap,
                   int W, int tile, bool pdl, cudaStream_t st) {
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
                              batch, heads, DL, (T*)o_lat, lse, seq_lens, cap, W, tile);
}

}  // namespace

cudaError_t launch_combine_planned(const DecodeArgs& a, int dtype, cudaStream_t st) {
    const int cap = a.max_blocks * a.block_size;
    if (dtype == MLA_DTYPE_BF16)
        return launch<__nv_bfloat16, true>(a.o_part, a.lse_part, 0, a.batch, a.heads,
                                           a.d_latent, a.o_lat, a.lse, a.seq_lens, cap,
                                           a.workers, a.tile, true, st);
    return launch<float, true>(a.o_part, a.lse_part, 0, a.batch, a.heads, a.d_latent, a.o_lat,
                               a.lse, a.seq_lens, cap, a.workers, a.tile, true, st);
}

cudaError_t launch_combine_dense(const float* o_part, const float* lse_part, int n_splits,
                                 int batch, int heads, int d_latent, void* o_lat, float* lse,
                                 int dtype, cudaStream_t st) {
    if (n_splits > kMaxSlots) return cudaErrorInvalidValue;
    if (dtype == MLA_DTYPE_BF16)
        return launch<__nv_bfloat16, false>(o_part, lse_part, n_splits, batch, heads, d_latent,
                                            o_lat, lse, nullptr, 0, 1, 1, false, st);
    return launch<float, false>(o_part, lse_part, n_splits, batch, heads, d_latent, o_lat, lse,
                                nullptr, 0, 1, 1, false, st);
}

}  // namespace mla
