// Internal helpers shared by the libmla.so translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

// ---------------------------------------------------------------- elements
template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void flag(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- split plan
// The decode work is the sequence of fixed-size token tiles (64 tokens on the
// CUDA cores, 128 on the tensor cores) of all sequences laid end to end.  Worker g of W takes the tile range [lo(g), lo(g+1)), which can
// cross sequence boundaries; each (worker, sequence) piece yields one partial
// result in slot g + b.  Slots are unique (ranges are ordered) and fewer than
// W + batch.
constexpr int kTile = 64;

__host__ __device__ __forceinline__ int64_t plan_lo(int g, int64_t total, int W) {
    return (int64_t)g * total / W;
}

// Rotation of RoPE pair j at position pos, as (cos, sin) in fp32.  The
// frequency theta_j = theta1^j comes from theta1 = rope_base^(-2/d_rope)
// (formed in fp64 on the host) by repeated squaring in fp64; the angle
// pos * theta_j is formed in fp64 and reduced to about [-pi, pi] by
// subtracting the nearest multiple of 2 pi, with 2 pi split into two
// doubles (Cody and Waite's reduction), so positions near 1e5 keep the
// angle's fp32 accuracy; sincosf then takes the small reduced angle.  Only
// multiplies and fused multiply-adds run in fp64, which is slow on this GPU.
__device__ __forceinline__ void rope_cos_sin(double theta1, int j, int pos, float* c, float* s) {
    double th = 1.0, b = theta1;
    for (int e = j; e; e >>= 1) {
        if (e & 1) th *= b;
        b *= b;
    }
    const double phi = (double)pos * th;
    const double k = rint(phi * 0.15915494309189535);     // nearest turn: phi / (2 pi)
    double r = fma(-k, 6.283185307179586, phi);           // 2 pi, leading double
    r = fma(-k, 2.4492935982947064e-16, r);               // 2 pi, remainder
    sincosf((float)r, s, c);
}

// Seq length actually used: out-of-range lengths are flagged and clamped.
__device__ __forceinline__ int clamp_len(int n, int cap, int* status) {
    if (n < 1 || n > cap) {
        flag(status, MLA_ERR_INVALID_ARG);
        return n < 1 ? 0 : cap;
    }
    return n;
}

// Block-wide exclusive prefix of ceil(len_b / tile) over b = 0..batch-1 into
// pre[0..batch] (shared); the clamped lengths go to lens[0..batch-1] when
// lens is not null.  All threads must call.
__device__ __forceinline__ void tile_prefix(const int32_t* seq_lens, int batch, int cap,
                                            int* pre, int* status, int* lens = nullptr,
                                            int tile = kTile) {
    __shared__ int warp_tot[32];
    const int tid = threadIdx.x, nt = blockDim.x;
    int carry = 0;
    for (int base = 0; base < batch; base += nt) {
        int b = base + tid;
        int v = 0;
        if (b < batch) {
            const int n = clamp_len(seq_lens[b], cap, status);
            if (lens) lens[b] = n;
            v = (n + tile - 1) / tile;
        }
        // inclusive scan within the warp
        int lane = tid & 31, w = tid >> 5;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[w] = x;
        __syncthreads();
        int off = 0;
        for (int k = 0; k < w; ++k) off += warp_tot[k];
        if (b < batch) pre[b] = carry + off + x - v;
        int chunk = 0;
        for (int k = 0; k < (nt + 31) / 32; ++k) chunk += warp_tot[k];
        __syncthreads();
        carry += chunk;
    }
    if (tid == 0) pre[batch] = carry;
    __syncthreads();
}

// Worker whose range [plan_lo(g), plan_lo(g+1)) holds tile t (0 <= t < total):
// the largest g with floor(g * total / W) <= t.
__host__ __device__ __forceinline__ int worker_of_tile(int64_t t, int64_t total, int W) {
    return (int)(((t + 1) * W - 1) / total);
}

// Publishes, for each sequence, the first and last worker whose range meets it
// and the total tile count: the merge kernel reads its partial slots from this
// instead of recomputing the tile prefix.  One CTA of the decode grid calls
// it (all its threads), after the prefix is in shared memory.
__device__ __forceinline__ void publish_seq_slots(const int* pre, int batch, int W, int4* out) {
    const int64_t total = pre[batch];
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        int4 v = make_int4(0, -1, (int)(total & 0xffffffff), (int)(total >> 32));
        if (pre[b + 1] > pre[b]) {
            v.x = worker_of_tile(pre[b], total, W);
            v.y = worker_of_tile(pre[b + 1] - 1, total, W);
        }
        out[b] = v;
    }
}

// Index of the sequence holding global tile t: largest b with pre[b] <= t.
__device__ __forceinline__ int seq_of_tile(const int* pre, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace mla
