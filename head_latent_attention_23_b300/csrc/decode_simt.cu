// Split-KV absorbed decode on CUDA cores (fp32 FMA), any shape.
//
// One CTA per (worker range, head).  Used for fp32 configurations, where the
// tensor cores would only offer tf32, and for shapes the tensor-core kernel
// does not take.  For each 64-token tile: scores of the head's absorbed query
// against the cached rows (one warp per token), online softmax with a running
// max, and the weighted sum of the latents, all in fp32 ("How DeepSeek
// Rewrote the Transformer (MLA)", section 03 steps, in latent space).
#include "common.cuh"
#include "kernels.h"

namespace mla {

template <typename T>
__global__ void __launch_bounds__(128) decode_simt_kernel(DecodeArgs a) {
    extern __shared__ float smem[];
    const int H = a.heads, DL = a.d_latent, DR = a.d_rope, D = DL + DR;
    float* q = smem;                 // [D]
    float* o = q + D;                // [DL]
    float* s = o + DL;               // [kTile]
    int* pre = (int*)(s + kTile);    // [batch + 1]
    __shared__ float sh_m, sh_l, sh_alpha;

    const int g = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int cap = a.max_blocks * a.block_size;
    // This kernel is launched in plain stream order (no programmatic overlap),
    // so the previous call's merge kernel has finished reading the workspace
    // (or mla_decode_noalloc's shared static array) before anything here
    // writes it.
    tile_prefix(a.seq_lens, a.batch, cap, pre, a.status);
    if (blockIdx.x == 0 && blockIdx.y == 0) publish_seq_slots(pre, a.batch, a.workers, a.seq_slots);
    const int64_t total = pre[a.batch];
    const int64_t lo = plan_lo(g, total, a.workers), hi = plan_lo(g + 1, total, a.workers);
    if (lo >= hi) return;

    for (int b = seq_of_tile(pre, a.batch, lo); b < a.batch && pre[b] < hi; ++b) {
        int64_t t0 = lo > pre[b] ? lo : pre[b];
        int64_t t1 = hi < pre[b + 1] ? hi : pre[b + 1];
        if (t0 >= t1) continue;
        const int n = clamp_len(a.seq_lens[b], cap, nullptr);
        const int i_begin = (int)(t0 - pre[b]) * kTile;
        const int i_end = min(n, (int)(t1 - pre[b]) * kTile);

        const T* ql = (const T*)a.q_lat + ((size_t)b * H + h) * DL;
        const T* qp = (const T*)a.q_pe + ((size_t)b * H + h) * DR;
        for (int j = tid; j < DL; j += blockDim.x) { q[j] = to_f(ql[j]); o[j] = 0.f; }
        for (int j = tid; j < DR; j += blockDim.x) q[DL + j] = to_f(qp[j]);
        if (tid == 0) { sh_m = -INFINITY; sh_l = 0.f; }
        __syncthreads();

        for (int i0 = i_begin; i0 < i_end; i0 += kTile) {
            const int cnt = min(kTile, i_end - i0);
            // scores: warp w takes tokens w, w+4, ...
            for (int k = warp; k < kTile; k += 4) {
                float sc = -INFINITY;
                if (k < cnt) {
                    int i = i0 + k;
                    int32_t blk = a.block_table[(size_t)b * a.max_blocks + i / a.block_size];
                    if (blk < 0 || blk >= a.num_blocks) {
                        flag(a.status, MLA_ERR_INDEX);
                    } else {
                        const T* row = (const T*)a.cache +
                                       ((size_t)blk * a.block_size + i % a.block_size) * D;
                        float acc = 0.f;
                        for (int j = lane; j < D; j += 32) acc = fmaf(q[j], to_f(row[j]), acc);
                        acc = warp_sum(acc);
                        sc = acc * a.scale;
                    }
                }
                if (lane == 0) s[k] = sc;
            }
            __syncthreads();
            if (warp == 0) {
                float v0 = s[lane], v1 = s[lane + 32];
                float mt = warp_max(fmaxf(v0, v1));
                float m_new = fmaxf(sh_m, mt);
                float p0 = (v0 == -INFINITY) ? 0.f : expf(v0 - m_new);
                float p1 = (v1 == -INFINITY) ? 0.f : expf(v1 - m_new);
                s[lane] = p0;
                s[lane + 32] = p1;
                float ps = warp_sum(p0 + p1);
                if (lane == 0) {
                    float alpha = (sh_m == -INFINITY) ? 0.f : expf(sh_m - m_new);
                    if (m_new == -INFINITY) alpha = 1.f;
                    sh_alpha = alpha;
                    sh_l = sh_l * alpha + ps;
                    sh_m = m_new;
                }
            }
            __syncthreads();
            const float alpha = sh_alpha;
            for (int j = tid; j < DL; j += blockDim.x) {
                float acc = o[j] * alpha;
                for (int k = 0; k < cnt; ++k) {
                    float p = s[k];
                    if (p == 0.f) continue;
                    int i = i0 + k;
                    int32_t blk = a.block_table[(size_t)b * a.max_blocks + i / a.block_size];
                    if (blk < 0 || blk >= a.num_blocks) continue;
                    const T* row = (const T*)a.cache +
                                   ((size_t)blk * a.block_size + i % a.block_size) * D;
                    acc = fmaf(p, to_f(row[j]), acc);
                }
                o[j] = acc;
            }
            __syncthreads();
        }
        // partial result of this (worker, sequence) piece, normalised
        const size_t slot = (size_t)g + b;
        const float l = sh_l, m = sh_m;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* op = a.o_part + (slot * H + h) * DL;
        for (int j = tid; j < DL; j += blockDim.x) op[j] = o[j] * inv;
        if (tid == 0) a.lse_part[slot * H + h] = l > 0.f ? m + logf(l) : -INFINITY;
        __syncthreads();
    }
}

size_t decode_simt_smem(const DecodeArgs& a) {
    return sizeof(float) * (size_t)(a.d_latent + a.d_rope + a.d_latent + kTile) +
           sizeof(int) * (size_t)(a.batch + 1);
}

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t st) {
    dim3 grid(a.workers, a.heads);
    size_t sm = decode_simt_smem(a);
    if (dtype == MLA_DTYPE_BF16) {
        if (sm > 48 * 1024)
            cudaFuncSetAttribute(decode_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        decode_simt_kernel<__nv_bfloat16><<<grid, 128, sm, st>>>(a);
    } else {
        if (sm > 48 * 1024)
            cudaFuncSetAttribute(decode_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        decode_simt_kernel<float><<<grid, 128, sm, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace mla
