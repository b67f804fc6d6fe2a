// Cache append: down-projection of new tokens to [latent | rotary key] rows,
// RoPE on the rotary part, scatter into the paged cache (CUDA cores; the bf16
// append runs in the tensor-core GEMM's epilogue).  Also the small kernels
// around the projections: the query split and rotation for fp32
// configurations, the per-(sequence, pair) rotation table of the fused bf16
// query epilogue, the positions of a layer step and the per-token rows of a
// multi-token decode.
//
// "Multi-Head Latent Attention (MLA)", "The construction": the cached object
// is L = X W_L, one d_latent row per token for all heads; "The RoPE problem":
// a separate non-latent key part carries the rotary embedding.  The rotation
// convention (a reading; the pages give no formula): pairs (2j, 2j+1) turn by
// pos * rope_base^(-2j/d_rope).  Angles are formed and reduced to [-pi, pi]
// in fp64 (rope_cos_sin), so positions near 1e5 keep full fp32 accuracy
// after the rotation.
#include "common.cuh"
#include "kernels.h"

namespace mla {

// One CTA per new token.  Threads stride over the d_latent + d_rope output
// columns; x_t is staged in shared memory and each thread walks a column of
// W (coalesced across the warp).  When rows_f32 is given the projection was
// already done elsewhere and only the epilogue runs.
template <typename T>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
    extern __shared__ float sm[];
    const int D = a.d_latent + a.d_rope;
    float* xs = sm;          // [d_in]
    float* row = xs + a.d_in;  // [D]
    const int t = blockIdx.x, tid = threadIdx.x;
    if (a.rows_f32) {
        for (int j = tid; j < D; j += blockDim.x) row[j] = a.rows_f32[(size_t)t * D + j];
    } else {
        const T* x = (const T*)a.x + (size_t)t * a.d_in;
        for (int k = tid; k < a.d_in; k += blockDim.x) xs[k] = to_f(x[k]);
        __syncthreads();
        const T* w = (const T*)a.w_dkv;
        for (int j = tid; j < D; j += blockDim.x) {
            float acc = 0.f;
            for (int k = 0; k < a.d_in; ++k) acc = fmaf(xs[k], to_f(w[(size_t)k * D + j]), acc);
            row[j] = acc;
        }
    }
    __syncthreads();
    const int p = a.pos[t];
    // rotary part: thread j < d_rope/2 rotates pair j
    for (int j = tid; j < a.d_rope / 2; j += blockDim.x) {
        float c, s;
        rope_cos_sin(a.rope_theta1, j, p, &c, &s);
        float x0 = row[a.d_latent + 2 * j], x1 = row[a.d_latent + 2 * j + 1];
        row[a.d_latent + 2 * j] = x0 * c - x1 * s;
        row[a.d_latent + 2 * j + 1] = x0 * s + x1 * c;
    }
    __syncthreads();
    const int b = a.seq_idx[t];
    int64_t slot = -1;
    if (b >= 0 && b < a.batch && p >= 0 && p < a.max_blocks * a.block_size) {
        int32_t blk = a.block_table[(size_t)b * a.max_blocks + p / a.block_size];
        if (blk >= 0 && blk < a.num_blocks) slot = (int64_t)blk * a.block_size + p % a.block_size;
    }
    if (slot < 0 && tid == 0) flag(a.status, MLA_ERR_INDEX);
    T* dst = slot >= 0 ? (T*)a.cache + slot * D : nullptr;
    T* dense = a.dense_out ? (T*)a.dense_out + (size_t)t * D : nullptr;
    for (int j = tid; j < D; j += blockDim.x) {
        T v = from_f<T>(row[j]);
        if (dst) dst[j] = v;
        if (dense) dense[j] = v;
    }
}

cudaError_t launch_append(const AppendArgs& a, int dtype, cudaStream_t st) {
    if (a.n_tok == 0) return cudaSuccess;
    size_t sm = sizeof(float) * (size_t)(a.d_in + a.d_latent + a.d_rope);
    if (dtype == MLA_DTYPE_BF16) {
        if (sm > 48 * 1024)
            cudaFuncSetAttribute(append_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        append_kernel<__nv_bfloat16><<<a.n_tok, 256, sm, st>>>(a);
    } else {
        if (sm > 48 * 1024)
            cudaFuncSetAttribute(append_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        append_kernel<float><<<a.n_tok, 256, sm, st>>>(a);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- queries
// q_all [batch][heads][d_nope + d_rope] fp32 -> q_nope (copy) and q_pe
// (rotated at the sequence's position), both in dtype.  A CTA takes one
// sequence and kQHeads heads: the rotation angles depend only on the
// position, so each pair's cosine and sine are formed once per CTA and shared
// by its heads.  Threads move element pairs (8-byte loads) and each does a
// few of them, so the many CTAs, not a long per-thread loop, hide the memory
// latency.
constexpr int kQHeads = 16;

template <typename T>
__device__ __forceinline__ void store_pair(T* dst, float a, float b);
template <>
__device__ __forceinline__ void store_pair<float>(float* dst, float a, float b) {
    *(float2*)dst = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b) {
    *(__nv_bfloat162*)dst = __floats2bfloat162_rn(a, b);
}

template <typename T>
__global__ void __launch_bounds__(256) q_split_rope_kernel(
    const float* __restrict__ q_all, int heads, int d_nope, int d_rope,
    const int32_t* __restrict__ pos, double rope_theta1, T* __restrict__ q_nope,
    T* __restrict__ q_pe) {
    extern __shared__ float cs[];   // [d_rope / 2][2]: cos, sin
    const int b = blockIdx.x, h0 = blockIdx.y * kQHeads, half_r = d_rope / 2;
    const int hn = min(kQHeads, heads - h0);
    const int p = pos[b];
    for (int j = threadIdx.x; j < half_r; j += blockDim.x)
        rope_cos_sin(rope_theta1, j, p, &cs[2 * j], &cs[2 * j + 1]);
    __syncthreads();
    const int dq = d_nope + d_rope;
    const float* src = q_all + ((size_t)b * heads + h0) * dq;
    T* dn = q_nope + ((size_t)b * heads + h0) * d_nope;
    T* dp = q_pe + ((size_t)b * heads + h0) * d_rope;
    if ((d_nope & 1) == 0) {
        const int half_n = d_nope / 2;
        for (int e = threadIdx.x; e < hn * half_n; e += blockDim.x) {
            const int h = e / half_n, j = 2 * (e - h * half_n);
            const float2 v = *(const float2*)(src + (size_t)h * dq + j);
            store_pair<T>(dn + (size_t)h * d_nope + j, v.x, v.y);
        }
        for (int e = threadIdx.x; e < hn * half_r; e += blockDim.x) {
            const int h = e / half_r, j = e - h * half_r;
            const float2 x = *(const float2*)(src + (size_t)h * dq + d_nope + 2 * j);
            const float c = cs[2 * j], sn = cs[2 * j + 1];
            store_pair<T>(dp + (size_t)h * d_rope + 2 * j, x.x * c - x.y * sn, x.x * sn + x.y * c);
        }
    } else {
        // odd d_nope: rows are not 8-byte aligned, move single elements
        for (int e = threadIdx.x; e < hn * d_nope; e += blockDim.x) {
            const int h = e / d_nope, j = e - h * d_nope;
            dn[(size_t)h * d_nope + j] = from_f<T>(src[(size_t)h * dq + j]);
        }
        for (int e = threadIdx.x; e < hn * half_r; e += blockDim.x) {
            const int h = e / half_r, j = e - h * half_r;
            const float x0 = src[(size_t)h * dq + d_nope + 2 * j];
            const float x1 = src[(size_t)h * dq + d_nope + 2 * j + 1];
            const float c = cs[2 * j], sn = cs[2 * j + 1];
            dp[(size_t)h * d_rope + 2 * j] = from_f<T>(x0 * c - x1 * sn);
            dp[(size_t)h * d_rope + 2 * j + 1] = from_f<T>(x0 * sn + x1 * c);
        }
    }
}

cudaError_t launch_q_split_rope(const float* q_all, int batch, int heads, int d_nope,
                                int d_rope, const int32_t* pos, double rope_theta1, void* q_nope,
                                void* q_pe, int dtype, cudaStream_t st) {
    const size_t sm = (size_t)(d_rope > 0 ? d_rope : 2) * sizeof(float);
    const dim3 grid(batch, (heads + kQHeads - 1) / kQHeads);
    if (dtype == MLA_DTYPE_BF16)
        q_split_rope_kernel<__nv_bfloat16><<<grid, 256, sm, st>>>(
            q_all, heads, d_nope, d_rope, pos, rope_theta1, (__nv_bfloat16*)q_nope,
            (__nv_bfloat16*)q_pe);
    else
        q_split_rope_kernel<float><<<grid, 256, sm, st>>>(q_all, heads, d_nope, d_rope, pos,
                                                         rope_theta1, (float*)q_nope,
                                                         (float*)q_pe);
    return cudaGetLastError();
}

// Position and sequence index of each sequence's newest token for one
// decode step: pos[b] = seq_lens[b] - 1 (the query and the appended row sit
// at the last position), seq_idx[b] = b.  A length below 1 gives pos -1,
// which the append flags as an invalid slot.
__global__ void step_positions_kernel(const int32_t* __restrict__ seq_lens, int batch,
                                      int32_t* __restrict__ pos, int32_t* __restrict__ seq_idx) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int n = seq_lens[b];
    pos[b] = n >= 1 ? n - 1 : -1;
    seq_idx[b] = b;
}

// Rows of a multi-token decode: query token j of sequence b (the last
// q_tokens tokens of a sequence of n) sits at position n - q_tokens + j and
// attends to the n - q_tokens + j + 1 tokens up to it, through the
// sequence's own block table.  Row r = b * q_tokens + j gets that length and
// a copy of row b of the block table.  Lengths below 1 stay as they are (the
// decode flags and skips them).
__global__ void expand_rows_kernel(const int32_t* __restrict__ seq_lens,
                                   const int32_t* __restrict__ block_table, int batch,
                                   int q_tokens, int max_blocks, int32_t* __restrict__ lens_x,
                                   int32_t* __restrict__ table_x) {
    const int r = blockIdx.x, b = r / q_tokens, j = r - b * q_tokens;
    if (threadIdx.x == 0) lens_x[r] = seq_lens[b] - q_tokens + 1 + j;
    for (int i = threadIdx.x; i < max_blocks; i += blockDim.x)
        table_x[(size_t)r * max_blocks + i] = block_table[(size_t)b * max_blocks + i];
}

cudaError_t launch_expand_rows(const int32_t* seq_lens, const int32_t* block_table, int batch,
                               int q_tokens, int max_blocks, int32_t* lens_x, int32_t* table_x,
                               cudaStream_t st) {
    expand_rows_kernel<<<batch * q_tokens, 128, 0, st>>>(seq_lens, block_table, batch, q_tokens,
                                                         max_blocks, lens_x, table_x);
    return cudaGetLastError();
}

// (cos, sin) of every RoPE pair at each sequence's position, for epilogues
// that rotate many heads' query parts: formed once per (sequence, pair).
__global__ void rope_table_kernel(const int32_t* __restrict__ pos, int half_r, double rope_theta1,
                                  float2* __restrict__ table) {
    const int b = blockIdx.x, p = pos[b];
    for (int j = threadIdx.x; j < half_r; j += blockDim.x) {
        float c, s;
        rope_cos_sin(rope_theta1, j, p, &c, &s);
        table[(size_t)b * half_r + j] = make_float2(c, s);
    }
}

cudaError_t launch_rope_table(const int32_t* pos, int batch, int d_rope, double rope_theta1,
                              float2* table, cudaStream_t st) {
    if (d_rope < 2) return cudaSuccess;
    rope_table_kernel<<<batch, 32, 0, st>>>(pos, d_rope / 2, rope_theta1, table);
    return cudaGetLastError();
}

cudaError_t launch_step_positions(const int32_t* seq_lens, int batch, int32_t* pos,
                                  int32_t* seq_idx, cudaStream_t st) {
    step_positions_kernel<<<(batch + 255) / 256, 256, 0, st>>>(seq_lens, batch, pos, seq_idx);
    return cudaGetLastError();
}

}  // namespace mla
