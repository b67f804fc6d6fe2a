// Cache append: down-projection of new tokens to [latent | rotary key] rows,
// RoPE on the rotary part, scatter into the paged cache.
//
// "Multi-Head Latent Attention (MLA)", "The construction": the cached object
// is L = X W_L, one d_latent row per token for all heads; "The RoPE problem":
// a separate non-latent key part carries the rotary embedding.  The rotation
// convention (a reading; the pages give no formula): pairs (2j, 2j+1) turn by
// pos * rope_base^(-2j/d_rope).  Angles are formed and reduced in fp64 so
// positions near 1e5 keep full fp32 accuracy after the rotation.
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
        double theta = pow(a.rope_base, -2.0 * (double)j / (double)a.d_rope);
        double phi = fmod((double)p * theta, 6.283185307179586476925286766559);
        double sn, cs;
        sincos(phi, &sn, &cs);
        float c = (float)cs, s = (float)sn;
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
// (rotated at the sequence's position), both in dtype.  One CTA per
// sequence: the rotation angles depend only on the position, so each pair's
// cosine and sine are formed once per sequence (in fp64, then rounded to
// fp32) and shared by all heads; fp64 transcendentals are slow on this GPU.
template <typename T>
__global__ void __launch_bounds__(256) q_split_rope_kernel(
    const float* __restrict__ q_all, int heads, int d_nope, int d_rope,
    const int32_t* __restrict__ pos, double rope_base, T* __restrict__ q_nope,
    T* __restrict__ q_pe) {
    extern __shared__ float cs[];   // [d_rope / 2][2]: cos, sin
    const int b = blockIdx.x, half_r = d_rope / 2;
    const int p = pos[b];
    for (int j = threadIdx.x; j < half_r; j += blockDim.x) {
        const double theta = pow(rope_base, -2.0 * (double)j / (double)d_rope);
        const double phi = fmod((double)p * theta, 6.283185307179586476925286766559);
        double sn, c;
        sincos(phi, &sn, &c);
        cs[2 * j] = (float)c;
        cs[2 * j + 1] = (float)sn;
    }
    __syncthreads();
    const int dq = d_nope + d_rope;
    const float* src = q_all + (size_t)b * heads * dq;
    T* dn = q_nope + (size_t)b * heads * d_nope;
    T* dp = q_pe + (size_t)b * heads * d_rope;
    for (int e = threadIdx.x; e < heads * d_nope; e += blockDim.x) {
        const int h = e / d_nope, j = e - h * d_nope;
        dn[e] = from_f<T>(src[(size_t)h * dq + j]);
    }
    for (int e = threadIdx.x; e < heads * half_r; e += blockDim.x) {
        const int h = e / half_r, j = e - h * half_r;
        const float x0 = src[(size_t)h * dq + d_nope + 2 * j];
        const float x1 = src[(size_t)h * dq + d_nope + 2 * j + 1];
        const float c = cs[2 * j], s = cs[2 * j + 1];
        dp[(size_t)h * d_rope + 2 * j] = from_f<T>(x0 * c - x1 * s);
        dp[(size_t)h * d_rope + 2 * j + 1] = from_f<T>(x0 * s + x1 * c);
    }
}

cudaError_t launch_q_split_rope(const float* q_all, int batch, int heads, int d_nope,
                                int d_rope, const int32_t* pos, double rope_base, void* q_nope,
                                void* q_pe, int dtype, cudaStream_t st) {
    const size_t sm = (size_t)(d_rope > 0 ? d_rope : 2) * sizeof(float);
    if (dtype == MLA_DTYPE_BF16)
        q_split_rope_kernel<__nv_bfloat16><<<batch, 256, sm, st>>>(
            q_all, heads, d_nope, d_rope, pos, rope_base, (__nv_bfloat16*)q_nope,
            (__nv_bfloat16*)q_pe);
    else
        q_split_rope_kernel<float><<<batch, 256, sm, st>>>(q_all, heads, d_nope, d_rope, pos,
                                                          rope_base, (float*)q_nope,
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

cudaError_t launch_step_positions(const int32_t* seq_lens, int batch, int32_t* pos,
                                  int32_t* seq_idx, cudaStream_t st) {
    step_positions_kernel<<<(batch + 255) / 256, 256, 0, st>>>(seq_lens, batch, pos, seq_idx);
    return cudaGetLastError();
}

}  // namespace mla
