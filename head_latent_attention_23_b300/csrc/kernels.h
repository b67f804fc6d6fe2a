// Internal launch interface between the C-ABI layer (mla_api.cu) and the
// kernel translation units.  Host code only; not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

struct DecodeArgs {
    int heads, d_latent, d_rope, block_size, max_blocks, batch;
    int workers;            // W: tile ranges the context is split into
    int tile;               // tokens per tile of the split plan
    int64_t num_blocks;
    float scale;
    const void* q_lat;      // [batch][heads][d_latent]
    const void* q_pe;       // [batch][heads][d_rope]
    const void* cache;      // [num_blocks][block_size][d_latent + d_rope]
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* o_part;          // [W + batch][heads][d_latent]
    float* lse_part;        // [W + batch][heads]
    int4* seq_slots;        // [batch]: first and last worker of each sequence and the
                            // total tile count, written by the decode kernel for the merge
    void* o_lat;            // [batch][heads][d_latent]
    float* lse;             // [batch][heads] or null
    int* status;
    uint64_t wait_ns;       // give-up time of the tensor-core kernel's pipeline waits
};

// (cos, sin) of every RoPE pair at each sequence's position: table[b][j].
cudaError_t launch_rope_table(const int32_t* pos, int batch, int d_rope, double rope_theta1,
                              float2* table, cudaStream_t st);

cudaError_t launch_decode_simt(const DecodeArgs& a, int dtype, cudaStream_t st);
size_t decode_simt_smem(const DecodeArgs& a);

// Tensor-core decode (bf16, 128 heads, d_latent 512, d_rope 64, pages of a
// multiple of 64 tokens).  Returns cudaErrorNotSupported when the device or
// the shapes do not fit it.
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
int decode_tc_workers(int num_sms);
int decode_tc_tile();   // tokens per tile of the tensor-core kernel's split plan
bool decode_tc_supported(int heads, int d_latent, int d_rope, int block_size, int dtype,
                         int batch);

// Merge of the partials written by a decode kernel (slots g + b of plan W).
cudaError_t launch_combine_planned(const DecodeArgs& a, int dtype, cudaStream_t st);
// Merge of dense partials [n_splits][batch][heads][d_latent].
cudaError_t launch_combine_dense(const float* o_part, const float* lse_part, int n_splits,
                                 int batch, int heads, int d_latent, void* o_lat, float* lse,
                                 int dtype, cudaStream_t st);

struct AppendArgs {
    int n_tok, d_in, d_latent, d_rope, block_size, max_blocks, batch;
    int64_t num_blocks;
    double rope_theta1;     // rope_base^(-2 / d_rope): the first pair's frequency
    const void* x;          // [n_tok][d_in]
    const void* w_dkv;      // [d_in][d_latent + d_rope]
    const int32_t* seq_idx;
    const int32_t* pos;
    const int32_t* block_table;
    void* cache;
    void* dense_out;        // or null
    float* rows_f32;        // optional precomputed fp32 rows [n_tok][d_latent + d_rope]
    int* status;
};
cudaError_t launch_append(const AppendArgs& a, int dtype, cudaStream_t st);

// Batched strided GEMM on CUDA cores, fp32 accumulation:
//   C[z][m][n] = sum_k A[z][m][k] * B[z][k][n]
// element (m,k) of A at A + z*sA + m*sAm + k*sAk (likewise B, C).
struct GemmArgs {
    int M, N, K, batch;
    const void* A; int64_t sA, sAm, sAk;
    const void* B; int64_t sB, sBk, sBn;
    void* C; int64_t sC, sCm, sCn;
};
// Element types of A, B and C: MLA_DTYPE_*.
cudaError_t launch_gemm_simt(const GemmArgs& g, int a_dtype, int b_dtype, int c_dtype,
                             cudaStream_t st);

// Splits fp32 per-head query rows [batch][heads][d_nope + d_rope] into
// q_nope and the rotated q_pe (dtype).
cudaError_t launch_q_split_rope(const float* q_all, int batch, int heads, int d_nope,
                                int d_rope, const int32_t* pos, double rope_theta1, void* q_nope,
                                void* q_pe, int dtype, cudaStream_t st);

// Multi-token decode rows: lens_x[b * T + j] = seq_lens[b] - T + 1 + j and a
// copy of block-table row b for each of them.
cudaError_t launch_expand_rows(const int32_t* seq_lens, const int32_t* block_table, int batch,
                               int q_tokens, int max_blocks, int32_t* lens_x, int32_t* table_x,
                               cudaStream_t st);

// pos[b] = seq_lens[b] - 1, seq_idx[b] = b (device arrays of one decode step).
cudaError_t launch_step_positions(const int32_t* seq_lens, int batch, int32_t* pos,
                                  int32_t* seq_idx, cudaStream_t st);

// ---------------------------------------------------------------- tcgen05 GEMM
// A bf16 operand seen by TMA as a 3-D array: dims[0] innermost (elements),
// strides[i] = byte stride of dims[i+1].  A: {K, M, batch}.  B: {K, N, batch}
// when K-major ([n][k] storage), {N, K, batch} when N-major ([k][n] storage).
struct TcOperand {
    const void* ptr;
    uint64_t dims[3];
    uint64_t strides[2];
};

struct TcGemmParams {
    int M, N, K;
    int b_mn;              // 1: B stored [k][n]
    int epi;               // 0: store C; 1: cache append (RoPE + paged scatter);
                           // 2: query split (columns of head h: d_nope to q_nope,
                           //    d_rope rotated at pos[m] to q_pe; bf16)
    void* C;               // epi 0: element (z, m, n) at C + z*sCz + m*sCm + n
    int64_t sCz, sCm;
    int c_dtype;
    // epi 1: rows are tokens, columns [0, d_latent) latent, [d_latent, N) rotary
    int d_latent, d_rope, block_size, max_blocks, batch;
    // epi 2: rows are sequences, N = heads x (d_nope + d_rope)
    int d_nope;
    __nv_bfloat16* q_nope;  // [M][heads][d_nope]
    __nv_bfloat16* q_pe;    // [M][heads][d_rope]
    const float2* rope_cs;  // [M][d_rope / 2] (cos, sin) at each row's position
    int64_t num_blocks;
    double rope_theta1;    // rope_base^(-2 / d_rope)
    const int32_t* seq_idx;
    const int32_t* pos;
    const int32_t* block_table;
    __nv_bfloat16* cache;
    __nv_bfloat16* dense_out;
    int* status;
    // split-K (batch-1 products only): fp32 scratch for the partial tiles, or
    // null to compute every tile in one pass; splits is chosen by the launcher
    float* partial;
    size_t partial_bytes;
    int splits;
    // skinny products (M <= 64, batched over z): the weights are the MMA's
    // A operand (128 output columns per tile as TMEM lanes) and the M rows of
    // activations its B operand, padded to np rows; set by
    // launch_gemm_tc_skinny
    int swap;
    int a_mn;              // swap: weights stored [k][n]
    int np;
};

// B must be weights: nothing that may run concurrently (the previous kernel
// on the stream, under programmatic dependent launch) writes it, because its
// first slices are read before the wait for that kernel.
cudaError_t launch_gemm_tc(const TcOperand& A, const TcOperand& B, const TcGemmParams& p,
                           int batch, cudaStream_t st);
// The same product C[z] = X[z] W[z] for few rows (M <= 64): X is [M][K]
// (K-major), W is [N][K] (w_kn = false) or [K][N] (w_kn = true); bf16 C.
cudaError_t launch_gemm_tc_skinny(const TcOperand& X, const TcOperand& W, bool w_kn,
                                  const TcGemmParams& p, int batch, cudaStream_t st);
// fp32 scratch bytes with which launch_gemm_tc would split a batch-1 M x N x K
// product over `sms` SMs (0: it would not split).
size_t gemm_tc_split_scratch(int M, int N, int K, int sms);

}  // namespace mla
