// Batched strided GEMM on CUDA cores with fp32 accumulation.
//
// Serves the small projections around the attention core where the shapes or
// the dtype (fp32) do not suit the tensor-core path: the query up-projection
// and absorption (first merge) and the value/output projections (second
// merge) of "Two merges are where the compute win comes from".  64x64 output
// tiles, 16-deep k slices staged in shared memory, 4x4 outputs per thread.
#include "common.cuh"
#include "kernels.h"

namespace mla {

template <typename TA, typename TB, typename Tout>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs g) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int z = blockIdx.z;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tid = threadIdx.x;
    const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
    const TA* A = (const TA*)g.A + (int64_t)z * g.sA;
    const TB* B = (const TB*)g.B + (int64_t)z * g.sB;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < g.K; k0 += BK) {
        for (int e = tid; e < BM * BK; e += 256) {
            int mm = e / BK, kk = e % BK;
            int m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.M && k < g.K) ? to_f(A[m * g.sAm + k * g.sAk]) : 0.f;
        }
        for (int e = tid; e < BN * BK; e += 256) {
            int kk = e / BN, nn = e % BN;
            int n = n0 + nn, k = k0 + kk;
            Bs[kk][nn] = (n < g.N && k < g.K) ? to_f(B[k * g.sBk + n * g.sBn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][tm + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tn + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    Tout* C = (Tout*)g.C + (int64_t)z * g.sC;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int m = m0 + tm + i, n = n0 + tn + j;
            if (m < g.M && n < g.N) C[m * g.sCm + n * g.sCn] = from_f<Tout>(acc[i][j]);
        }
}

template <typename TA, typename TB>
static void launch_ab(const GemmArgs& g, int c_dtype, dim3 grid, cudaStream_t st) {
    if (c_dtype == MLA_DTYPE_BF16)
        gemm_simt_kernel<TA, TB, __nv_bfloat16><<<grid, 256, 0, st>>>(g);
    else
        gemm_simt_kernel<TA, TB, float><<<grid, 256, 0, st>>>(g);
}

cudaError_t launch_gemm_simt(const GemmArgs& g, int a_dtype, int b_dtype, int c_dtype,
                             cudaStream_t st) {
    if (g.M == 0 || g.N == 0 || g.batch == 0) return cudaSuccess;
    dim3 grid((g.N + 63) / 64, (g.M + 63) / 64, g.batch);
    const bool ab = a_dtype == MLA_DTYPE_BF16, bb = b_dtype == MLA_DTYPE_BF16;
    if (ab && bb) launch_ab<__nv_bfloat16, __nv_bfloat16>(g, c_dtype, grid, st);
    else if (ab) launch_ab<__nv_bfloat16, float>(g, c_dtype, grid, st);
    else if (bb) launch_ab<float, __nv_bfloat16>(g, c_dtype, grid, st);
    else launch_ab<float, float>(g, c_dtype, grid, st);
    return cudaGetLastError();
}

}  // namespace mla
