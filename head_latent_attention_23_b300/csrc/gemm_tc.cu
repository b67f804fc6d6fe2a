// Tensor-core GEMM for the projections around the attention core (bf16
// operands, fp32 accumulation in TMEM): the query up-projection, whose
// epilogue splits each head's columns into q_nope and the rotated q_pe, and
// its absorption into latent space (first merge), the value/output
// projections (second merge) and the cache append's down-projection, whose
// epilogue applies RoPE and scatters rows into the paged cache.
//
//   C[z][m][n] = sum_k A[z][m][k] * B[z][k][n]
//
// 128 x 128 tiles of C, K in 64-deep slices of A (K-major) and B (K-major or
// N-major) streamed into a ring of stages with TMA (128-byte swizzle);
// tcgen05.mma (M=128, N=128, K=16) accumulates in TMEM.  The kernel is
// persistent (at most one CTA per SM, looping over work items) so that, at
// decode batch sizes where a tile is a few k slices, the weight stream never
// stops for a CTA's set-up or epilogue.
//
// Split-K.  A product with fewer output tiles than SMs (W_O, the query and
// cache down-projections at decode batch sizes) would leave most SMs idle
// while a few stream long K ranges.  With p.splits > 1 a work item is a
// (tile, K range) pair; its epilogue writes an fp32 partial tile to
// p.partial[split][m][n], and splitk_reduce_kernel adds the partials and
// applies the product's epilogue (store, RoPE and the paged scatter, or the
// query split and rotation).
//
// B (or, for a skinny product, A) is the weights: the first stages' weight
// slices are requested before the wait for the previous kernel, since no
// kernel that may overlap this one writes them.
//
// Skinny products (p.swap).  The per-head query absorption and value
// projection at decode batch sizes have M = batch rows: as the MMA's M side
// they would fill 16 of its 128 rows and leave 7/8 of every epilogue idle.
// They run transposed instead, C^T = W^T X^T: a tile is 128 output columns
// (128 weight rows as the A operand, TMEM lanes) by the M activation rows
// padded to np (the B operand, N = np of the MMA), so the weight stream is
// the only large operand and each epilogue thread writes one output column.
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace mla {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kTileBytes = 16384;   // one 128 x 64 bf16 slice of A or of B
// Ring: six stages of A and B slices (96 KB of weights in flight per SM:
// with HBM latency near 2 us under load, fewer stages cap a CTA's weight
// stream below its share of the bandwidth); a skinny product's stage is a
// weight slice and at most 64 activation rows (8 KB), so seven stages fit
// next to two CTAs of the merge kernel, which it may overlap.
template <bool kSwap>
struct Ring {
    static constexpr int stages = kSwap ? 7 : 6;
    static constexpr int b_bytes = kSwap ? 8192 : kTileBytes;
    static constexpr int smem = 1024 + stages * (kTileBytes + b_bytes) + 256;
};
constexpr int kSkinnyMaxRows = Ring<true>::b_bytes / 128;   // 64
constexpr int kAcc = 2;             // TMEM accumulators: the epilogue drains one tile
                                    // while the MMAs fill the other

using namespace tc;

// Query split epilogue (epi 2): columns (n, n + 1) of row m, n even, are a
// pair of head n / (d_nope + d_rope): the latent-side part goes to q_nope as
// is, the rotary part is rotated by the row's (cos, sin) from p.rope_cs and
// goes to q_pe (one rounding to bf16 after fp32 sums and the rotation).
__device__ __forceinline__ void query_pair(const TcGemmParams& p, int m, int n, float x0,
                                           float x1) {
    const int dq = p.d_nope + p.d_rope, hq = p.N / dq;
    const int h = n / dq, j = n - h * dq;
    if (j < p.d_nope) {
        *(__nv_bfloat162*)(p.q_nope + ((size_t)m * hq + h) * p.d_nope + j) =
            __floats2bfloat162_rn(x0, x1);
    } else {
        const int jr = (j - p.d_nope) >> 1;
        const float2 r = p.rope_cs[(size_t)m * (p.d_rope >> 1) + jr];
        const float cs = r.x, sn = r.y;
        *(__nv_bfloat162*)(p.q_pe + ((size_t)m * hq + h) * p.d_rope + 2 * jr) =
            __floats2bfloat162_rn(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
    }
}

// Output tile `t` of the (n, m, z) grid of 128 x 128 tiles.
struct TileId {
    int n0, m0, z;
};
__device__ __forceinline__ TileId tile_of(int t, int tiles_n, int tiles_m) {
    TileId r;
    r.n0 = (t % tiles_n) * kBN;
    r.m0 = ((t / tiles_n) % tiles_m) * kBM;
    r.z = t / (tiles_n * tiles_m);
    return r;
}

// Persistent: CTA c takes work items c, c + gridDim.x, ...  Warp 0 streams
// the k slices of all its items through one ring; one thread of warp 1
// accumulates each item into one of two TMEM buffers; warps 2-5 drain a
// finished buffer (128 rows = TMEM lanes) while the next item is computed.
// Item i is tile i / splits, K range i % splits.
__device__ __forceinline__ void item_range(int item, int splits, int nk, int* tile, int* kt0,
                                           int* kt1) {
    const int sp = item % splits;
    *tile = item / splits;
    *kt0 = (int)((int64_t)sp * nk / splits);
    *kt1 = (int)((int64_t)(sp + 1) * nk / splits);
}

template <bool kSwap>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                   const TcGemmParams p, int tiles_n, int tiles_m, int num_items) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    constexpr int kStages = Ring<kSwap>::stages, kBBytes = Ring<kSwap>::b_bytes;
    uint8_t* sB = smem + kStages * kTileBytes;
    uint64_t* full = (uint64_t*)(sB + kStages * kBBytes);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + kAcc;
    uint64_t* done = acc_empty + kAcc;
    uint32_t* tslot = (uint32_t*)(done + 1);
    volatile int* abort_flag = (volatile int*)(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = (p.K + kBK - 1) / kBK;
    int pre = 0;    // slices whose weight copies went out before the wait

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kAcc; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 128);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tA);
        prefetch_tmap(&tB);
        // The weights (B, or A of a skinny product) are never written by a
        // kernel this one may overlap, so the first stages' weight slices are
        // requested before the previous kernel has finished: their
        // first-touch latency hides behind its tail.
        for (int t = blockIdx.x; t < num_items && pre < kStages; t += gridDim.x) {
            int tile, kt0, kt1;
            item_range(t, p.splits, nk, &tile, &kt0, &kt1);
            const TileId ti = tile_of(tile, tiles_n, tiles_m);
            for (int kt = kt0; kt < kt1 && pre < kStages; ++kt, ++pre) {
                if (kSwap) {
                    uint8_t* dst = sA + pre * kTileBytes;
                    mbar_arrive_expect_tx(&full[pre], kTileBytes + p.np * 128);
                    if (p.a_mn) {
                        tma_load_3d(dst, &tA, ti.n0, kt * kBK, ti.z, &full[pre]);
                        tma_load_3d(dst + kTileBytes / 2, &tA, ti.n0 + 64, kt * kBK, ti.z,
                                    &full[pre]);
                    } else {
                        tma_load_3d(dst, &tA, kt * kBK, ti.n0, ti.z, &full[pre]);
                    }
                } else {
                    uint8_t* dst = sB + pre * kBBytes;
                    mbar_arrive_expect_tx(&full[pre], 2 * kTileBytes);
                    if (p.b_mn) {
                        tma_load_3d(dst, &tB, ti.n0, kt * kBK, ti.z, &full[pre]);
                        tma_load_3d(dst + kTileBytes / 2, &tB, ti.n0 + 64, kt * kBK, ti.z,
                                    &full[pre]);
                    } else {
                        tma_load_3d(dst, &tB, kt * kBK, ti.n0, ti.z, &full[pre]);
                    }
                }
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tslot, kAcc * kBN);
        tmem_relinquish();
    }
    // set-up above overlaps the previous kernel's tail; the activations are
    // read, and C written, only once it has finished
    pdl_wait_primary();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_items && ok; t += gridDim.x) {
                int tile, kt0, kt1;
                item_range(t, p.splits, nk, &tile, &kt0, &kt1);
                const TileId ti = tile_of(tile, tiles_n, tiles_m);
                for (int kt = kt0; kt < kt1; ++kt, ++it) {
                    const int s = it % kStages;
                    if (it < pre) {
                        // weights requested before the wait: the activations now
                        if (kSwap)
                            tma_load_3d(sB + s * kBBytes, &tB, kt * kBK, 0, ti.z, &full[s]);
                        else
                            tma_load_3d(sA + s * kTileBytes, &tA, kt * kBK, ti.m0, ti.z, &full[s]);
                        continue;
                    }
                    if (!mbar_wait_fast(&empty[s], ((it / kStages) & 1) ^ 1, abort_flag,
                                        p.status)) {
                        ok = false;
                        break;
                    }
                    if (kSwap) {
                        // weights: 128 output columns x 64 k; activations: np rows x 64 k
                        mbar_arrive_expect_tx(&full[s], kTileBytes + p.np * 128);
                        if (p.a_mn) {
                            tma_load_3d(sA + s * kTileBytes, &tA, ti.n0, kt * kBK, ti.z, &full[s]);
                            tma_load_3d(sA + s * kTileBytes + kTileBytes / 2, &tA, ti.n0 + 64,
                                        kt * kBK, ti.z, &full[s]);
                        } else {
                            tma_load_3d(sA + s * kTileBytes, &tA, kt * kBK, ti.n0, ti.z, &full[s]);
                        }
                        tma_load_3d(sB + s * kBBytes, &tB, kt * kBK, 0, ti.z, &full[s]);
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
                    tma_load_3d(sA + s * kTileBytes, &tA, kt * kBK, ti.m0, ti.z, &full[s]);
                    if (p.b_mn) {
                        tma_load_3d(sB + s * kBBytes, &tB, ti.n0, kt * kBK, ti.z, &full[s]);
                        tma_load_3d(sB + s * kBBytes + kTileBytes / 2, &tB, ti.n0 + 64,
                                    kt * kBK, ti.z, &full[s]);
                    } else {
                        tma_load_3d(sB + s * kBBytes, &tB, kt * kBK, ti.n0, ti.z, &full[s]);
                    }
                }
            }
            // every copy this thread started has landed before the CTA exits
            for (int i = it > kStages ? it - kStages : 0; i < it; ++i)
                drain_wait(&full[i % kStages], (i / kStages) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = kSwap ? idesc_bf16(kBM, p.np, p.a_mn != 0, false)
                                          : idesc_bf16(kBM, kBN, false, p.b_mn != 0);
            int it = 0, lt = 0;
            bool ok = true;
            // descriptors advance by the k step: 32 bytes (2) along K for a
            // K-major operand, 16 rows (2048 bytes, 128) for an M- or N-major one
            const bool a_mn = kSwap && p.a_mn;
            const bool b_mn = !kSwap && p.b_mn;
            const uint64_t astep = a_mn ? 128 : 2;
            const uint64_t bstep = b_mn ? 128 : 2;
            for (int t = blockIdx.x; t < num_items && ok; t += gridDim.x, ++lt) {
                int tile, kt0, kt1;
                item_range(t, p.splits, nk, &tile, &kt0, &kt1);
                const int ab = lt % kAcc;
                if (!mbar_wait_fast(&acc_empty[ab], ((lt / kAcc) & 1) ^ 1, abort_flag, p.status))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(ab * kBN);
                for (int kt = kt0; kt < kt1; ++kt, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait_fast(&full[s], (it / kStages) & 1, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_mn
                                            ? sdesc(smem_u32(sA + s * kTileBytes), kTileBytes / 2, 1024, 2)
                                            : sdesc(smem_u32(sA + s * kTileBytes), 16, 1024, 2);
                    const uint64_t bd = b_mn
                                            ? sdesc(smem_u32(sB + s * kBBytes), kTileBytes / 2, 1024, 2)
                                            : sdesc(smem_u32(sB + s * kBBytes), 16, 1024, 2);
                    mma_ss(d, ad, bd, idesc, kt != kt0);
#pragma unroll
                    for (int k = 1; k < kBK / 16; ++k)
                        asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d),
                                     "l"(ad + astep * k), "l"(bd + bstep * k), "r"(idesc)
                                     : "memory");
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&acc_full[ab]);
            }
            // every MMA this thread issued has finished before the CTA exits
            tc_commit(done);
            drain_wait(done, 0);
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = tile rows
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int lt = 0;
        for (int t = blockIdx.x; t < num_items; t += gridDim.x, ++lt) {
            int tile, kt0, kt1;
            item_range(t, p.splits, nk, &tile, &kt0, &kt1);
            const int split = t % p.splits;
            const int ab = lt % kAcc;
            const TileId ti = tile_of(tile, tiles_n, tiles_m);
            const int n0 = ti.n0, z = ti.z;
            const int m = ti.m0 + row;
            bool ok = mbar_wait_fast(&acc_full[ab], (lt / kAcc) & 1, abort_flag, p.status);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (kSwap) {
                // lane = output column n; TMEM columns = activation rows
                const int n = n0 + row;
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kBN);
                __nv_bfloat16* C = (__nv_bfloat16*)p.C + (int64_t)z * p.sCz + n;
                for (int c = 0; c < p.np; c += 16) {
                    uint32_t r[16];
                    __syncwarp();
                    MLA_TMEM_LD_X16(ta + (uint32_t)c, r);
                    tmem_ld_wait();
                    if (n >= p.N) continue;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c + i < p.M) C[(int64_t)(c + i) * p.sCm] = __float2bfloat16_rn(__uint_as_float(r[i]));
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[ab]);
                continue;
            }
            int64_t slot = -1;
            if (p.splits == 1 && p.epi == 1 && m < p.M) {
                const int b = p.seq_idx[m], ps = p.pos[m];
                if (b >= 0 && b < p.batch && ps >= 0 && ps < p.max_blocks * p.block_size) {
                    const int32_t blk = p.block_table[(size_t)b * p.max_blocks + ps / p.block_size];
                    if (blk >= 0 && blk < p.num_blocks)
                        slot = (int64_t)blk * p.block_size + ps % p.block_size;
                }
                if (slot < 0 && n0 == 0) flag(p.status, MLA_ERR_INDEX);
            }
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kBN);
            for (int c = 0; c < kBN; c += 16) {
                uint32_t r[16];
                __syncwarp();
                MLA_TMEM_LD_X16(taddr + (uint32_t)c, r);
                tmem_ld_wait();
                if (m >= p.M) continue;
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
                const int nb = n0 + c;
                if (p.splits > 1) {
                    // fp32 partial of this K range; splitk_reduce_kernel finishes
                    float* P = p.partial + ((size_t)split * p.M + m) * p.N + nb;
                    if (nb + 16 <= p.N) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *(float4*)(P + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else {
                        for (int i = 0; i < 16; ++i)
                            if (nb + i < p.N) P[i] = v[i];
                    }
                } else if (p.epi == 2) {
                    if (nb >= p.N) continue;
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        if (nb + i < p.N) query_pair(p, m, nb + i, v[i], v[i + 1]);
                } else if (p.epi == 1) {
                    if (nb >= p.N) continue;
                    if (nb >= p.d_latent) {
                        const int ps = p.pos[m];
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const int j = (nb + i - p.d_latent) / 2;
                            float cs, sn;
                            rope_cos_sin(p.rope_theta1, j, ps, &cs, &sn);
                            const float x0 = v[i], x1 = v[i + 1];
                            v[i] = x0 * cs - x1 * sn;
                            v[i + 1] = x0 * sn + x1 * cs;
                        }
                    }
                    const int D = p.N;
                    __nv_bfloat16* dst = slot >= 0 ? p.cache + slot * D + nb : nullptr;
                    __nv_bfloat16* dn = p.dense_out ? p.dense_out + (size_t)m * D + nb : nullptr;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const __nv_bfloat16 h = __float2bfloat16_rn(v[i]);
                        if (dst) dst[i] = h;
                        if (dn) dn[i] = h;
                    }
                } else {
                    const int64_t base = (int64_t)z * p.sCz + (int64_t)m * p.sCm + nb;
                    if (p.c_dtype == MLA_DTYPE_BF16) {
                        __nv_bfloat16* C = (__nv_bfloat16*)p.C + base;
                        if (nb + 16 <= p.N && ((uintptr_t)C & 15) == 0) {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
                            *(uint4*)C = make_uint4(w[0], w[1], w[2], w[3]);
                            *(uint4*)(C + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (nb + i < p.N) C[i] = __float2bfloat16_rn(v[i]);
                        }
                    } else {
                        float* C = (float*)p.C + base;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (nb + i < p.N) C[i] = v[i];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[ab]);
        }
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kAcc * kBN);
}

// Sum of the split-K partials and the product's epilogue: thread = four
// consecutive columns of one row.  Same arithmetic as the one-pass epilogue
// of gemm_tc_kernel (fp32 sums, one rounding to the output type; RoPE angles
// in fp64), so a split changes only the order of the fp32 additions.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const TcGemmParams p) {
    pdl_wait_primary();
    const int n4 = p.N / 4;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < (int64_t)p.M * n4) {
        const int m = (int)(idx / n4), n = (int)(idx % n4) * 4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        const float* part = p.partial + (size_t)m * p.N + n;
        const size_t sstride = (size_t)p.M * p.N;
        // four partials' loads in flight at a time; the sum keeps split order
        int sp = 0;
        for (; sp + 4 <= p.splits; sp += 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = *(const float4*)(part + (size_t)(sp + u) * sstride);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                v[0] += x[u].x; v[1] += x[u].y; v[2] += x[u].z; v[3] += x[u].w;
            }
        }
        for (; sp < p.splits; ++sp) {
            const float4 x = *(const float4*)(part + (size_t)sp * sstride);
            v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
        }
        if (p.epi == 2) {
            query_pair(p, m, n, v[0], v[1]);
            query_pair(p, m, n + 2, v[2], v[3]);
        } else if (p.epi == 1) {
            int64_t slot = -1;
            const int b = p.seq_idx[m], ps = p.pos[m];
            if (b >= 0 && b < p.batch && ps >= 0 && ps < p.max_blocks * p.block_size) {
                const int32_t blk = p.block_table[(size_t)b * p.max_blocks + ps / p.block_size];
                if (blk >= 0 && blk < p.num_blocks)
                    slot = (int64_t)blk * p.block_size + ps % p.block_size;
            }
            if (slot < 0 && n == 0) flag(p.status, MLA_ERR_INDEX);
            if (n >= p.d_latent) {
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int j = (n + i - p.d_latent) / 2;
                    float cs, sn;
                    rope_cos_sin(p.rope_theta1, j, ps, &cs, &sn);
                    const float x0 = v[i], x1 = v[i + 1];
                    v[i] = x0 * cs - x1 * sn;
                    v[i + 1] = x0 * sn + x1 * cs;
                }
            }
            uint2 w;
            w.x = pack_bf16(v[0], v[1]);
            w.y = pack_bf16(v[2], v[3]);
            if (slot >= 0) *(uint2*)(p.cache + slot * p.N + n) = w;
            if (p.dense_out) *(uint2*)(p.dense_out + (size_t)m * p.N + n) = w;
        } else if (p.c_dtype == MLA_DTYPE_BF16) {
            uint2 w;
            w.x = pack_bf16(v[0], v[1]);
            w.y = pack_bf16(v[2], v[3]);
            *(uint2*)((__nv_bfloat16*)p.C + (int64_t)m * p.sCm + n) = w;
        } else {
            *(float4*)((float*)p.C + (int64_t)m * p.sCm + n) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
    pdl_launch_dependents();
}

// Number of K ranges for a product of `tiles` output tiles and `nk` k
// slices on `sms` SMs: the smallest count that keeps at least 85% of the
// SMs' item slots busy (items = tiles x splits, in waves of `sms`), with at
// least four k slices per range and partials that fit the scratch.
int choose_splits(int64_t tiles, int nk, int sms, size_t bytes_per_split, size_t scratch) {
    if (tiles <= 0 || scratch < bytes_per_split * 2) return 1;
    const int max_s = nk / 4 < 32 ? nk / 4 : 32;
    for (int s = 1; s <= max_s; ++s) {
        if ((size_t)s * bytes_per_split > scratch) return s > 1 ? s - 1 : 1;
        const double waves = (double)(tiles * s) / sms;
        if (waves / ceil(waves) >= 0.85) return s;
    }
    return max_s > 1 ? max_s : 1;
}

}  // namespace

size_t gemm_tc_split_scratch(int M, int N, int K, int sms) {
    if (M <= 0 || N <= 0 || K <= 0 || N % 4) return 0;
    const int64_t tiles = (int64_t)((N + kBN - 1) / kBN) * ((M + kBM - 1) / kBM);
    const size_t per = (size_t)M * N * sizeof(float);
    const int s = choose_splits(tiles, (K + kBK - 1) / kBK, sms, per, (size_t)-1 / 2);
    return s > 1 ? (size_t)s * per : 0;
}

cudaError_t launch_gemm_tc(const TcOperand& A, const TcOperand& B, const TcGemmParams& pin,
                           int batch, cudaStream_t st) {
    TcGemmParams p = pin;
    if (p.M <= 0 || p.N <= 0 || p.K <= 0 || batch <= 0) return cudaErrorInvalidValue;
    CUtensorMap ta, tb;
    const uint32_t boxA[3] = {64, 128, 1};
    const uint32_t boxBk[3] = {64, 128, 1};
    const uint32_t boxBn[3] = {64, 64, 1};
    if (!make_tmap_bf16(&ta, A.ptr, 3, A.dims, A.strides, boxA, 128)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tb, B.ptr, 3, B.dims, B.strides, p.b_mn ? boxBn : boxBk, 128))
        return cudaErrorInvalidValue;
    // the shared-memory opt-in is a per-device setting
    static bool attr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Ring<false>::smem);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    static int sms[64] = {};
    if (!sms[dev] &&
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int tiles_n = (p.N + kBN - 1) / kBN, tiles_m = (p.M + kBM - 1) / kBM;
    const int64_t tiles = (int64_t)tiles_n * tiles_m * batch;
    const int nk = (p.K + kBK - 1) / kBK;
    p.splits = 1;
    if (batch == 1 && p.partial && p.N % 4 == 0 && ((uintptr_t)p.partial & 15) == 0)
        p.splits = choose_splits(tiles, nk, sms[dev], (size_t)p.M * p.N * sizeof(float),
                                 p.partial_bytes);
    const int64_t items = tiles * p.splits;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    const int grid = (int)(items < sms[dev] ? items : sms[dev]);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = Ring<false>::smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    cudaError_t e =
        cudaLaunchKernelEx(&cfg, gemm_tc_kernel<false>, ta, tb, p, tiles_n, tiles_m, (int)items);
    if (e != cudaSuccess || p.splits == 1) return e;
    const int64_t threads = (int64_t)p.M * (p.N / 4);
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3((unsigned)((threads + 255) / 256));
    rc.blockDim = dim3(256);
    rc.stream = st;
    rc.attrs = la;
    rc.numAttrs = 1;
    return cudaLaunchKernelEx(&rc, splitk_reduce_kernel, p);
}

cudaError_t launch_gemm_tc_skinny(const TcOperand& X, const TcOperand& W, bool w_kn,
                                  const TcGemmParams& pin, int batch, cudaStream_t st) {
    TcGemmParams p = pin;
    if (p.M <= 0 || p.M > kSkinnyMaxRows || p.N <= 0 || p.K <= 0 || batch <= 0 || p.epi != 0 ||
        p.c_dtype != MLA_DTYPE_BF16)
        return cudaErrorInvalidValue;
    p.swap = 1;
    p.a_mn = w_kn ? 1 : 0;
    p.np = (p.M + 15) / 16 * 16;
    p.splits = 1;
    p.b_mn = 0;
    CUtensorMap tw, tx;
    const uint32_t boxWk[3] = {64, 128, 1};   // [n][k]: 128 columns x 64 k
    const uint32_t boxWn[3] = {64, 64, 1};    // [k][n]: 64 k rows x 64 columns, twice
    const uint32_t boxX[3] = {64, (uint32_t)p.np, 1};
    if (!make_tmap_bf16(&tw, W.ptr, 3, W.dims, W.strides, w_kn ? boxWn : boxWk, 128) ||
        !make_tmap_bf16(&tx, X.ptr, 3, X.dims, X.strides, boxX, 128))
        return cudaErrorInvalidValue;
    static bool attr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Ring<true>::smem);
        if (e != cudaSuccess) return e;
        attr[dev] = true;
    }
    static int sms[64] = {};
    if (!sms[dev] &&
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const int tiles_n = (p.N + kBM - 1) / kBM;
    const int64_t items = (int64_t)tiles_n * batch;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;
    const int grid = (int)(items < sms[dev] ? items : sms[dev]);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = Ring<true>::smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<true>, tw, tx, p, tiles_n, 1, (int)items);
}

}  // namespace mla
