// Tensor-core split-KV absorbed decode: bf16 cache, 128 heads, 512-wide
// latent, 64-wide rotary part, pages of a multiple of 64 tokens.
//
// What one decode step computes per sequence b and head h ("How DeepSeek
// Rewrote the Transformer (MLA)", section 03, applied in latent space as the
// first merge of "Multi-Head Latent Attention (MLA)" allows):
//   s_i = scale * (q_lat_h . c_i + q_pe_h . kr_i),  p = softmax(s),
//   o_lat_h = sum_i p_i c_i
// The 128 heads share every cache row, so S = Q C^T (M = 128 heads) and
// O = P C are dense contractions and run on tcgen05 with TMEM accumulators.
//
// Work split.  The 64-token tiles of all sequences, laid end to end, are cut
// into W equal ranges; each range goes to a cluster of two CTAs.  CTA r of the
// pair owns latent columns [256r, 256r+256) and rotary columns
// [512+32r, 512+32r+32), so the pair reads each cache row exactly once:
//   - TMA streams CTA r's 288 columns of each 64-token tile into a 5-stage
//     ring (four 64x64 boxes, 128-byte swizzle, plus one 64x32 box, 64-byte
//     swizzle);
//   - one thread issues S_r = Q_r C_r^T (M=128, N=64, 18 k-steps, Q_r held in
//     TMEM as the A operand) into TMEM;
//   - the softmax warpgroup (thread = head) reads S_r, swaps it with the
//     partner through distributed shared memory, and both CTAs form
//     S = S_0 + S_1 in the same order, so they take bit-identical softmax
//     decisions; the running max is only moved when a row's tile max exceeds
//     it by more than 2^8 (rescaling O in TMEM is then rare and exact, since O
//     and the row sum share the stale max); P (bf16) goes back into TMEM;
//   - the same thread issues O_r += P C_r (M=128, N=256, 4 k-steps, C_r read
//     N-major from the same smem stage), so O_r lives in 256 TMEM columns.
// A range that ends a sequence writes the normalised partial o and its
// log-sum-exp to slot g + b; the merge kernel combines the slots.
//
// Every wait is bounded (see tc_ptx.cuh); on a timeout the kernel records
// MLA_ERR_TIMEOUT, lets its copies land, frees TMEM and returns.
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace mla {

namespace {

using namespace tc;

constexpr int kHeads = 128, kDL = 512, kDR = 64, kD = kDL + kDR;
constexpr int kT = 64;                 // tokens per tile
constexpr int kStages = 5;
constexpr int kLatBox = kT * 64 * 2;   // 8 KB: 64 tokens x 64 latent columns
constexpr int kRopeBox = kT * 32 * 2;  // 4 KB: 64 tokens x 32 rotary columns
constexpr int kStageBytes = 4 * kLatBox + kRopeBox;   // 36 KB
constexpr int kXBytes = kHeads * kT * 4;               // 32 KB partial-score swap
constexpr int kMaxBatch = 1024;
constexpr int kBarOff = kStages * kStageBytes + kXBytes;
constexpr int kPreOff = kBarOff + 256;
constexpr int kSmemBytes = 1024 + kPreOff + (kMaxBatch + 1) * 4;
constexpr int kThreads = 192;

// TMEM columns
constexpr uint32_t kColO = 0;      // 256: O_r, fp32 [head][latent col]
constexpr uint32_t kColQ = 256;    // 144: Q_r, bf16 pairs [head][k]
constexpr uint32_t kColS = 400;    // 64:  S_r, fp32 [head][token]
constexpr uint32_t kColP = 464;    // 32:  P, bf16 pairs [head][token]
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;   // log2 units

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t s_full, s_empty, p_full, p_empty, q_ready, o_free, x_full, x_empty, mma_done;
    uint32_t tmem_slot;
    int abort_flag;
};

// Walks the tiles of one worker range in order.
struct Cursor {
    const int* pre;
    int batch;
    int b;
    int64_t t;
    __device__ void init(const int* p, int nb, int64_t lo) {
        pre = p;
        batch = nb;
        t = lo;
        b = seq_of_tile(p, nb, lo);
        while (b + 1 < nb && pre[b + 1] <= t) ++b;
    }
    __device__ void next() {
        ++t;
        while (b + 1 < batch && pre[b + 1] <= t) ++b;
    }
    __device__ int tile_in_seq() const { return (int)(t - pre[b]); }
    __device__ bool first(int64_t lo) const { return t == lo || t == pre[b]; }
    __device__ bool last(int64_t hi) const { return t + 1 == hi || t + 1 == pre[b + 1]; }
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap t_lat,
                     const __grid_constant__ CUtensorMap t_rope, const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* X = (float*)(smem + kStages * kStageBytes);
    Bars* bars = (Bars*)(smem + kBarOff);
    int* pre = (int*)(smem + kPreOff);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int g = blockIdx.x >> 1;
    const int cap = a.max_blocks * a.block_size;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_empty, 128);
        mbar_init(&bars->p_full, 128);
        mbar_init(&bars->p_empty, 1);
        mbar_init(&bars->q_ready, 128);
        mbar_init(&bars->o_free, 128);
        mbar_init(&bars->x_full, 128);
        mbar_init(&bars->x_empty, 128);
        mbar_init(&bars->mma_done, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&t_lat);
        prefetch_tmap(&t_rope);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tile_prefix(a.seq_lens, a.batch, cap, pre, a.status);   // ends with __syncthreads
    tc_fence_before();
    cluster_sync();        // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    const int64_t total = pre[a.batch];
    const int64_t lo = plan_lo(g, total, a.workers), hi = plan_lo(g + 1, total, a.workers);
    const int K = (int)(hi - lo);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && K > 0) {
            Cursor cur;
            cur.init(pre, a.batch, lo);
            int issued = 0;
            for (int k = 0; k < K; ++k, cur.next()) {
                const int s = k % kStages;
                if (!mbar_wait(&bars->empty[s], ((k / kStages) & 1) ^ 1, abort_flag, a.status))
                    break;
                const int tok = cur.tile_in_seq() * kT;
                int32_t blk = a.block_table[(size_t)cur.b * a.max_blocks + tok / a.block_size];
                if (blk < 0 || blk >= a.num_blocks) {
                    flag(a.status, MLA_ERR_INDEX);
                    blk = 0;   // load a valid page; the softmax masks the whole tile
                }
                const int y = blk * a.block_size + tok % a.block_size;
                uint8_t* st = smem + s * kStageBytes;
                mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    tma_load_2d(st + i * kLatBox, &t_lat, 256 * rank + 64 * i, y, &bars->full[s]);
                tma_load_2d(st + 4 * kLatBox, &t_rope, kDL + 32 * rank, y, &bars->full[s]);
                issued = k + 1;
            }
            for (int k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
                drain_wait(&bars->full[k % kStages], (k / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && K > 0) {
            const uint32_t id_s = idesc_bf16(128, kT, false, false);
            const uint32_t id_pv = idesc_bf16(128, 256, false, true);
            Cursor cur, pvc;
            cur.init(pre, a.batch, lo);
            pvc.init(pre, a.batch, lo);
            int seg = 0, pv_seg = 0;
            bool ok = true;
            auto issue_pv = [&](int k) -> bool {
                const int s = k % kStages;
                const bool first = pvc.first(lo);
                if (first && pv_seg > 0 &&
                    !mbar_wait(&bars->o_free, (pv_seg - 1) & 1, abort_flag, a.status))
                    return false;
                if (!mbar_wait(&bars->p_full, k & 1, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
                for (int i = 0; i < kT / 16; ++i) {
                    const uint64_t bd = sdesc(st + 2048 * i, kLatBox, 1024, 2);
                    mma_ts(tmem + kColO, tmem + kColP + 8 * i, bd, id_pv,
                           (first && i == 0) ? 0 : 1);
                }
                tc_commit(&bars->empty[s]);
                tc_commit(&bars->p_empty);
                if (pvc.last(hi)) ++pv_seg;
                pvc.next();
                return true;
            };
            for (int k = 0; k < K && ok; ++k, cur.next()) {
                const int s = k % kStages;
                if (cur.first(lo) && !mbar_wait(&bars->q_ready, seg & 1, abort_flag, a.status))
                    break;
                if (!mbar_wait(&bars->full[s], (k / kStages) & 1, abort_flag, a.status)) break;
                if (!mbar_wait(&bars->s_empty, (k & 1) ^ 1, abort_flag, a.status)) break;
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * kStageBytes);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t bd = sdesc(st + (i >> 2) * kLatBox + 32 * (i & 3), 16, 1024, 2);
                    mma_ts(tmem + kColS, tmem + kColQ + 8 * i, bd, id_s, i > 0);
                }
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint64_t bd = sdesc(st + 4 * kLatBox + 32 * i, 16, 512, 4);
                    mma_ts(tmem + kColS, tmem + kColQ + 128 + 8 * i, bd, id_s, 1);
                }
                tc_commit(&bars->s_full);
                if (k > 0) ok = issue_pv(k - 1);
                if (cur.last(hi)) ++seg;
                if (ok && k == K - 1) ok = issue_pv(k);
            }
            tc_commit(&bars->mma_done);
            drain_wait(&bars->mma_done, 0);
        }
    } else {
        // ------------------------------------------------ softmax warpgroup
        const int q4 = warp & 3;
        const int h = q4 * 32 + lane;                 // head = TMEM lane
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int tid = threadIdx.x - 64;             // 0..127
        const float c2 = a.scale * 1.4426950408889634f;
        const uint32_t x_local = smem_u32(X);
        const uint32_t x_peer = mapa(x_local, peer);
        const uint32_t xfull_peer = mapa(smem_u32(&bars->x_full), peer);
        const uint32_t xempty_peer = mapa(smem_u32(&bars->x_empty), peer);
        const __nv_bfloat16* qlat = (const __nv_bfloat16*)a.q_lat;
        const __nv_bfloat16* qpe = (const __nv_bfloat16*)a.q_pe;

        auto load_q = [&](int b) {
            const uint4* src = (const uint4*)(qlat + ((size_t)b * kHeads + h) * kDL + 256 * rank);
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
                uint4 v0 = src[2 * c], v1 = src[2 * c + 1];
                uint32_t r[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                MLA_TMEM_ST_X8(tmem + lane_off + kColQ + 8 * c, r);
            }
            const uint4* sp = (const uint4*)(qpe + ((size_t)b * kHeads + h) * kDR + 32 * rank);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint4 v0 = sp[2 * c], v1 = sp[2 * c + 1];
                uint32_t r[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                MLA_TMEM_ST_X8(tmem + lane_off + kColQ + 128 + 8 * c, r);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->q_ready);
        };

        if (K > 0) {
            Cursor cur;
            cur.init(pre, a.batch, lo);
            load_q(cur.b);
            float m = -INFINITY, l = 0.f;
            for (int k = 0; k < K; ++k, cur.next()) {
                const bool first = cur.first(lo), last = cur.last(hi);
                const int b = cur.b;
                const int n = clamp_len(a.seq_lens[b], cap, nullptr);
                const int tok = cur.tile_in_seq() * kT;
                int n_valid = min(kT, n - tok);
                const int32_t blk = a.block_table[(size_t)b * a.max_blocks + tok / a.block_size];
                if (blk < 0 || blk >= a.num_blocks) n_valid = 0;

                // ---- partial scores S_r
                if (!mbar_wait(&bars->s_full, k & 1, abort_flag, a.status)) break;
                tc_fence_after();
                float sv[kT];
                {
                    uint32_t r[16];
#pragma unroll
                    for (int c = 0; c < kT; c += 16) {
                        MLA_TMEM_LD_X16(tmem + lane_off + kColS + c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) sv[c + i] = __uint_as_float(r[i]);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->s_empty);

                // ---- swap partial scores with the peer CTA
                if (!mbar_wait<true>(&bars->x_empty, (k & 1) ^ 1, abort_flag, a.status)) break;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int pc = c ^ (h & 7);
                    st_cluster_v4(x_peer + (uint32_t)((h * kT + 4 * pc) * 4), sv[4 * c],
                                  sv[4 * c + 1], sv[4 * c + 2], sv[4 * c + 3]);
                }
                mbar_arrive_remote(xfull_peer);
                if (!mbar_wait<true>(&bars->x_full, k & 1, abort_flag, a.status)) break;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int pc = c ^ (h & 7);
                    const float4 o = *(const float4*)(X + h * kT + 4 * pc);
                    // S = S_0 + S_1 in this order on both CTAs
                    if (rank == 0) {
                        sv[4 * c] += o.x; sv[4 * c + 1] += o.y;
                        sv[4 * c + 2] += o.z; sv[4 * c + 3] += o.w;
                    } else {
                        sv[4 * c] = o.x + sv[4 * c]; sv[4 * c + 1] = o.y + sv[4 * c + 1];
                        sv[4 * c + 2] = o.z + sv[4 * c + 2]; sv[4 * c + 3] = o.w + sv[4 * c + 3];
                    }
                }
                mbar_arrive_remote(xempty_peer);

                // the next segment's query may replace Q now: S(k) is done
                if (last && k + 1 < K) {
                    Cursor nx = cur;
                    nx.next();
                    load_q(nx.b);
                }

                // ---- online softmax (log2 domain), lazy rescale
                float mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < kT; ++i) {
                    const float v = (i < n_valid) ? sv[i] * c2 : -INFINITY;
                    sv[i] = v;
                    mt = fmaxf(mt, v);
                }
                const bool grow = mt > m + kRescaleThreshold;
                float alpha = 1.f;
                if (grow) {
                    alpha = exp2f(m - mt);    // 0 when m = -inf
                    l *= alpha;
                    m = mt;
                }
                if (!first && __any_sync(0xffffffffu, grow)) {
                    // O must hold every earlier PV of this segment: PV(k-1) done
                    if (!mbar_wait(&bars->p_empty, (k - 1) & 1, abort_flag, a.status)) break;
                    tc_fence_after();
                    uint32_t r[16];
                    for (int c = 0; c < 256; c += 16) {
                        MLA_TMEM_LD_X16(tmem + lane_off + kColO + c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        MLA_TMEM_ST_X16(tmem + lane_off + kColO + c, r);
                    }
                    tmem_st_wait();
                }
                uint32_t pk[kT / 2];
                float ps = 0.f;
#pragma unroll
                for (int i = 0; i < kT; i += 2) {
                    const float p0 = (sv[i] == -INFINITY) ? 0.f : exp2f(sv[i] - m);
                    const float p1 = (sv[i + 1] == -INFINITY) ? 0.f : exp2f(sv[i + 1] - m);
                    ps += p0 + p1;
                    pk[i / 2] = pack_bf16(p0, p1);
                }
                l += ps;

                // ---- rows past the sequence end hold arbitrary bytes: zero
                // them so 0 * garbage cannot reach O
                if (n_valid < kT) {
                    uint8_t* st = smem + (k % kStages) * kStageBytes;
                    const int rows = kT - n_valid;
                    for (int e = tid; e < rows * 4 * 8; e += 128) {
                        const int box = e / (rows * 8), rem = e % (rows * 8);
                        const int row = n_valid + rem / 8, ch = rem % 8;
                        *(uint4*)(st + box * kLatBox + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async();
                }

                // ---- P into TMEM once PV(k-1) has read the previous P
                if (!mbar_wait(&bars->p_empty, (k & 1) ^ 1, abort_flag, a.status)) break;
                tc_fence_after();
                MLA_TMEM_ST_X16(tmem + lane_off + kColP, pk);
                MLA_TMEM_ST_X16(tmem + lane_off + kColP + 16, (pk + 16));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars->p_full);

                if (last) {
                    // ---- segment done: normalised partial and its lse
                    if (!mbar_wait(&bars->p_empty, k & 1, abort_flag, a.status)) break;
                    tc_fence_after();
                    const size_t slot = (size_t)g + b;
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    float* dst = a.o_part + (slot * kHeads + h) * kDL + 256 * rank;
                    uint32_t r[16];
                    for (int c = 0; c < 256; c += 16) {
                        MLA_TMEM_LD_X16(tmem + lane_off + kColO + c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *(float4*)(dst + c + i) =
                                make_float4(__uint_as_float(r[i]) * inv,
                                            __uint_as_float(r[i + 1]) * inv,
                                            __uint_as_float(r[i + 2]) * inv,
                                            __uint_as_float(r[i + 3]) * inv);
                    }
                    if (rank == 0)
                        a.lse_part[slot * kHeads + h] =
                            l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
                    tc_fence_before();
                    mbar_arrive(&bars->o_free);
                    m = -INFINITY;
                    l = 0.f;
                }
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();        // the peer no longer writes our smem or barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool decode_tc_supported(int heads, int d_latent, int d_rope, int block_size, int dtype,
                         int batch) {
    if (heads != kHeads || d_latent != kDL || d_rope != kDR || dtype != MLA_DTYPE_BF16)
        return false;
    if (block_size % kT != 0 || batch > kMaxBatch) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    return major >= 10;
}

// Clusters that can be resident at once (pairs of SMs within one GPC), at most
// one per SM pair.
int decode_tc_workers(int num_sms) {
    int w = num_sms / 2 > 0 ? num_sms / 2 : 1;
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
        return w;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * w);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) == cudaSuccess && n > 0 &&
        n < w)
        w = n;
    cudaGetLastError();   // a refused query is not an error of the caller's
    return w;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
    if ((uint64_t)a.num_blocks * a.block_size > 0x7fffffffull) return cudaErrorInvalidValue;
    if (!a.cache || ((uintptr_t)a.q_lat & 15) || ((uintptr_t)a.q_pe & 15))
        return cudaErrorInvalidValue;
    CUtensorMap t_lat, t_rope;
    const uint64_t rows = (uint64_t)a.num_blocks * a.block_size;
    const uint64_t dims[2] = {(uint64_t)kD, rows};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box_lat[2] = {64, kT};
    const uint32_t box_rope[2] = {32, kT};
    if (!make_tmap_bf16(&t_lat, a.cache, 2, dims, strides, box_lat, 128))
        return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&t_rope, a.cache, 2, dims, strides, box_rope, 64))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    decode_tc_kernel<<<2 * a.workers, kThreads, kSmemBytes, st>>>(t_lat, t_rope, a);
    return cudaGetLastError();
}

}  // namespace mla
