// Tensor-core split-KV absorbed decode: bf16 cache, 128 heads, 512-wide
// latent, 64-wide rotary part, pages of a multiple of 64 tokens.
//
// What one decode step computes per sequence b and head h ("How DeepSeek
// Rewrote the Transformer (MLA)", section 03, applied in latent space as the
// first merge of "Multi-Head Latent Attention (MLA)" allows):
//   s_i = scale * (q_lat_h . c_i + q_pe_h . kr_i),  p = softmax(s),
//   o_lat_h = sum_i p_i c_i
// The 128 heads share every cache row, so S = Q C^T (M = 128 heads) and
// O = P C are dense contractions; they run on tcgen05 with TMEM accumulators.
//
// Layout across an SM pair.  O for 128 heads x 512 latent columns in fp32 is
// 256 KB, all of one SM's tensor memory, and the absorbed query Q (128 x 576
// bf16, 144 KB) is too large to sit next to any part of O.  A 2-CTA cluster
// therefore splits the work by kind, not by columns:
//   - the score CTA (rank 0) keeps the latent part of Q in TMEM (256 columns,
//     brought in by TMA and tcgen05.cp at the start of each sequence's range,
//     through the chunk ring except, on a worker's first range, the last two
//     groups, which use the idle P staging slot so the first cache chunk
//     starts loading with the query; the rotary part sits in shared memory)
//     and computes S = Q C^T for 128-token tiles (M=128, N=128, K=576: 36
//     MMAs) into two alternating 128-column TMEM buffers, so S(k) runs while
//     S(k-1) is read; its softmax warps turn S into bf16 P, stage P in the
//     operand layout of the next product and push it, 34 KB per tile, into
//     the value CTA's shared memory with one bulk copy;
//   - the value CTA (rank 1) keeps O in all 512 TMEM columns and computes
//     O += P C (M=128, N=256, K=128: 16 MMAs) from its own copy of the tile's
//     latent columns.
// Each CTA streams what it needs with TMA (128-byte swizzle), in large boxes
// because a TMA box costs a roughly fixed time on top of its bytes: the score
// CTA takes all 576 columns of a tile in three 48 KB chunks of three 64-column
// groups x 128 tokens (one box of a 3-D [group][row][column] view of the cache
// when the tile's two pages are adjacent in the pool, else 64-row boxes), the
// value CTA takes the 512 latent columns in four (column half, page) chunks,
// each one box of 64 rows x four 64-column groups of a 3-D view of the cache,
// which hit L2 right after the score CTA brought them in.  Only P crosses the
// cluster; distributed shared memory moves about 12 bytes per clock, so the
// fp32 partial scores of a column split (64 KB per tile each way) would not fit.
//
// Issue paths.  One thread issues every MMA of a CTA and one every TMA copy,
// and each SM sub-partition runs one of them next to two softmax or epilogue
// warps.  Two things keep those threads fast: the MMA operand descriptors are
// computed once per operand tile and advanced by constant adds (a descriptor
// computed inline before each MMA makes the tensor pipe wait for the issuing
// thread), and the hot loops are small (bounded waits keep their slow path
// out of line, the softmax walks S in four 16-column pieces), because the
// warps of a sub-partition share one small instruction cache.
//
// Softmax.  Thread h of the score CTA owns head h (TMEM lane h).  The running
// max m only moves when a tile's max exceeds it by more than 2^8; the tile's
// message then carries the factor 2^(m_old - m_new) per head and the value
// CTA rescales its O rows before adding the tile (rare, and exact because O
// and the row sum share the stale max).  The last tile of a sequence's range
// also carries the row sums, so the value CTA writes the normalised partial o
// and the score CTA its log-sum-exp (slot g + b); the merge kernel combines
// the slots.
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
constexpr int kT = 128;                  // tokens per tile
constexpr int kHalf = 64;                // rows per TMA box (a tile = two boxes)
constexpr int kBox = kHalf * 64 * 2;     // 8 KB: 64 rows x 64 columns
// score CTA ring: chunks of three 64-column groups x 128 tokens (48 KB), three
// chunks per tile (576 columns = 9 groups); a group's tile is 128 rows x 128 B
constexpr int kGroup = 2 * kBox;             // 16 KB: one 64-column group, 128 rows
constexpr int kSGroups = 3;                  // groups per chunk
constexpr int kSChunk = kSGroups * kGroup;   // 48 KB
constexpr int kSChunks = 3;                  // chunks per tile
constexpr int kSSlots = 3;
// value CTA ring: 256 columns x 64 tokens per chunk, four chunks per tile
constexpr int kVChunk = 4 * kBox;
constexpr int kVChunks = 4;
constexpr int kVSlots = 4;
constexpr int kRingBytes = kSSlots * kSChunk;
static_assert(kRingBytes >= kVSlots * kVChunk, "one ring region for both roles");
// message: P [128 heads x 128 tokens] bf16 as two K-major 128-byte-swizzled
// blocks of 64 tokens, then the per-head factors
constexpr int kPBytes = kHeads * kT * 2;   // 32 KB
constexpr int kAuxBytes = 2048;    // factors, row sums, flags, valid rows
constexpr int kMsgBytes = kPBytes + kAuxBytes;
constexpr int kMsgSlots = 2;             // value CTA: two receive slots
constexpr int kQGroups = 8;              // latent query: eight 64-column groups of 128 heads
constexpr int kQChunks = 3;              // ... in chunks of three groups (the last has two)
constexpr int kQpeBytes = kHeads * kDR * 2;   // 16 KB
constexpr int kMaxBatch = 1024;
// The score CTA stages one outgoing message at kMsgOff and keeps the rotary
// query of two consecutive ranges in the space of the second receive slot.
constexpr int kMsgOff = kRingBytes;
constexpr int kQpeOff = kMsgOff + kMsgBytes;
static_assert(2 * kQpeBytes <= kMsgBytes, "rotary query buffers");
static_assert((kQGroups - 2 * kSGroups) * kGroup <= kMsgBytes, "staged query chunk");
static_assert(kQChunks == 3 && kQGroups - 2 * kSGroups == 2, "query chunking");
constexpr int kBarOff = kMsgOff + kMsgSlots * kMsgBytes;
constexpr int kRedOff = kBarOff + 512;     // softmax exchange: [4][128] fp32
constexpr int kPreOff = kRedOff + 4 * 128 * 4;
constexpr int kLenOff = kPreOff + (kMaxBatch + 1) * 4;
constexpr int kSmemBytes = 1024 + kLenOff + kMaxBatch * 4;
constexpr int kThreads = 320;      // producer, MMA, 8 softmax / epilogue warps
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kMsgBytes % 1024 == 0, "message slots keep the 1 KB swizzle alignment");

// aux block of a message (offsets in 4-byte words after P)
constexpr int kAuxAlpha = 0;     // [128] factor applied to O rows before this tile
constexpr int kAuxSum = 128;     // [2][128] row sums of the two token halves (last tile)
constexpr int kAuxFlags = 384;   // [4] per softmax warp: some row of it rescales
constexpr int kAuxValid = 388;   // [2] valid rows of the two 64-token halves
static_assert((kAuxValid + 2) * 4 <= kAuxBytes, "aux block");

// TMEM columns
constexpr uint32_t kColQ = 0;      // score CTA: 256 columns, latent Q bf16 pairs [head][k]
constexpr uint32_t kColS = 256;    // score CTA: 2 x 128 columns, S fp32 [head][token]
constexpr uint32_t kColO = 0;      // value CTA: 512 columns, O fp32 [head][latent]
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;   // log2 units

// Optional timeline of a launch (built only with -DMLA_DECODE_TRACE): per CTA
// and tile, %globaltimer stamps of pipeline events; per CTA, its start and end.
#ifdef MLA_DECODE_TRACE
constexpr int kTraceCtas = 256, kTraceTiles = 16, kTraceEvents = 8;
__device__ unsigned long long g_decode_trace[kTraceCtas * kTraceTiles * kTraceEvents];
__device__ unsigned long long g_decode_trace_cta[kTraceCtas * 4];
#define DECODE_TRACE(ev, k)                                                              \
    do {                                                                                 \
        if ((k) < kTraceTiles && blockIdx.x < kTraceCtas)                                \
            g_decode_trace[((size_t)blockIdx.x * kTraceTiles + (k)) * kTraceEvents + (ev)] = \
                globaltimer_ns();                                                        \
    } while (0)
#define DECODE_TRACE_CTA(ev)                                                             \
    do {                                                                                 \
        if (blockIdx.x < kTraceCtas) g_decode_trace_cta[blockIdx.x * 4 + (ev)] = globaltimer_ns(); \
    } while (0)
#else
#define DECODE_TRACE(ev, k) \
    do {                    \
    } while (0)
#define DECODE_TRACE_CTA(ev) \
    do {                     \
    } while (0)
#endif

struct Bars {
    uint64_t cfull[4], cempty[4];           // chunk ring
    uint64_t s_full[2], s_empty[2];         // score CTA: S double buffer
    uint64_t qpe_full[2], qpe_free[2];      // score CTA: rotary query of a range
    uint64_t qs_full;                       // score CTA: first range's last query chunk
    uint64_t p_empty[kMsgSlots];            // score CTA: value CTA freed a message slot
    uint64_t p_full[kMsgSlots];             // value CTA: message landed
    uint64_t pv_done[kMsgSlots];            // value CTA: PV of the slot's tile finished
    uint64_t zeroed, resc_done, o_free, mma_done;
    uint64_t wg;                            // softmax-warpgroup rendezvous
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

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

// Cache rows of the two 64-token halves of tile `t0` (first token) of
// sequence b with n tokens, and how many of each half's rows are real.
// Halves past the sequence end or on an invalid page read row 0 (always in
// the pool) and count zero valid rows.
struct TileRows {
    int row[2];
    int valid[2];
};
__device__ __forceinline__ TileRows tile_rows(const DecodeArgs& a, int b, int n, int t0,
                                              bool report) {
    TileRows r;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int tok = t0 + half * kHalf;
        r.row[half] = 0;
        r.valid[half] = 0;
        if (tok < n) {
            const int32_t blk = a.block_table[(size_t)b * a.max_blocks + tok / a.block_size];
            if (blk >= 0 && blk < a.num_blocks) {
                r.row[half] = blk * a.block_size + tok % a.block_size;
                r.valid[half] = min(kHalf, n - tok);
            } else if (report) {
                flag(a.status, MLA_ERR_INDEX);
            }
        }
    }
    return r;
}

// MMA issue with precomputed operands.  A single thread issues every MMA of
// a CTA, so the instructions between two MMAs are a dependent chain on the
// issue path: descriptors are computed once per operand tile and advanced by
// adding the k step (32 bytes = 2 in the descriptor's address field, which
// cannot carry: shared addresses stay below 256 KB), and the accumulate flag
// is an immediate wherever it is known at compile time.
__device__ __forceinline__ void mma_ss_acc(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d), "l"(a), "l"(b),
                 "r"(idesc)
                 : "memory");
}
__device__ __forceinline__ void mma_ts_acc(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d), "r"(a), "l"(b),
                 "r"(idesc)
                 : "memory");
}
__device__ __forceinline__ void mma_ts_new(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc) {
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d), "r"(a), "l"(b),
                 "r"(idesc)
                 : "memory");
}

__device__ __forceinline__ void bulk_s2s(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                         uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N bulk groups of this thread still read their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap t_cache,
                     const __grid_constant__ CUtensorMap t_chunk,
                     const __grid_constant__ CUtensorMap t_page,
                     const __grid_constant__ CUtensorMap t_qlat,
                     const __grid_constant__ CUtensorMap t_qpe,
                     const __grid_constant__ CUtensorMap t_qlat2,
                     const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;
    uint8_t* msg = smem + kMsgOff;
    Bars* bars = (Bars*)(smem + kBarOff);
    int* pre = (int*)(smem + kPreOff);
    int* lens = (int*)(smem + kLenOff);
    volatile int* abort_flag = &bars->abort_flag;
    const uint64_t wl = a.wait_ns;          // give-up time of the pipeline waits

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool scorer = rank == 0;
    const int g = blockIdx.x >> 1;
    const int cap = a.max_blocks * a.block_size;

    if (threadIdx.x == 0) {
        DECODE_TRACE_CTA(0);
        for (int s = 0; s < 4; ++s) {
            mbar_init(&bars->cfull[s], 1);
            mbar_init(&bars->cempty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->s_empty[s], 256);
            mbar_init(&bars->qpe_full[s], 1);
            mbar_init(&bars->qpe_free[s], 1);
        }
        for (int s = 0; s < kMsgSlots; ++s) {
            mbar_init(&bars->p_empty[s], 8);     // one remote arrive per value-CTA warp
            mbar_init(&bars->p_full[s], 1);      // local expect_tx + the bulk copy
            mbar_init(&bars->pv_done[s], 1);
        }
        mbar_init(&bars->zeroed, 256);
        mbar_init(&bars->resc_done, 256);
        mbar_init(&bars->o_free, 256);
        mbar_init(&bars->mma_done, 1);
        mbar_init(&bars->qs_full, 1);
        mbar_init(&bars->wg, 256);
        bars->abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&t_cache);
        prefetch_tmap(&t_chunk);
        prefetch_tmap(&t_page);
        prefetch_tmap(&t_qlat);
        prefetch_tmap(&t_qpe);
        prefetch_tmap(&t_qlat2);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // Everything above overlaps the previous kernel's tail.  Inputs are read,
    // and global memory is written, only after this wait: the workspace (or
    // mla_decode_noalloc's static array) of the previous call on the stream is
    // still being read by that call's merge kernel until then, so no global
    // write (partials, lse, the published slot ranges) may move above it.
    pdl_wait_primary();
    tile_prefix(a.seq_lens, a.batch, cap, pre, scorer ? a.status : nullptr, lens, kT);
    if (blockIdx.x == 0) publish_seq_slots(pre, a.batch, a.workers, a.seq_slots);
    tc_fence_before();
    cluster_sync();        // both CTAs' barriers exist before any remote access
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
            int c = 0, seg = 0;
            bool ok = true, staged = false;
            const uint64_t evict_first = policy_evict_first();
            auto ring_slot = [&](int slots, int bytes) -> int {
                const int s = c % slots;
                if (!mbar_wait_fast(&bars->cempty[s], ((c / slots) & 1) ^ 1, abort_flag,
                                    a.status, wl)) {
                    ok = false;
                    return -1;
                }
                mbar_arrive_expect_tx(&bars->cfull[s], bytes);
                return s;
            };
            for (int k = 0; k < K && ok; ++k, cur.next()) {
                const int t0 = cur.tile_in_seq() * kT;
                if (scorer) {
                    if (cur.first(lo)) {
                        // the range's query: the rotary part into its own buffer
                        // (free once the previous use's products are done), the
                        // latent part through the ring for tcgen05.cp into TMEM
                        const int qb = seg & 1;
                        if (!mbar_wait_fast(&bars->qpe_free[qb], ((seg >> 1) & 1) ^ 1,
                                            abort_flag, a.status, wl))
                            break;
                        mbar_arrive_expect_tx(&bars->qpe_full[qb], kQpeBytes);
                        tma_load_2d(smem + kQpeOff + qb * kQpeBytes, &t_qpe, 0, cur.b * kHeads,
                                    &bars->qpe_full[qb]);
                        // the first range's last query chunk (two groups) goes to
                        // the P staging slot, idle until the first P, so that the
                        // tile's first cache chunk takes its ring slot at once
                        const bool stage_q = seg == 0;
                        ++seg;
                        for (int j = 0; j < kQChunks && ok; ++j) {
                            if (stage_q && j == kQChunks - 1) {
                                mbar_arrive_expect_tx(&bars->qs_full, 2 * kGroup);
                                tma_load_3d(msg, &t_qlat2, 0, cur.b * kHeads, kSGroups * j,
                                            &bars->qs_full);
                                staged = true;
                                continue;
                            }
                            // three groups per box; the last box's third group
                            // lies past the query row and is zero-filled
                            const int s = ring_slot(kSSlots, kSChunk);
                            if (s < 0) break;
                            tma_load_3d(ring + s * kSChunk, &t_qlat, 0, cur.b * kHeads,
                                        kSGroups * j, &bars->cfull[s]);
                            ++c;
                        }
                        if (!ok) break;
                    }
                    // the tile's pages: a block-table read, issued after the
                    // range's query copies so that their latency covers it
                    const TileRows tr = tile_rows(a, cur.b, lens[cur.b], t0, true);
                    // the two pages of the tile in one 128-row box when they are
                    // adjacent in the pool (fewer, larger TMA requests), else one
                    // 64-row box each; the shared-memory image is the same
                    const bool adjacent = tr.valid[1] > 0 && tr.row[1] == tr.row[0] + kHalf;
                    for (int j = 0; j < kSChunks && ok; ++j, ++c) {
                        const int s = ring_slot(kSSlots, kSChunk);
                        if (s < 0) break;
                        uint8_t* dst = ring + s * kSChunk;
                        if (adjacent) {
                            tma_load_3d(dst, &t_chunk, 0, tr.row[0], kSGroups * j, &bars->cfull[s]);
                        } else {
                            for (int gg = 0; gg < kSGroups; ++gg) {
                                const int x = 64 * (kSGroups * j + gg);
                                tma_load_2d(dst + gg * kGroup, &t_cache, x, tr.row[0],
                                            &bars->cfull[s]);
                                tma_load_2d(dst + gg * kGroup + kBox, &t_cache, x, tr.row[1],
                                            &bars->cfull[s]);
                            }
                        }
                    }
                } else {
                    const TileRows tr = tile_rows(a, cur.b, lens[cur.b], t0, false);
                    // one box per chunk: 64 rows of a page x four 64-column
                    // groups.  This is the last read of these rows: their L2
                    // lines go first, ahead of the partials, queries and weights
                    // that are read again
                    for (int j = 0; j < kVChunks && ok; ++j, ++c) {
                        const int s = ring_slot(kVSlots, kVChunk);
                        if (s < 0) break;
                        tma_load_3d_hint(ring + s * kVChunk, &t_page, 0, tr.row[j & 1],
                                         4 * (j >> 1), &bars->cfull[s], evict_first);
                    }
                }
            }
            // every copy this thread started has landed before the CTA exits
            const int slots = scorer ? kSSlots : kVSlots;
            for (int i = c > slots ? c - slots : 0; i < c; ++i)
                drain_wait(&bars->cfull[i % slots], (i / slots) & 1);
            if (scorer)
                for (int i = seg > 2 ? seg - 2 : 0; i < seg; ++i)
                    drain_wait(&bars->qpe_full[i & 1], (i >> 1) & 1);
            if (staged) drain_wait(&bars->qs_full, 0);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && K > 0) {
            Cursor cur;
            cur.init(pre, a.batch, lo);
            bool ok = true;
            if (scorer) {
                // S = Q C^T, K = 576 in nine 64-column chunks of four k-steps
                const uint32_t id_s = idesc_bf16(128, kT, false, false);
                int c = 0, seg = 0, qb = 0;
                for (int k = 0; k < K && ok; ++k, cur.next()) {
                    if (cur.first(lo)) {
                        // new range: its latent query chunks into TMEM (in order
                        // after the previous range's products), then its rotary
                        // part; the first range's last chunk comes from the
                        // staging slot (the softmax warps write P there only
                        // after S(0), whose commit covers this copy)
                        const bool staged = seg == 0;
                        for (int j = 0; j < kQChunks; ++j) {
                            const bool from_staging = staged && j == kQChunks - 1;
                            const int s = c % kSSlots;
                            uint64_t* full = from_staging ? &bars->qs_full : &bars->cfull[s];
                            const uint32_t par = from_staging ? 0u : (uint32_t)((c / kSSlots) & 1);
                            if (!mbar_wait_fast(full, par, abort_flag, a.status, wl)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t st = smem_u32(from_staging ? msg : ring + s * kSChunk);
                            for (int gg = 0; gg < kSGroups; ++gg) {
                                const int qg = kSGroups * j + gg;
                                if (qg >= kQGroups) break;
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    tmem_cp_128x256b(tmem + kColQ + 32 * qg + 8 * kk,
                                                     sdesc(st + gg * kGroup + 32 * kk, 16, 1024, 2));
                            }
                            if (!from_staging) {
                                tc_commit(&bars->cempty[s]);
                                ++c;
                            }
                        }
                        if (!ok) break;
                        qb = seg & 1;
                        if (!mbar_wait_fast(&bars->qpe_full[qb], (seg >> 1) & 1, abort_flag,
                                            a.status, wl))
                            break;
                        ++seg;
                    }
                    const int sb = k & 1;   // S buffer: the softmax warps read S(k-1) meanwhile
                    if (!mbar_wait_fast(&bars->s_empty[sb], ((k >> 1) & 1) ^ 1, abort_flag,
                                        a.status, wl))
                        break;
                    tc_fence_after();
                    const uint32_t d_s = tmem + kColS + 128 * sb;
                    const uint32_t qa = smem_u32(smem + kQpeOff + qb * kQpeBytes);
                    for (int j = 0; j < kSChunks; ++j, ++c) {
                        const int s = c % kSSlots;
                        if (!mbar_wait_fast(&bars->cfull[s], (c / kSSlots) & 1, abort_flag,
                                            a.status, wl)) {
                            ok = false;
                            break;
                        }
                        DECODE_TRACE(j, k);
                        tc_fence_after();
                        const uint64_t b0 = sdesc(smem_u32(ring + s * kSChunk), 16, 1024, 2);
                        if (j == 0) {
                            // chunk 0: groups 0-2, the tile's first MMA starts the sum
                            const uint32_t a0 = tmem + kColQ;
                            mma_ts_new(d_s, a0, b0, id_s);
#pragma unroll
                            for (int q = 1; q < 12; ++q)
                                mma_ts_acc(d_s, a0 + 8 * q, b0 + (uint64_t)(q >> 2) * 1024 + 2 * (q & 3), id_s);
                        } else if (j == 1) {
                            const uint32_t a0 = tmem + kColQ + 32 * kSGroups;
#pragma unroll
                            for (int q = 0; q < 12; ++q)
                                mma_ts_acc(d_s, a0 + 8 * q, b0 + (uint64_t)(q >> 2) * 1024 + 2 * (q & 3), id_s);
                        } else {
                            // groups 6, 7 (latent) and 8 (rotary part, Q_pe from shared memory)
                            const uint32_t a0 = tmem + kColQ + 32 * 2 * kSGroups;
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                mma_ts_acc(d_s, a0 + 8 * q, b0 + (uint64_t)(q >> 2) * 1024 + 2 * (q & 3), id_s);
                            const uint64_t qd = sdesc(qa, 16, 1024, 2);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss_acc(d_s, qd + 2 * kk, b0 + 2048 + 2 * kk, id_s);
                        }
                        tc_commit(&bars->cempty[s]);
                    }
                    if (!ok) break;
                    tc_commit(&bars->s_full[sb]);
                    DECODE_TRACE(3, k);
                    if (cur.last(hi)) tc_commit(&bars->qpe_free[qb]);
                }
            } else {
                // O += P C, per column half: K = 128 tokens = two 64-token chunks
                const uint32_t id_pv = idesc_bf16(128, 256, false, true);
                int c = 0, seg = 0, resc = 0, zer = 0;
                for (int k = 0; k < K && ok; ++k, cur.next()) {
                    const int slot = k % kMsgSlots;
                    const bool first = cur.first(lo);
                    mbar_arrive_expect_tx(&bars->p_full[slot], kMsgBytes);
                    if (!mbar_wait_fast<true>(&bars->p_full[slot], (k / kMsgSlots) & 1,
                                              abort_flag, a.status, wl))
                        break;
                    DECODE_TRACE(0, k);
                    const uint8_t* m = msg + slot * kMsgBytes;
                    const int* aux = (const int*)(m + kPBytes);
                    const bool need_resc =
                        !first && (aux[kAuxFlags] | aux[kAuxFlags + 1] | aux[kAuxFlags + 2] |
                                   aux[kAuxFlags + 3]) != 0;
                    const bool partial = aux[kAuxValid] < kHalf || aux[kAuxValid + 1] < kHalf;
                    if (first && seg > 0 &&
                        !mbar_wait_fast(&bars->o_free, (seg - 1) & 1, abort_flag, a.status, wl))
                        break;
                    if (need_resc &&
                        !mbar_wait_fast(&bars->resc_done, (resc++) & 1, abort_flag, a.status, wl))
                        break;
                    if (partial &&
                        !mbar_wait_fast(&bars->zeroed, (zer++) & 1, abort_flag, a.status, wl))
                        break;
                    tc_fence_after();
                    const uint64_t pdesc = sdesc(smem_u32(m), 16, 1024, 2);
                    for (int j = 0; j < kVChunks; ++j, ++c) {
                        const int s = c % kVSlots, hh = j >> 1, pg = j & 1;
                        if (!mbar_wait_fast(&bars->cfull[s], (c / kVSlots) & 1, abort_flag,
                                            a.status, wl)) {
                            ok = false;
                            break;
                        }
                        if (j == 0) DECODE_TRACE(1, k);
                        if (j == kVChunks - 1) DECODE_TRACE(2, k);
                        tc_fence_after();
                        const uint64_t bd = sdesc(smem_u32(ring + s * kVChunk), kBox, 1024, 2);
                        const uint64_t ad = pdesc + (uint64_t)pg * (kPBytes / 2 / 16);
                        const uint32_t dst = tmem + kColO + 256 * hh;
                        if (pg == 0)
                            mma_ss(dst, ad, bd, id_pv, first ? 0 : 1);
                        else
                            mma_ss_acc(dst, ad, bd, id_pv);
#pragma unroll
                        for (int i = 1; i < 4; ++i) mma_ss_acc(dst, ad + 2 * i, bd + 128 * i, id_pv);
                        tc_commit(&bars->cempty[s]);
                    }
                    if (!ok) break;
                    tc_commit(&bars->pv_done[slot]);
                    DECODE_TRACE(3, k);
                    if (cur.last(hi)) ++seg;
                }
            }
            tc_commit(&bars->mma_done);
            drain_wait(&bars->mma_done, 0);
        }
    } else if (K > 0) {
        // warps 2-9: two threads per head.  TMEM lanes are reachable from the
        // warps with the same (warp % 4), so warps w and w+4 share head
        // h = 32 (w % 4) + lane; `half` picks 64 of the tile's 128 tokens (score
        // CTA) or 256 of the 512 latent columns (value CTA).
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;
        const int h = q4 * 32 + lane;                 // head = TMEM lane
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int tid = threadIdx.x - 64;             // 0..255
        Cursor cur;
        cur.init(pre, a.batch, lo);
        if (scorer) {
            // ------------------------------------------ softmax warpgroup
            const float c2 = a.scale * 1.4426950408889634f;   // log2(e) / sqrt(d)
            const uint32_t msg_peer = mapa(smem_u32(msg), 1);
            const uint32_t pfull_peer = mapa(smem_u32(&bars->p_full[0]), 1);
            float* red = (float*)(smem + kRedOff);     // [2][128] per-half tile max

            // rendezvous of the 256 softmax threads: an mbarrier with a bounded
            // wait, so a timeout anywhere releases everyone
            uint32_t wg_phase = 0;
            auto wg_sync = [&]() -> bool {
                mbar_arrive(&bars->wg);
                return mbar_wait_fast(&bars->wg, (wg_phase++) & 1, abort_flag, a.status, wl);
            };

            float m = -INFINITY, l = 0.f;     // m: running max (log2 units); l: this half's sum
            for (int k = 0; k < K; ++k, cur.next()) {
                const int b = cur.b;
                const bool first = cur.first(lo), last = cur.last(hi);
                const TileRows tr = tile_rows(a, b, lens[b], cur.tile_in_seq() * kT, false);
                const int nv = tr.valid[half];          // valid tokens of this thread's 64
                const int buf = k % kMsgSlots;

                // ---- this thread's 64 scores, read from TMEM in four 16-column
                // pieces: a first pass takes the maximum, a second one the
                // weights (runtime loops keep this hot code small)
                const int sb = k & 1;
                if (!mbar_wait_fast(&bars->s_full[sb], (k >> 1) & 1, abort_flag, a.status, wl))
                    break;
                if (tid == 0) DECODE_TRACE(4, k);
                tc_fence_after();
                const uint32_t src = tmem + lane_off + kColS + 128 * sb + 64 * half;
                float mloc = -INFINITY;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t r[16];
                    MLA_TMEM_LD_X16(src + 16 * c4, r);
                    tmem_ld_wait();
                    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const float v0 = 16 * c4 + i < nv ? __uint_as_float(r[i]) : -INFINITY;
                        const float v1 = 16 * c4 + i + 1 < nv ? __uint_as_float(r[i + 1]) : -INFINITY;
                        mx0 = fmaxf(mx0, v0);
                        mx1 = fmaxf(mx1, v1);
                    }
                    mloc = fmaxf(mloc, fmaxf(mx0, mx1));
                }
                // the staging buffer is free once the copy of tile k-1 read it
                if (tid == 0) bulk_wait_read<0>();
                red[half * kHeads + h] = mloc;
                if (!wg_sync()) break;
                const float mt = fmaxf(mloc, red[(half ^ 1) * kHeads + h]) * c2;

                // ---- online softmax (log2 domain), lazy rescale; both threads
                // of a head take the same decisions from the same values
                const bool grow = mt > m + kRescaleThreshold;
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2(m - mt);    // 0 when m = -inf
                    l *= alpha;
                    m = mt;
                }
                const bool resc = grow && !first;

                // ---- P: bf16 weights, two 16-byte chunks (16 tokens) per piece,
                // in the 128-byte-swizzled K-major layout of the PV operand
                uint8_t* mb = msg;     // the one staging buffer
                uint8_t* row = mb + half * (kPBytes / 2) + h * 128;
                const float nm = m == -INFINITY ? 0.f : -m;   // all-masked tile: p = 0
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t r[16];
                    MLA_TMEM_LD_X16(src + 16 * c4, r);
                    tmem_ld_wait();
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int t = 16 * c4 + 2 * i;
                        // tokens past the valid ones weigh 0
                        const float p0 = t < nv ? ex2(fmaf(__uint_as_float(r[2 * i]), c2, nm)) : 0.f;
                        const float p1 = t + 1 < nv ? ex2(fmaf(__uint_as_float(r[2 * i + 1]), c2, nm)) : 0.f;
                        ps0 += p0;
                        ps1 += p1;
                        w[i] = pack_bf16(p0, p1);
                    }
                    const int cc = 2 * c4;
                    *(uint4*)(row + ((cc ^ (h & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *(uint4*)(row + (((cc + 1) ^ (h & 7)) * 16)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                tc_fence_before();
                mbar_arrive(&bars->s_empty[sb]);
                l += ps0 + ps1;

                float* aux = (float*)(mb + kPBytes);
                if (half == 0) {
                    aux[kAuxAlpha + h] = resc ? alpha : 1.f;
                    const bool any = __any_sync(0xffffffffu, resc);
                    if (lane == 0) ((int*)aux)[kAuxFlags + q4] = any ? 1 : 0;
                }
                if (last) aux[kAuxSum + half * kHeads + h] = l;
                if (tid == 0) {
                    ((int*)aux)[kAuxValid] = tr.valid[0];
                    ((int*)aux)[kAuxValid + 1] = tr.valid[1];
                }
                fence_proxy_async();
                if (last) red[kHeads * 2 + half * kHeads + h] = l;
                if (!wg_sync()) break;
                if (tid == 0 && mbar_wait_fast<true>(&bars->p_empty[buf],
                                                     ((k / kMsgSlots) & 1) ^ 1, abort_flag,
                                                     a.status, wl)) {
                    DECODE_TRACE(5, k);
                    bulk_s2s(msg_peer + buf * kMsgBytes, smem_u32(mb), kMsgBytes,
                             pfull_peer + 8 * buf);
                    bulk_commit();
                    DECODE_TRACE(6, k);
                }
                if (last) {
                    if (half == 0) {
                        const float lt = l + red[kHeads * 3 + h];
                        a.lse_part[((size_t)g + b) * kHeads + h] =
                            lt > 0.f ? (m + __log2f(lt)) * 0.6931471805599453f : -INFINITY;
                    }
                    m = -INFINITY;
                    l = 0.f;
                }
            }
            if (tid == 0) bulk_wait_all();
        } else {
            // ------------------------------------------ value-CTA warpgroup:
            // rare O rescales, zeroing of rows past a sequence end, the
            // normalised partial at the end of a range (thread: head h,
            // latent columns [256 half, 256 half + 256))
            const uint32_t pempty_peer = mapa(smem_u32(&bars->p_empty[0]), 0);
            const uint32_t col0 = kColO + 256 * half;
            int c = 0;
            for (int k = 0; k < K; ++k, cur.next()) {
                const int slot = k % kMsgSlots;
                const bool first = cur.first(lo), last = cur.last(hi);
                const int b = cur.b;
                if (!mbar_wait_fast<true>(&bars->p_full[slot], (k / kMsgSlots) & 1, abort_flag,
                                          a.status, wl))
                    break;
                const float* aux = (const float*)(msg + slot * kMsgBytes + kPBytes);
                const int* auxi = (const int*)aux;
                const float alpha = aux[kAuxAlpha + h];
                const bool need_resc = !first && (auxi[kAuxFlags] | auxi[kAuxFlags + 1] |
                                                  auxi[kAuxFlags + 2] | auxi[kAuxFlags + 3]) != 0;
                const int v0 = auxi[kAuxValid], v1 = auxi[kAuxValid + 1];
                float inv_l = 0.f;
                if (last) {
                    const float lt = aux[kAuxSum + h] + aux[kAuxSum + kHeads + h];
                    inv_l = lt > 0.f ? 1.f / lt : 0.f;
                }
                bool ok = true;
                if (need_resc) {
                    // O must hold every earlier tile of this range: PV(k-1) done
                    const int pk_ = k - 1;
                    ok = mbar_wait_fast(&bars->pv_done[pk_ % kMsgSlots], (pk_ / kMsgSlots) & 1,
                                        abort_flag, a.status, wl);
                    if (!ok) break;
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
                        uint32_t r[32];
#pragma unroll 1
                        for (int cc = 0; cc < 256; cc += 32) {
                            MLA_TMEM_LD_X32(tmem + lane_off + col0 + cc, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            MLA_TMEM_ST_X32(tmem + lane_off + col0 + cc, r);
                        }
                        tmem_st_wait();
                    }
                    tc_fence_before();
                    mbar_arrive(&bars->resc_done);
                }
                if (v0 < kHalf || v1 < kHalf) {
                    // rows past the sequence end (or on an invalid page) hold
                    // arbitrary bytes: zero them so 0 * garbage cannot reach O
                    for (int j = 0; j < kVChunks && ok; ++j) {
                        const int cj = c + j, s = cj % kVSlots, pg = j & 1;
                        const int valid = pg ? v1 : v0;
                        if (valid >= kHalf) continue;
                        ok = mbar_wait_fast(&bars->cfull[s], (cj / kVSlots) & 1, abort_flag,
                                            a.status, wl);
                        if (!ok) break;
                        uint8_t* st = ring + s * kVChunk;
                        const int rows = kHalf - valid;
                        for (int e = tid; e < rows * 4 * 8; e += 256) {
                            const int box = e / (rows * 8), rem = e % (rows * 8);
                            const int row = valid + rem / 8, ch = rem % 8;
                            *(uint4*)(st + box * kBox + row * 128 + ch * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async();
                    mbar_arrive(&bars->zeroed);
                }
                c += kVChunks;
                if (!mbar_wait_fast(&bars->pv_done[slot], (k / kMsgSlots) & 1, abort_flag,
                                    a.status, wl))
                    break;
                if (tid == 0) DECODE_TRACE(4, k);
                if (last) {
                    // ---- the range's normalised partial.  A warp holds a
                    // 32-head x 32-column block per TMEM load (one row per
                    // thread); it goes through 4 KB of the consumed message slot
                    // so that each store instruction writes whole 128-byte rows.
                    tc_fence_after();
                    float* xb = (float*)(msg + slot * kMsgBytes) + (warp - 2) * 1024;
                    float* dst0 = a.o_part + (((size_t)g + b) * kHeads + q4 * 32) * kDL +
                                  256 * half;
                    uint32_t r[32];
#pragma unroll 1
                    for (int cc = 0; cc < 256; cc += 32) {
                        MLA_TMEM_LD_X32(tmem + lane_off + col0 + cc, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *(float4*)(xb + lane * 32 + 4 * (i ^ (lane & 7))) =
                                make_float4(__uint_as_float(r[4 * i]) * inv_l,
                                            __uint_as_float(r[4 * i + 1]) * inv_l,
                                            __uint_as_float(r[4 * i + 2]) * inv_l,
                                            __uint_as_float(r[4 * i + 3]) * inv_l);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = 4 * i + (lane >> 3), ch = lane & 7;
                            *(float4*)(dst0 + (size_t)rr * kDL + cc + 4 * ch) =
                                *(const float4*)(xb + rr * 32 + 4 * (ch ^ (rr & 7)));
                        }
                        __syncwarp();
                    }
                    fence_proxy_async();   // the next bulk copy into this slot comes after
                    tc_fence_before();
                    if (tid == 0) DECODE_TRACE(5, k);
                    mbar_arrive(&bars->o_free);
                }
                // the message slot (P and its factors) may be overwritten now
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(pempty_peer + 8 * slot);
            }
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncwarp();
    __syncthreads();
    cluster_sync();        // the peer no longer writes our smem or barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

struct DeviceState {
    bool init = false;
    bool attr = false;
    int major = 0;
    int workers = 0;
};
constexpr int kMaxDev = 64;
DeviceState g_dev[kMaxDev];

DeviceState* device_state() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess)
            return nullptr;
        d.attr = cudaFuncSetAttribute(decode_tc_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kSmemBytes) == cudaSuccess;
        cudaGetLastError();
        d.init = true;
    }
    return &d;
}

}  // namespace

bool decode_tc_supported(int heads, int d_latent, int d_rope, int block_size, int dtype,
                         int batch) {
    if (heads != kHeads || d_latent != kDL || d_rope != kDR || dtype != MLA_DTYPE_BF16)
        return false;
    if (block_size % kHalf != 0 || batch > kMaxBatch) return false;
    DeviceState* d = device_state();
    return d && d->major >= 10 && d->attr;
}

int decode_tc_tile() { return kT; }

#ifdef MLA_DECODE_TRACE
extern "C" int mla_decode_trace_copy(unsigned long long* tiles, unsigned long long* ctas) {
    cudaDeviceSynchronize();
    if (cudaMemcpyFromSymbol(tiles, g_decode_trace, sizeof(g_decode_trace)) != cudaSuccess ||
        cudaMemcpyFromSymbol(ctas, g_decode_trace_cta, sizeof(g_decode_trace_cta)) != cudaSuccess)
        return 1;
    return 0;
}
#endif

// Clusters that can be resident at once (pairs of SMs within one GPC), at most
// one per SM pair.  Computed once per device.
int decode_tc_workers(int num_sms) {
    int w = num_sms / 2 > 0 ? num_sms / 2 : 1;
    DeviceState* d = device_state();
    if (!d || !d->attr) return w;
    if (d->workers > 0) return d->workers;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * w);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) == cudaSuccess && n > 0 &&
        n < w)
        w = n;
    cudaGetLastError();   // a refused query is not an error of the caller's
    d->workers = w;
    return w;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
    if ((uint64_t)a.num_blocks * a.block_size > 0x7fffffffull) return cudaErrorInvalidValue;
    if (!a.cache || ((uintptr_t)a.q_lat & 15) || ((uintptr_t)a.q_pe & 15) || a.tile != kT)
        return cudaErrorInvalidValue;
    DeviceState* d = device_state();
    if (!d || !d->attr) return cudaErrorNotSupported;
    CUtensorMap t_cache, t_chunk, t_page, t_qlat, t_qpe, t_qlat2;
    const uint64_t rows = (uint64_t)a.num_blocks * a.block_size;
    // cache rows, 64 x 64 boxes
    const uint64_t dims[2] = {(uint64_t)kD, rows};
    const uint64_t strides[1] = {(uint64_t)kD * 2};
    const uint32_t box[2] = {64, kHalf};
    // the same rows seen as [64-column group][row][64 columns]: one box holds
    // 64 rows of four groups, each group a 128-byte-swizzled 64 x 64 tile
    const uint64_t dims3[3] = {64, rows, (uint64_t)kD / 64};
    const uint64_t strides3[2] = {(uint64_t)kD * 2, 128};
    const uint32_t box3[3] = {64, kHalf, 4};
    const uint32_t boxc[3] = {64, kT, kSGroups};     // score chunk: 128 rows x 3 groups
    // queries: [batch * heads] rows of 512 latent / 64 rotary values; the
    // latent part seen as [group][row][64 columns] like the cache
    const uint64_t qrows = (uint64_t)a.batch * kHeads;
    const uint64_t dq[3] = {64, qrows, (uint64_t)kQGroups};
    const uint64_t sq[2] = {(uint64_t)kDL * 2, 128};
    const uint32_t bq3[3] = {64, kHeads, kSGroups};
    const uint32_t bq2[3] = {64, kHeads, kQGroups - 2 * kSGroups};   // last two groups
    const uint64_t dp[2] = {(uint64_t)kDR, qrows}, sp[1] = {(uint64_t)kDR * 2};
    const uint32_t bq[2] = {64, kHeads};
    if (!make_tmap_bf16(&t_cache, a.cache, 2, dims, strides, box, 128) ||
        !make_tmap_bf16(&t_chunk, a.cache, 3, dims3, strides3, boxc, 128) ||
        !make_tmap_bf16(&t_page, a.cache, 3, dims3, strides3, box3, 128) ||
        !make_tmap_bf16(&t_qlat, a.q_lat, 3, dq, sq, bq3, 128) ||
        !make_tmap_bf16(&t_qpe, a.q_pe, 2, dp, sp, bq, 128) ||
        !make_tmap_bf16(&t_qlat2, a.q_lat, 3, dq, sq, bq2, 128))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * a.workers);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel, t_cache, t_chunk, t_page, t_qlat, t_qpe,
                              t_qlat2, a);
}

}  // namespace mla
