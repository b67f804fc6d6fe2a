/*
 * mla.h -- C ABI of libmla.so, Multi-Head Latent Attention (MLA) decode on
 * NVIDIA B300 (sm_103a).
 *
 * What is computed (row-vector notation of "Multi-Head Latent Attention
 * (MLA)", section "The construction"):
 *   every cached token i keeps ONE row [c_i | kr_i] shared by all heads:
 *     c_i  = x_i W_L               latent, d_latent values
 *     kr_i = RoPE(x_i W_KR, i)     decoupled rotary key part, d_rope values
 *   a decode step for the newest token t of a sequence of n tokens computes,
 *   per head h, attention of its query over the n cached rows
 *     s_i   = scale * (q_lat_h . c_i + q_pe_h . kr_i),  i = 0..n-1
 *     p     = softmax(s)
 *     o_lat_h = sum_i p_i c_i
 *   where q_lat_h = q_nope_h W_LK_h^T is the query pre-multiplied by the
 *   head's latent-to-key weights (the first merge of "Two merges are where
 *   the compute win comes from"), and the head output is o_lat_h W_LV_h,
 *   stacked over heads and multiplied by W_O (the second merge).  Per-head
 *   keys and values are never formed.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE memory owned by the caller, row-major,
 *     of the element type given by mla_config.dtype unless stated otherwise
 *     (int32 index arrays, float32 log-sum-exp and partial outputs).  The
 *     library never allocates device memory; scratch space is passed in.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream)
 *     and returns an mla_status.  Host-side validation failures launch
 *     nothing.  Faults that only the device can see (a block id outside the
 *     pool, a sequence length out of range) are recorded in a per-device
 *     status word; the offending rows are skipped, never read out of bounds.
 *     Read and clear it with mla_get_status().
 *   - No C++ exception crosses this boundary.
 *   - Weights use the [in][out] layout of the row-vector formulas: a vector
 *     times W_X means  y[j] = sum_k x[k] * W_X[k][j].
 *   - Paged cache: `cache` is [num_blocks][block_size][d_latent + d_rope].
 *     Logical token i of sequence b lives in row
 *       block_table[b * max_blocks + i / block_size] * block_size + i % block_size.
 *     ("MLA: how DeepSeek cuts KV cache memory", section "Where MLA sits in
 *     the taxonomy": paged cache management.)
 *   - Positions: key i of a sequence sits at position i; the sequence's
 *     current (query) token sits at position seq_len - 1, so decode attends
 *     to rows 0..seq_len-1 (the causal mask of section 03 of "How DeepSeek
 *     Rewrote the Transformer (MLA)" for the newest row, section 04).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* mla_stream_t; /* same object as cudaStream_t */

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1, /* bad pointer, size, or configuration value        */
    MLA_ERR_UNSUPPORTED = 2, /* valid, but a shape/dtype the library cannot run  */
    MLA_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small       */
    MLA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed             */
    MLA_ERR_TIMEOUT = 5,     /* device: a bounded wait in a kernel gave up       */
    MLA_ERR_INDEX = 6        /* device: a block id or sequence index was invalid */
} mla_status;

typedef enum mla_dtype { MLA_DTYPE_BF16 = 0, MLA_DTYPE_F32 = 1 } mla_dtype;

/*
 * Shapes and parameters of one MLA layer.
 *   heads       H, number of attention heads (128 for DeepSeek-V2 shapes)
 *   d_latent    d_L, latent width shared by keys and values (512)
 *   d_rope      d_R, decoupled rotary key/query width, even (64)
 *   d_nope      d_n, per-head query/key width on the latent side (128)
 *   d_v         per-head value width (128)
 *   block_size  tokens per cache page
 *   dtype       element type of cache, queries, weights and outputs
 *   softmax_scale  multiplies q.k before the softmax ("divide by the square
 *               root of the dimension": 1/sqrt(d_n + d_R) is the usual value)
 *   rope_base   base of the rotary frequencies theta_j = rope_base^(-2j/d_R)
 *               (rotation of interleaved pairs (2j, 2j+1) by pos * theta_j)
 */
typedef struct mla_config {
    int heads;
    int d_latent;
    int d_rope;
    int d_nope;
    int d_v;
    int block_size;
    int dtype;
    float softmax_scale;
    double rope_base;
} mla_config;

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(int status);

/* Library ABI version: MAJOR * 10000 + MINOR * 100 + PATCH. */
int mla_version(void);

/*
 * Which decode kernel mla_decode runs for `cfg`: 1 = tensor-core kernel
 * (tcgen05/TMEM, TMA-fed), 0 = CUDA-core kernel (fp32 FMA; fp32 configs and
 * shapes the tensor-core kernel does not take), -1 = invalid config.
 */
int mla_decode_path(const mla_config* cfg);

/*
 * Diagnostic: how long a pipeline wait inside the tensor-core decode kernel
 * may last before the kernel gives up (default 1 s; ns <= 0 restores it).
 * A kernel that gives up records MLA_ERR_TIMEOUT in the status word, lets
 * its copies land, waits for its tensor-core operations, frees its tensor
 * memory and returns, so the next call on the device runs normally.  The
 * value applies to decode calls issued afterwards from any thread.  It exists
 * so that tests can make the give-up path run; the pages describe nothing
 * like it.  Always returns MLA_OK.
 */
int mla_set_wait_limit_ns(int64_t ns);

/*
 * Reads and clears the current device's status word (see above).  Waits for
 * `stream` to finish first.  *out receives MLA_OK or the first device-side
 * error recorded since the last call.
 */
int mla_get_status(mla_stream_t stream, int* out);

/*
 * Down-projects new tokens into cache rows and writes them to their paged
 * slots ("The construction": L = X W_L; "The RoPE problem": the rotary part
 * is kept apart from the latent; "How DeepSeek Rewrote the Transformer
 * (MLA)", section 04: appending leaves every earlier row untouched).
 *   x            [n_tok][d_in]                   hidden states of the new tokens
 *   w_dkv        [d_in][d_latent + d_rope]       [W_L | W_KR]
 *   seq_idx      [n_tok] int32                   sequence of each token, in [0, batch)
 *   pos          [n_tok] int32                   position of each token in its sequence
 *   block_table  [batch][max_blocks] int32
 *   cache        [num_blocks][block_size][d_latent + d_rope]   (written)
 *   dense_out    [n_tok][d_latent + d_rope] or NULL: also receives each row,
 *                bit-identical to what is written into the cache
 * Row t = [x_t W_L | RoPE(x_t W_KR, pos_t)], accumulated in fp32, rotary
 * angles in fp64, rounded once to dtype.  Tokens whose slot is invalid are
 * skipped and flagged MLA_ERR_INDEX on the device.
 */
int mla_append_latent(const mla_config* cfg, const void* x, int n_tok, int d_in,
                      const void* w_dkv, const int32_t* seq_idx, const int32_t* pos,
                      const int32_t* block_table, int batch, int max_blocks, void* cache,
                      int64_t num_blocks, void* dense_out, mla_stream_t stream);

/*
 * Query absorption, the first merge of "Two merges are where the compute win
 * comes from" (section of "Multi-Head Latent Attention (MLA)"):
 *   q_lat[b][h][:] = q_nope[b][h][:] . W_LK_h^T
 *   q_nope  [batch][heads][d_nope]
 *   w_uk    [heads][d_latent][d_nope]   W_LK_h maps a latent to the head's key
 *   q_lat   [batch][heads][d_latent]    (written; fp32 accumulation)
 */
int mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* w_uk, int batch,
                 void* q_lat, mla_stream_t stream);

/*
 * Bytes of scratch that mla_decode needs for `batch` sequences on the current
 * device (split-KV partial results).  The size depends only on the config,
 * the batch and the device, never on sequence lengths.
 */
int mla_decode_workspace_size(const mla_config* cfg, int batch, size_t* bytes);

/*
 * Absorbed decode attention over the shared latent cache, for one new query
 * token per sequence (section 03 steps of "How DeepSeek Rewrote the
 * Transformer (MLA)" applied in latent space; section 04: only the newest
 * query row is computed).
 *   q_lat        [batch][heads][d_latent]   absorbed query (mla_absorb_q)
 *   q_pe         [batch][heads][d_rope]     rotary query part, already rotated
 *   cache        [num_blocks][block_size][d_latent + d_rope]
 *   block_table  [batch][max_blocks] int32
 *   seq_lens     [batch] int32, attended tokens incl. the current one, >= 1
 *   o_lat        [batch][heads][d_latent]   (written) sum_i p_i c_i
 *   lse          [batch][heads] float32 or NULL: natural-log log-sum-exp of
 *                the scaled scores
 *   workspace    >= mla_decode_workspace_size() bytes, 256-byte aligned
 * The context is split into ranges that keep every SM busy; each range
 * yields a partial (o, lse) pair that a combine kernel merges.  The result
 * does not depend on how the ranges fall, up to rounding.
 */
int mla_decode(const mla_config* cfg, const void* q_lat, const void* q_pe, const void* cache,
               int64_t num_blocks, const int32_t* block_table, int max_blocks,
               const int32_t* seq_lens, int batch, void* o_lat, float* lse, void* workspace,
               size_t ws_bytes, mla_stream_t stream);

/*
 * Decode of several new query tokens per sequence at once (a chunk of
 * prefill, or the tokens a speculative step proposes): the last q_tokens
 * tokens of each sequence, token j at position seq_lens[b] - q_tokens + j,
 * each attending to the cached rows up to and including its own position
 * (the causal mask of section 03 of "How DeepSeek Rewrote the Transformer
 * (MLA)"; section 04: with one token this is mla_decode).  The rows of the
 * new tokens must already be in the cache.
 *   q_lat   [batch][q_tokens][heads][d_latent]   absorbed queries
 *   q_pe    [batch][q_tokens][heads][d_rope]     rotary parts, rotated at each token's position
 *   seq_lens [batch] int32, tokens including the q_tokens new ones, >= q_tokens
 *   o_lat   [batch][q_tokens][heads][d_latent]   (written)
 *   lse     [batch][q_tokens][heads] float32 or NULL
 *   workspace >= mla_decode_multi_workspace_size() bytes, 256-byte aligned
 *   1 <= q_tokens <= 64, batch * q_tokens <= 8192.
 * Each token is decoded as its own row of the split-KV plan, with the
 * sequence's block table; the rows of one sequence are adjacent in the plan,
 * so workers reading the same cache tiles run at about the same time and
 * most repeated reads hit L2 (16 sequences of 4096 tokens, 4 new tokens
 * each: 1.6 times the cache bytes read from HBM).
 */
int mla_decode_multi_workspace_size(const mla_config* cfg, int batch, int q_tokens,
                                    int max_blocks, size_t* bytes);
int mla_decode_multi(const mla_config* cfg, const void* q_lat, const void* q_pe,
                     const void* cache, int64_t num_blocks, const int32_t* block_table,
                     int max_blocks, const int32_t* seq_lens, int batch, int q_tokens,
                     void* o_lat, float* lse, void* workspace, size_t ws_bytes,
                     mla_stream_t stream);

/*
 * Merges partial decode results computed over disjoint token ranges of the
 * same sequences (e.g. ranges held by different devices):
 *   LSE = log sum_s exp(lse_s),  o = sum_s exp(lse_s - LSE) o_s.
 *   o_part    [n_splits][batch][heads][d_latent] float32, 1 <= n_splits <= 512
 *   lse_part  [n_splits][batch][heads] float32; -inf marks an empty range
 *   o_lat     [batch][heads][d_latent] (written, dtype); all-empty rows give 0
 *   lse       [batch][heads] float32 or NULL (written)
 */
int mla_decode_combine(const mla_config* cfg, const float* o_part, const float* lse_part,
                       int n_splits, int batch, void* o_lat, float* lse, mla_stream_t stream);

/*
 * Output side, the second merge: o_v[b][h] = o_lat[b][h] . W_LV_h, then
 * out[b] = concat_h(o_v[b][h]) . W_O (section 03: stack the heads and
 * multiply by W_O).
 *   o_lat  [batch][heads][d_latent]
 *   w_uv   [heads][d_latent][d_v]
 *   o_v    [batch][heads][d_v]             (written)
 *   w_o    [heads * d_v][d_model] or NULL  (then `out` is not written)
 *   out    [batch][d_model]                (written when w_o != NULL)
 */
int mla_project_out(const mla_config* cfg, const void* o_lat, const void* w_uv, int batch,
                    void* o_v, const void* w_o, int d_model, void* out, mla_stream_t stream);

/*
 * Query of the current tokens ("Latent Space Strikes Again", "The Core
 * Idea": optional query compression; "Multi-Head Latent Attention (MLA)":
 * W_Q = W_LQ W_LQQ plus a rotary query part per head):
 *   c_q = x W_DQ (skipped when w_dq == NULL: c_q = x)
 *   [q_nope_h | r_h] = c_q W_UQ_h,  q_pe_h = RoPE(r_h, pos_b)
 *   x       [batch][d_in]
 *   w_dq    [d_in][d_lq] or NULL
 *   w_uq    [d_q][heads][d_nope + d_rope]   d_q = d_lq, or d_in without w_dq
 *   pos     [batch] int32
 *   q_nope  [batch][heads][d_nope], q_pe [batch][heads][d_rope]  (written)
 *   scratch >= mla_query_proj_workspace_size() bytes, 256-byte aligned
 */
int mla_query_proj_workspace_size(const mla_config* cfg, int batch, int d_lq, size_t* bytes);
int mla_query_proj(const mla_config* cfg, const void* x, int batch, int d_in, const void* w_dq,
                   int d_lq, const void* w_uq, const int32_t* pos, void* q_nope, void* q_pe,
                   void* scratch, size_t scratch_bytes, mla_stream_t stream);

/*
 * Whole decode steps in one call.  Each issues, on `stream`, every kernel of
 * one step in the order of section 03 of "How DeepSeek Rewrote the
 * Transformer (MLA)" (queries, scores against the cached rows, softmax,
 * weighted sum, stack the heads and multiply by W_O), in latent space as the
 * two merges of "Multi-Head Latent Attention (MLA)" allow, with the newest
 * token's cache row appended first (section 04: the step reads every earlier
 * row and adds one).  The intermediate tensors live in the caller's
 * workspace.
 *
 * io_flags: MLA_IO_HOST_INPUTS means the per-step inputs (x or q_nope / q_pe,
 * seq_lens and block_table) are pinned host memory and are copied to the
 * workspace on `stream` before the first kernel; MLA_IO_HOST_OUTPUT means
 * the result (out or o_v) is pinned host memory written by a copy after the
 * last kernel.  Without the flags every pointer is device memory.  Weights
 * and the cache are always device memory.
 */
#define MLA_IO_HOST_INPUTS 1
#define MLA_IO_HOST_OUTPUT 2

/*
 * Weights of one MLA layer (device memory, dtype of the config, [in][out]):
 *   w_dkv  [d_model][d_latent + d_rope]      [W_L | W_KR], the cache row of x
 *   w_dq   [d_model][d_lq] or NULL            query compression W_LQ
 *   w_uq   [d_q][heads][d_nope + d_rope]      per head [W_LQQ_h | W_QR_h],
 *                                             d_q = d_lq, or d_model without w_dq
 *   w_uk   [heads][d_latent][d_nope]          W_LK_h
 *   w_uv   [heads][d_latent][d_v]             W_LV_h
 *   w_o    [heads * d_v][d_model]             W_O
 */
typedef struct mla_layer_weights {
    int d_model;
    int d_lq;
    const void* w_dkv;
    const void* w_dq;
    const void* w_uq;
    const void* w_uk;
    const void* w_uv;
    const void* w_o;
} mla_layer_weights;

/*
 * Full decode step of one layer for one new token per sequence:
 *   row b of the cache at position seq_lens[b] - 1 = [x_b W_L | RoPE(x_b W_KR)]
 *   (mla_append_latent), the query of x_b at the same position
 *   (mla_query_proj), q_lat (mla_absorb_q), attention over rows
 *   0 .. seq_lens[b] - 1 (mla_decode), out_b = concat_h(o_lat W_LV_h) W_O
 *   (mla_project_out).
 *   x         [batch][d_model]   hidden state of each sequence's new token
 *   seq_lens  [batch] int32      tokens including the new one, >= 1
 *   cache     [num_blocks][block_size][d_latent + d_rope]  (new rows written)
 *   out       [batch][d_model]   (written)
 *   workspace >= mla_layer_decode_step_workspace_size() bytes, 256-byte aligned
 * Errors are those of the calls above; nothing is launched when host-side
 * validation fails.
 */
int mla_layer_decode_step_workspace_size(const mla_config* cfg, const mla_layer_weights* w,
                                         int batch, int max_blocks, size_t* bytes);
int mla_layer_decode_step(const mla_config* cfg, const mla_layer_weights* w, const void* x,
                          const int32_t* seq_lens, int batch, void* cache, int64_t num_blocks,
                          const int32_t* block_table, int max_blocks, void* out, int io_flags,
                          void* workspace, size_t ws_bytes, mla_stream_t stream);

/*
 * Decode step over a cache whose rows are given (no new row, no W_O):
 * q_lat = q_nope W_LK_h^T (mla_absorb_q), attention (mla_decode) and
 * o_v[b][h] = o_lat[b][h] W_LV_h (mla_project_out without W_O).
 *   q_nope [batch][heads][d_nope], q_pe [batch][heads][d_rope]
 *   o_v    [batch][heads][d_v]                     (written)
 *   o_lat  [batch][heads][d_latent] or NULL         device, written when given
 *   lse    [batch][heads] float32 or NULL           device, written when given
 */
int mla_cached_decode_step_workspace_size(const mla_config* cfg, int batch, int max_blocks,
                                          size_t* bytes);
int mla_cached_decode_step(const mla_config* cfg, const void* q_nope, const void* q_pe,
                           const void* w_uk, const void* w_uv, const int32_t* seq_lens,
                           int batch, const void* cache, int64_t num_blocks,
                           const int32_t* block_table, int max_blocks, void* o_v, void* o_lat,
                           float* lse, int io_flags, void* workspace, size_t ws_bytes,
                           mla_stream_t stream);

/*
 * mla_decode without a workspace argument: the split-KV partial results go to
 * a static device array of MLA_NOALLOC_SCRATCH_BYTES that the library itself
 * holds on every GPU that loads it, until the process exits.  The pages
 * describe no such call; it exists for callers that cannot allocate device
 * memory at the point where they decode (a framework that owns all device
 * memory through its own pool and forbids direct cudaMalloc, a plugin
 * interface that passes only inputs and outputs, or a latency-critical loop
 * where an allocation's implicit device synchronisation is not allowed).
 *
 * Arguments and results are those of mla_decode.  The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *   - Limit: the array must hold the partials of at least one worker plus one
 *     per sequence, (1 + batch) * heads * (d_latent + 1) * 4 bytes, and 16
 *     bytes per sequence, each part rounded up to 256 bytes.  Larger requests return MLA_ERR_UNSUPPORTED and
 *     launch nothing.  When the array is smaller than what mla_decode would
 *     use, the context is split into fewer ranges (same result up to rounding).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its partials
 *     there.  Nothing in it has to start at zero.  Calls that overlap on the
 *     GPU (concurrent streams, or several host threads) race on the array and
 *     give wrong results: serialise them.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
int mla_decode_noalloc(const mla_config* cfg, const void* q_lat, const void* q_pe,
                       const void* cache, int64_t num_blocks, const int32_t* block_table,
                       int max_blocks, const int32_t* seq_lens, int batch, void* o_lat,
                       float* lse, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
