// C ABI of libmla.so: argument validation, workspace carving and kernel
// launches.  Every entry point is declared, with its contract, in mla.h.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

using namespace mla;

namespace {

// Device-side error word (first error wins).  Its device address is looked
// up once per device and handed to the kernels as a plain pointer.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Give-up time of the decode kernels' pipeline waits (mla_set_wait_limit_ns).
constexpr uint64_t kDefaultWaitNs = 1000ull * 1000ull * 1000ull;
uint64_t g_wait_ns = kDefaultWaitNs;

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices)
        return MLA_ERR_CUDA;
    return MLA_OK;
}

int status_ptr(int** out) {
    int dev;
    if (int rc = current_device(&dev)) return rc;
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MLA_ERR_CUDA;
        g_status_ptr[dev] = (int*)p;
    }
    *out = g_status_ptr[dev];
    return MLA_OK;
}

int num_sms(int* out) {
    int dev;
    if (int rc = current_device(&dev)) return rc;
    if (!g_num_sms[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MLA_ERR_CUDA;
        g_num_sms[dev] = v;
    }
    *out = g_num_sms[dev];
    return MLA_OK;
}

int check_cfg(const mla_config* c) {
    if (!c) return MLA_ERR_INVALID_ARG;
    if (c->heads < 1 || c->heads > 1024) return MLA_ERR_INVALID_ARG;
    if (c->d_latent < 1 || c->d_latent > 4096) return MLA_ERR_INVALID_ARG;
    if (c->d_rope < 0 || c->d_rope > 1024 || (c->d_rope & 1)) return MLA_ERR_INVALID_ARG;
    if (c->d_nope < 1 || c->d_nope > 4096 || c->d_v < 1 || c->d_v > 4096)
        return MLA_ERR_INVALID_ARG;
    if (c->block_size < 1 || c->block_size > (1 << 20)) return MLA_ERR_INVALID_ARG;
    if (c->dtype != MLA_DTYPE_BF16 && c->dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARG;
    if (!isfinite(c->softmax_scale) || !isfinite(c->rope_base) || c->rope_base <= 0.0)
        return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}


int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// Frequency of the first RoPE pair, rope_base^(-2 / d_rope); pair j turns
// by theta1^j per position (interleaved pairs, theta_j = base^(-2j/d_rope)).
double rope_theta1(const mla_config* c) {
    return c->d_rope > 0 ? pow(c->rope_base, -2.0 / (double)c->d_rope) : 1.0;
}

constexpr int kMaxDecodeBatch = 8192;

// The tensor-core kernel takes the maximum of the raw scores, which needs a
// positive softmax scale; other scales go to the CUDA-core kernel.
bool use_tc(const mla_config* c, int batch) {
    return c->softmax_scale > 0.f &&
           decode_tc_supported(c->heads, c->d_latent, c->d_rope, c->block_size, c->dtype, batch);
}

// Split-KV worker count of the decode kernel that (c, batch) selects.
int decode_workers(const mla_config* c, int batch, int* W) {
    int sms;
    if (int rc = num_sms(&sms)) return rc;
    *W = use_tc(c, batch) ? decode_tc_workers(sms) : sms;
    return MLA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Per-head products with at most this many rows run transposed (weights as
// the MMA's 128-row side): the rows would otherwise fill a small part of it.
constexpr int kSkinnyRows = 64;

bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// 3-D bf16 operand view for the tensor-core GEMM.
TcOperand op3(const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
              uint64_t s2_bytes) {
    TcOperand o;
    o.ptr = ptr;
    o.dims[0] = d0; o.dims[1] = d1; o.dims[2] = d2;
    o.strides[0] = s1_bytes; o.strides[1] = s2_bytes;
    return o;
}

// fp32 scratch a projection may use for split-K partials (none: one pass)
struct SplitScratch {
    float* ptr = nullptr;
    size_t bytes = 0;
};

TcGemmParams gemm_params(int M, int N, int K, bool b_mn, void* C, int64_t sCz, int64_t sCm,
                         int c_dtype, int* status, SplitScratch sp = SplitScratch{}) {
    TcGemmParams g{};
    g.M = M; g.N = N; g.K = K; g.b_mn = b_mn ? 1 : 0; g.epi = 0;
    g.C = C; g.sCz = sCz; g.sCm = sCm; g.c_dtype = c_dtype; g.status = status;
    g.partial = sp.ptr; g.partial_bytes = sp.bytes;
    return g;
}

// Workspace of a decode call: split-KV partials (W + batch slots of
// heads x d_latent fp32), their log-sum-exps, and per sequence the range of
// workers that produced its partials (int4).
size_t decode_ws_bytes(const mla_config* c, int W, int batch) {
    size_t slots = (size_t)W + (size_t)batch;
    return align256(slots * c->heads * c->d_latent * sizeof(float)) +
           align256(slots * c->heads * sizeof(float)) + align256((size_t)batch * 16);
}

// Points the partial, lse and slot-range arrays of `a` into `ws`.
void carve_decode_ws(DecodeArgs& a, const mla_config* c, void* ws, int W, int batch) {
    const size_t slots = (size_t)W + batch;
    char* p = (char*)ws;
    a.o_part = (float*)p;
    p += align256(slots * c->heads * c->d_latent * sizeof(float));
    a.lse_part = (float*)p;
    p += align256(slots * c->heads * sizeof(float));
    a.seq_slots = (int4*)p;
}

}  // namespace

extern "C" {

const char* mla_status_string(int s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case MLA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_TIMEOUT: return "device wait timed out";
        case MLA_ERR_INDEX: return "block id or sequence index out of range";
        default: return "unknown status";
    }
}

int mla_version(void) { return 100; }

int mla_set_wait_limit_ns(int64_t ns) {
    g_wait_ns = ns > 0 ? (uint64_t)ns : kDefaultWaitNs;
    return MLA_OK;
}

int mla_get_status(mla_stream_t stream, int* out) {
    if (!out) return MLA_ERR_INVALID_ARG;
    int* p;
    if (int rc = status_ptr(&p)) return rc;
    int v = 0, zero = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
    *out = v;
    return MLA_OK;
}

int mla_decode_path(const mla_config* cfg) {
    if (check_cfg(cfg)) return -1;
    return use_tc(cfg, 1) ? 1 : 0;
}

}  // extern "C"

namespace {

int append_latent_impl(const mla_config* cfg, const void* x, int n_tok, int d_in,
                      const void* w_dkv, const int32_t* seq_idx, const int32_t* pos,
                      const int32_t* block_table, int batch, int max_blocks, void* cache,
                      int64_t num_blocks, void* dense_out, mla_stream_t stream, SplitScratch sp) {
    if (int rc = check_cfg(cfg)) return rc;
    if (n_tok < 0 || d_in < 1 || d_in > 65536 || batch < 1 || max_blocks < 1 ||
        num_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    if (n_tok == 0) return MLA_OK;
    if (!x || !w_dkv || !seq_idx || !pos || !block_table || !cache) return MLA_ERR_INVALID_ARG;
    if ((size_t)(d_in + cfg->d_latent + cfg->d_rope) * sizeof(float) > 200 * 1024)
        return MLA_ERR_UNSUPPORTED;
    int* status;
    if (int rc = status_ptr(&status)) return rc;
    const int D = cfg->d_latent + cfg->d_rope;
    if (cfg->dtype == MLA_DTYPE_BF16 && d_in % 8 == 0 && D % 8 == 0 && cfg->d_latent % 16 == 0 &&
        al16(x) && al16(w_dkv) && al16(cache) && (!dense_out || al16(dense_out))) {
        // rows = x . [W_L | W_KR] on the tensor cores; the epilogue rotates the
        // rotary part and writes each row to its paged slot (and dense_out)
        TcOperand A = op3(x, d_in, n_tok, 1, (uint64_t)d_in * 2, (uint64_t)d_in * 2 * n_tok);
        TcOperand B = op3(w_dkv, D, d_in, 1, (uint64_t)D * 2, (uint64_t)D * 2 * d_in);
        TcGemmParams g = gemm_params(n_tok, D, d_in, true, nullptr, 0, 0, MLA_DTYPE_BF16, status, sp);
        g.epi = 1;
        g.d_latent = cfg->d_latent; g.d_rope = cfg->d_rope; g.block_size = cfg->block_size;
        g.max_blocks = max_blocks; g.batch = batch; g.num_blocks = num_blocks;
        g.rope_theta1 = rope_theta1(cfg); g.seq_idx = seq_idx; g.pos = pos;
        g.block_table = block_table; g.cache = (__nv_bfloat16*)cache;
        g.dense_out = (__nv_bfloat16*)dense_out;
        return cuda_rc(launch_gemm_tc(A, B, g, 1, (cudaStream_t)stream));
    }
    AppendArgs a{};
    a.n_tok = n_tok; a.d_in = d_in; a.d_latent = cfg->d_latent; a.d_rope = cfg->d_rope;
    a.block_size = cfg->block_size; a.max_blocks = max_blocks; a.batch = batch;
    a.num_blocks = num_blocks; a.rope_theta1 = rope_theta1(cfg); a.x = x; a.w_dkv = w_dkv;
    a.seq_idx = seq_idx; a.pos = pos; a.block_table = block_table; a.cache = cache;
    a.dense_out = dense_out; a.rows_f32 = nullptr; a.status = status;
    return cuda_rc(launch_append(a, cfg->dtype, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

int mla_append_latent(const mla_config* cfg, const void* x, int n_tok, int d_in,
                      const void* w_dkv, const int32_t* seq_idx, const int32_t* pos,
                      const int32_t* block_table, int batch, int max_blocks, void* cache,
                      int64_t num_blocks, void* dense_out, mla_stream_t stream) {
    return append_latent_impl(cfg, x, n_tok, d_in, w_dkv, seq_idx, pos, block_table, batch, max_blocks, cache, num_blocks, dense_out, stream, SplitScratch{});
}

int mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* w_uk, int batch,
                 void* q_lat, mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 0) return MLA_ERR_INVALID_ARG;
    if (batch == 0) return MLA_OK;
    if (!q_nope || !w_uk || !q_lat) return MLA_ERR_INVALID_ARG;
    const int H = cfg->heads, DL = cfg->d_latent, DN = cfg->d_nope;
    cudaStream_t st = (cudaStream_t)stream;
    if (cfg->dtype == MLA_DTYPE_BF16 && DN % 8 == 0 && al16(q_nope) && al16(w_uk)) {
        int* status;
        if (int rc = status_ptr(&status)) return rc;
        // per head h (batch index of the GEMM): [batch x DN] . W_LK_h^T, W_LK_h = [DL][DN]
        TcOperand A = op3(q_nope, DN, batch, H, (uint64_t)H * DN * 2, (uint64_t)DN * 2);
        TcOperand B = op3(w_uk, DN, DL, H, (uint64_t)DN * 2, (uint64_t)DL * DN * 2);
        TcGemmParams g = gemm_params(batch, DL, DN, false, q_lat, DL, (int64_t)H * DL,
                                     MLA_DTYPE_BF16, status);
        if (batch <= kSkinnyRows) return cuda_rc(launch_gemm_tc_skinny(A, B, false, g, H, st));
        return cuda_rc(launch_gemm_tc(A, B, g, H, st));
    }
    // per head h: q_lat[:, h, :] (batch x DL) = q_nope[:, h, :] (batch x DN) . W_LK_h^T
    GemmArgs g{};
    g.M = batch; g.N = DL; g.K = DN; g.batch = H;
    g.A = q_nope; g.sA = DN; g.sAm = (int64_t)H * DN; g.sAk = 1;
    g.B = w_uk; g.sB = (int64_t)DL * DN; g.sBk = 1; g.sBn = DN;
    g.C = q_lat; g.sC = DL; g.sCm = (int64_t)H * DL; g.sCn = 1;
    return cuda_rc(launch_gemm_simt(g, cfg->dtype, cfg->dtype, cfg->dtype, st));
}

int mla_decode_workspace_size(const mla_config* cfg, int batch, size_t* bytes) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!bytes || batch < 1 || batch > kMaxDecodeBatch) return MLA_ERR_INVALID_ARG;
    int W;
    if (int rc = decode_workers(cfg, batch, &W)) return rc;
    *bytes = decode_ws_bytes(cfg, W, batch);
    return MLA_OK;
}

int mla_decode(const mla_config* cfg, const void* q_lat, const void* q_pe, const void* cache,
               int64_t num_blocks, const int32_t* block_table, int max_blocks,
               const int32_t* seq_lens, int batch, void* o_lat, float* lse, void* workspace,
               size_t ws_bytes, mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1 || num_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    if ((int64_t)max_blocks * cfg->block_size > (int64_t)1 << 30) return MLA_ERR_INVALID_ARG;
    if (!q_lat || (!q_pe && cfg->d_rope > 0) || !cache || !block_table || !seq_lens || !o_lat)
        return MLA_ERR_INVALID_ARG;
    int W;
    if (int rc = decode_workers(cfg, batch, &W)) return rc;
    const size_t need = decode_ws_bytes(cfg, W, batch);
    if (!workspace || ws_bytes < need || ((uintptr_t)workspace & 255)) return MLA_ERR_WORKSPACE;
    int* status;
    if (int rc = status_ptr(&status)) return rc;
    DecodeArgs a{};
    a.heads = cfg->heads; a.d_latent = cfg->d_latent; a.d_rope = cfg->d_rope;
    a.block_size = cfg->block_size; a.max_blocks = max_blocks; a.batch = batch;
    a.workers = W; a.num_blocks = num_blocks; a.scale = cfg->softmax_scale;
    a.q_lat = q_lat; a.q_pe = q_pe; a.cache = cache; a.block_table = block_table;
    a.seq_lens = seq_lens; a.o_lat = o_lat; a.lse = lse; a.status = status;
    a.wait_ns = g_wait_ns;
    carve_decode_ws(a, cfg, workspace, W, batch);
    cudaStream_t st = (cudaStream_t)stream;
    const bool tc = use_tc(cfg, batch) && al16(q_lat) && al16(q_pe) && al16(cache);
    a.tile = tc ? decode_tc_tile() : kTile;
    cudaError_t e = tc ? launch_decode_tc(a, st) : launch_decode_simt(a, cfg->dtype, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_rc(launch_combine_planned(a, cfg->dtype, st));
}

int mla_decode_multi_workspace_size(const mla_config* cfg, int batch, int q_tokens,
                                    int max_blocks, size_t* bytes) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!bytes || batch < 1 || q_tokens < 1 || q_tokens > 64 || max_blocks < 1 ||
        (int64_t)batch * q_tokens > kMaxDecodeBatch)
        return MLA_ERR_INVALID_ARG;
    const int rows = batch * q_tokens;
    int W;
    if (int rc = decode_workers(cfg, rows, &W)) return rc;
    *bytes = align256((size_t)rows * 4) + align256((size_t)rows * max_blocks * 4) +
             decode_ws_bytes(cfg, W, rows);
    return MLA_OK;
}

int mla_decode_multi(const mla_config* cfg, const void* q_lat, const void* q_pe,
                     const void* cache, int64_t num_blocks, const int32_t* block_table,
                     int max_blocks, const int32_t* seq_lens, int batch, int q_tokens,
                     void* o_lat, float* lse, void* workspace, size_t ws_bytes,
                     mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 1 || q_tokens < 1 || q_tokens > 64 || max_blocks < 1 || num_blocks < 1 ||
        (int64_t)batch * q_tokens > kMaxDecodeBatch)
        return MLA_ERR_INVALID_ARG;
    if (!q_lat || (!q_pe && cfg->d_rope > 0) || !cache || !block_table || !seq_lens || !o_lat)
        return MLA_ERR_INVALID_ARG;
    size_t need;
    if (int rc = mla_decode_multi_workspace_size(cfg, batch, q_tokens, max_blocks, &need))
        return rc;
    if (!workspace || ws_bytes < need || ((uintptr_t)workspace & 255)) return MLA_ERR_WORKSPACE;
    const int rows = batch * q_tokens;
    char* p = (char*)workspace;
    int32_t* lens_x = (int32_t*)p;
    p += align256((size_t)rows * 4);
    int32_t* table_x = (int32_t*)p;
    p += align256((size_t)rows * max_blocks * 4);
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_expand_rows(seq_lens, block_table, batch, q_tokens, max_blocks, lens_x, table_x,
                           st) != cudaSuccess)
        return MLA_ERR_CUDA;
    return mla_decode(cfg, q_lat, q_pe, cache, num_blocks, table_x, max_blocks, lens_x, rows,
                      o_lat, lse, p, ws_bytes - (size_t)(p - (char*)workspace), stream);
}

int mla_decode_combine(const mla_config* cfg, const float* o_part, const float* lse_part,
                       int n_splits, int batch, void* o_lat, float* lse, mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (n_splits < 1 || n_splits > 512 || batch < 1) return MLA_ERR_INVALID_ARG;
    if (!o_part || !lse_part || !o_lat) return MLA_ERR_INVALID_ARG;
    return cuda_rc(launch_combine_dense(o_part, lse_part, n_splits, batch, cfg->heads,
                                        cfg->d_latent, o_lat, lse, cfg->dtype,
                                        (cudaStream_t)stream));
}

}  // extern "C"

namespace {

int project_out_impl(const mla_config* cfg, const void* o_lat, const void* w_uv, int batch,
                    void* o_v, const void* w_o, int d_model, void* out, mla_stream_t stream, SplitScratch sp) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 0 || (w_o && d_model < 1)) return MLA_ERR_INVALID_ARG;
    if (batch == 0) return MLA_OK;
    if (!o_lat || !w_uv || !o_v || (w_o && !out)) return MLA_ERR_INVALID_ARG;
    const int H = cfg->heads, DL = cfg->d_latent, DV = cfg->d_v;
    cudaStream_t st = (cudaStream_t)stream;
    const bool tc = cfg->dtype == MLA_DTYPE_BF16 && DL % 8 == 0 && DV % 8 == 0 &&
                    (!w_o || d_model % 8 == 0) && al16(o_lat) && al16(w_uv) && al16(o_v) &&
                    (!w_o || al16(w_o));
    if (tc) {
        int* status;
        if (int rc = status_ptr(&status)) return rc;
        // per head h: o_v[:, h, :] = o_lat[:, h, :] . W_LV_h, W_LV_h = [DL][DV] (N-major)
        TcOperand A = op3(o_lat, DL, batch, H, (uint64_t)H * DL * 2, (uint64_t)DL * 2);
        TcOperand B = op3(w_uv, DV, DL, H, (uint64_t)DV * 2, (uint64_t)DL * DV * 2);
        TcGemmParams g = gemm_params(batch, DV, DL, true, o_v, DV, (int64_t)H * DV,
                                     MLA_DTYPE_BF16, status);
        if (int rc = cuda_rc(batch <= kSkinnyRows ? launch_gemm_tc_skinny(A, B, true, g, H, st)
                                                  : launch_gemm_tc(A, B, g, H, st)))
            return rc;
        if (!w_o) return MLA_OK;
        const uint64_t KO = (uint64_t)H * DV;
        TcOperand A2 = op3(o_v, KO, batch, 1, KO * 2, KO * 2 * batch);
        TcOperand B2 = op3(w_o, d_model, KO, 1, (uint64_t)d_model * 2, KO * d_model * 2);
        TcGemmParams g2 = gemm_params(batch, d_model, (int)KO, true, out, 0, d_model,
                                      MLA_DTYPE_BF16, status, sp);
        return cuda_rc(launch_gemm_tc(A2, B2, g2, 1, st));
    }
    // per head h: o_v[:, h, :] (batch x DV) = o_lat[:, h, :] (batch x DL) . W_LV_h (DL x DV)
    GemmArgs g{};
    g.M = batch; g.N = DV; g.K = DL; g.batch = H;
    g.A = o_lat; g.sA = DL; g.sAm = (int64_t)H * DL; g.sAk = 1;
    g.B = w_uv; g.sB = (int64_t)DL * DV; g.sBk = DV; g.sBn = 1;
    g.C = o_v; g.sC = DV; g.sCm = (int64_t)H * DV; g.sCn = 1;
    if (int rc = cuda_rc(launch_gemm_simt(g, cfg->dtype, cfg->dtype, cfg->dtype, st))) return rc;
    if (!w_o) return MLA_OK;
    // out (batch x d_model) = o_v viewed as batch x (H*DV) . W_O
    GemmArgs o{};
    o.M = batch; o.N = d_model; o.K = H * DV; o.batch = 1;
    o.A = o_v; o.sAm = (int64_t)H * DV; o.sAk = 1;
    o.B = w_o; o.sBk = d_model; o.sBn = 1;
    o.C = out; o.sCm = d_model; o.sCn = 1;
    return cuda_rc(launch_gemm_simt(o, cfg->dtype, cfg->dtype, cfg->dtype, st));
}

}  // namespace

extern "C" {

int mla_project_out(const mla_config* cfg, const void* o_lat, const void* w_uv, int batch,
                    void* o_v, const void* w_o, int d_model, void* out, mla_stream_t stream) {
    return project_out_impl(cfg, o_lat, w_uv, batch, o_v, w_o, d_model, out, stream, SplitScratch{});
}

int mla_query_proj_workspace_size(const mla_config* cfg, int batch, int d_lq, size_t* bytes) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!bytes || batch < 1 || d_lq < 0) return MLA_ERR_INVALID_ARG;
    *bytes = align256((size_t)batch * d_lq * sizeof(float)) +
             align256((size_t)batch * cfg->heads * (cfg->d_nope + cfg->d_rope) * sizeof(float));
    return MLA_OK;
}

}  // extern "C"

namespace {

int query_proj_impl(const mla_config* cfg, const void* x, int batch, int d_in, const void* w_dq,
                   int d_lq, const void* w_uq, const int32_t* pos, void* q_nope, void* q_pe,
                   void* scratch, size_t scratch_bytes, mla_stream_t stream, SplitScratch sp) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 1 || d_in < 1 || (w_dq && d_lq < 1)) return MLA_ERR_INVALID_ARG;
    if (!x || !w_uq || !pos || !q_nope || (!q_pe && cfg->d_rope > 0)) return MLA_ERR_INVALID_ARG;
    const int dlq = w_dq ? d_lq : 0;
    size_t need;
    mla_query_proj_workspace_size(cfg, batch, dlq, &need);
    if (!scratch || scratch_bytes < need || ((uintptr_t)scratch & 255)) return MLA_ERR_WORKSPACE;
    const int H = cfg->heads, DQ = cfg->d_nope + cfg->d_rope;
    cudaStream_t st = (cudaStream_t)stream;
    float* cq = (float*)scratch;
    float* q_all = (float*)((char*)scratch + align256((size_t)batch * dlq * sizeof(float)));
    if (cfg->dtype == MLA_DTYPE_BF16 && d_in % 8 == 0 && (!w_dq || d_lq % 8 == 0) &&
        (H * DQ) % 8 == 0 && al16(x) && al16(w_uq) && (!w_dq || al16(w_dq))) {
        int* status;
        if (int rc = status_ptr(&status)) return rc;
        const void* a_in = x;
        int k_in = d_in;
        // the query split and rotation run in W_UQ's epilogue when the halves
        // of a head's columns are whole bf16 pairs; the rotations' (cos, sin)
        // are formed once per (sequence, pair) into the scratch, first, since
        // they depend only on the positions
        const bool fused = cfg->d_nope % 2 == 0 && al16(q_nope) && (cfg->d_rope == 0 || al16(q_pe));
        float2* rope_cs = (float2*)q_all;
        if (fused &&
            launch_rope_table(pos, batch, cfg->d_rope, rope_theta1(cfg), rope_cs, st) != cudaSuccess)
            return MLA_ERR_CUDA;
        if (w_dq) {
            // c_q = x . W_DQ, kept in bf16 (scratch) as the next GEMM's A operand
            TcOperand A = op3(x, d_in, batch, 1, (uint64_t)d_in * 2, (uint64_t)d_in * 2 * batch);
            TcOperand B = op3(w_dq, d_lq, d_in, 1, (uint64_t)d_lq * 2,
                              (uint64_t)d_lq * 2 * d_in);
            TcGemmParams g = gemm_params(batch, d_lq, d_in, true, cq, 0, d_lq, MLA_DTYPE_BF16,
                                         status, sp);
            if (int rc = cuda_rc(launch_gemm_tc(A, B, g, 1, st))) return rc;
            a_in = cq;
            k_in = d_lq;
        }
        const uint64_t NQ = (uint64_t)H * DQ;
        TcOperand A = op3(a_in, k_in, batch, 1, (uint64_t)k_in * 2, (uint64_t)k_in * 2 * batch);
        TcOperand B = op3(w_uq, NQ, k_in, 1, NQ * 2, NQ * 2 * k_in);
        if (fused) {
            TcGemmParams g = gemm_params(batch, (int)NQ, k_in, true, nullptr, 0, 0,
                                         MLA_DTYPE_BF16, status, sp);
            g.epi = 2;
            g.d_nope = cfg->d_nope;
            g.d_rope = cfg->d_rope;
            g.q_nope = (__nv_bfloat16*)q_nope;
            g.q_pe = (__nv_bfloat16*)q_pe;
            g.rope_cs = rope_cs;
            return cuda_rc(launch_gemm_tc(A, B, g, 1, st));
        }
        TcGemmParams g = gemm_params(batch, (int)NQ, k_in, true, q_all, 0, (int64_t)NQ,
                                     MLA_DTYPE_F32, status, sp);
        if (int rc = cuda_rc(launch_gemm_tc(A, B, g, 1, st))) return rc;
        return cuda_rc(launch_q_split_rope(q_all, batch, H, cfg->d_nope, cfg->d_rope, pos,
                                           rope_theta1(cfg), q_nope, q_pe, cfg->dtype, st));
    }
    const void* a_in = x;
    int a_dtype = cfg->dtype, k_in = d_in;
    if (w_dq) {
        GemmArgs g{};
        g.M = batch; g.N = d_lq; g.K = d_in; g.batch = 1;
        g.A = x; g.sAm = d_in; g.sAk = 1;
        g.B = w_dq; g.sBk = d_lq; g.sBn = 1;
        g.C = cq; g.sCm = d_lq; g.sCn = 1;
        if (int rc = cuda_rc(launch_gemm_simt(g, cfg->dtype, cfg->dtype, MLA_DTYPE_F32, st)))
            return rc;
        a_in = cq; a_dtype = MLA_DTYPE_F32; k_in = d_lq;
    }
    GemmArgs u{};
    u.M = batch; u.N = H * DQ; u.K = k_in; u.batch = 1;
    u.A = a_in; u.sAm = k_in; u.sAk = 1;
    u.B = w_uq; u.sBk = (int64_t)H * DQ; u.sBn = 1;
    u.C = q_all; u.sCm = (int64_t)H * DQ; u.sCn = 1;
    if (int rc = cuda_rc(launch_gemm_simt(u, a_dtype, cfg->dtype, MLA_DTYPE_F32, st))) return rc;
    return cuda_rc(launch_q_split_rope(q_all, batch, H, cfg->d_nope, cfg->d_rope, pos,
                                       rope_theta1(cfg), q_nope, q_pe, cfg->dtype, st));
}

}  // namespace

extern "C" {

int mla_query_proj(const mla_config* cfg, const void* x, int batch, int d_in, const void* w_dq,
                   int d_lq, const void* w_uq, const int32_t* pos, void* q_nope, void* q_pe,
                   void* scratch, size_t scratch_bytes, mla_stream_t stream) {
    return query_proj_impl(cfg, x, batch, d_in, w_dq, d_lq, w_uq, pos, q_nope, q_pe, scratch, scratch_bytes, stream, SplitScratch{});
}

// ---------------------------------------------------------------------------
// Whole decode steps in one call.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

size_t dtype_size(const mla_config* c) { return c->dtype == MLA_DTYPE_BF16 ? 2 : 4; }

// Sequential carving of a workspace into 256-byte aligned pieces.  With a
// null base it only counts bytes.
struct Carver {
    char* base;
    size_t used;
    void* take(size_t bytes) {
        void* p = base ? base + used : nullptr;
        used += align256(bytes);
        return p;
    }
};

// Per-step inputs that the caller may pass in host memory: copied into the
// workspace on the stream (cudaMemcpyAsync, one per tensor).
int stage_in(const void** ptr, void* dev, size_t bytes, bool host, cudaStream_t st) {
    if (!host) return MLA_OK;
    if (cudaMemcpyAsync(dev, *ptr, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    *ptr = dev;
    return MLA_OK;
}

struct LayerWs {
    int32_t *seq_lens, *block_table, *pos, *seq_idx;
    void *x, *q_nope, *q_pe, *q_lat, *o_lat, *o_v, *out, *q_scratch, *dec;
    size_t q_scratch_bytes, dec_bytes;
    SplitScratch split;   // split-K partials of the batch-1 projections
};

int layer_ws(const mla_config* c, const mla_layer_weights* w, int batch, int max_blocks,
             char* base, LayerWs* ws, size_t* total) {
    const size_t es = dtype_size(c), B = (size_t)batch, H = (size_t)c->heads;
    int W;
    if (int rc = decode_workers(c, batch, &W)) return rc;
    size_t qs;
    if (int rc = mla_query_proj_workspace_size(c, batch, w->w_dq ? w->d_lq : 0, &qs)) return rc;
    Carver k{base, 0};
    ws->seq_lens = (int32_t*)k.take(B * 4);
    ws->block_table = (int32_t*)k.take(B * (size_t)max_blocks * 4);
    ws->pos = (int32_t*)k.take(B * 4);
    ws->seq_idx = (int32_t*)k.take(B * 4);
    ws->x = k.take(B * (size_t)w->d_model * es);
    ws->q_nope = k.take(B * H * c->d_nope * es);
    ws->q_pe = k.take(B * H * c->d_rope * es);
    ws->q_lat = k.take(B * H * c->d_latent * es);
    ws->o_lat = k.take(B * H * c->d_latent * es);
    ws->o_v = k.take(B * H * c->d_v * es);
    ws->out = k.take(B * (size_t)w->d_model * es);
    ws->q_scratch_bytes = qs;
    ws->q_scratch = k.take(qs);
    ws->dec_bytes = decode_ws_bytes(c, W, batch);
    ws->dec = k.take(ws->dec_bytes);
    // the largest split-K scratch of the step's batch-1 products: W_DQ, W_UQ
    // (query), W_DKV (cache row), W_O (output)
    int sms;
    if (int rc = num_sms(&sms)) return rc;
    const int nh = c->heads, dq = c->d_nope + c->d_rope, D = c->d_latent + c->d_rope;
    const int qin = w->w_dq ? w->d_lq : w->d_model;
    size_t sb = 0;
    auto upd = [&](int M, int N, int K) {
        const size_t b = gemm_tc_split_scratch(M, N, K, sms);
        if (b > sb) sb = b;
    };
    if (w->w_dq) upd(batch, w->d_lq, w->d_model);
    upd(batch, nh * dq, qin);
    upd(batch, D, w->d_model);
    upd(batch, w->d_model, nh * c->d_v);
    ws->split.bytes = sb;
    ws->split.ptr = (float*)k.take(sb);
    *total = k.used;
    return MLA_OK;
}

struct CachedWs {
    int32_t *seq_lens, *block_table;
    void *q_nope, *q_pe, *q_lat, *o_lat, *o_v, *dec;
    float* lse;
    size_t dec_bytes;
};

int cached_ws(const mla_config* c, int batch, int max_blocks, char* base, CachedWs* ws,
              size_t* total) {
    const size_t es = dtype_size(c), B = (size_t)batch, H = (size_t)c->heads;
    int W;
    if (int rc = decode_workers(c, batch, &W)) return rc;
    Carver k{base, 0};
    ws->seq_lens = (int32_t*)k.take(B * 4);
    ws->block_table = (int32_t*)k.take(B * (size_t)max_blocks * 4);
    ws->q_nope = k.take(B * H * c->d_nope * es);
    ws->q_pe = k.take(B * H * c->d_rope * es);
    ws->q_lat = k.take(B * H * c->d_latent * es);
    ws->o_lat = k.take(B * H * c->d_latent * es);
    ws->lse = (float*)k.take(B * H * 4);
    ws->o_v = k.take(B * H * c->d_v * es);
    ws->dec_bytes = decode_ws_bytes(c, W, batch);
    ws->dec = k.take(ws->dec_bytes);
    *total = k.used;
    return MLA_OK;
}

bool valid_weights(const mla_layer_weights* w) {
    return w && w->d_model >= 1 && w->w_dkv && w->w_uq && w->w_uk && w->w_uv && w->w_o &&
           (!w->w_dq || w->d_lq >= 1);
}

}  // namespace

extern "C" {

int mla_layer_decode_step_workspace_size(const mla_config* cfg, const mla_layer_weights* w,
                                         int batch, int max_blocks, size_t* bytes) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!bytes || !valid_weights(w) || batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    LayerWs ws;
    return layer_ws(cfg, w, batch, max_blocks, nullptr, &ws, bytes);
}

int mla_layer_decode_step(const mla_config* cfg, const mla_layer_weights* w, const void* x,
                          const int32_t* seq_lens, int batch, void* cache, int64_t num_blocks,
                          const int32_t* block_table, int max_blocks, void* out, int io_flags,
                          void* workspace, size_t ws_bytes, mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!valid_weights(w) || batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1 ||
        num_blocks < 1 || (io_flags & ~(MLA_IO_HOST_INPUTS | MLA_IO_HOST_OUTPUT)))
        return MLA_ERR_INVALID_ARG;
    if (!x || !seq_lens || !cache || !block_table || !out) return MLA_ERR_INVALID_ARG;
    LayerWs ws;
    size_t need;
    if (int rc = layer_ws(cfg, w, batch, max_blocks, (char*)workspace, &ws, &need)) return rc;
    if (!workspace || ws_bytes < need || ((uintptr_t)workspace & 255)) return MLA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const bool hin = io_flags & MLA_IO_HOST_INPUTS, hout = io_flags & MLA_IO_HOST_OUTPUT;
    const size_t es = dtype_size(cfg);
    const void* xs = x;
    const void* sl = seq_lens;
    const void* bt = block_table;
    if (int rc = stage_in(&xs, ws.x, (size_t)batch * w->d_model * es, hin, st)) return rc;
    if (int rc = stage_in(&sl, ws.seq_lens, (size_t)batch * 4, hin, st)) return rc;
    if (int rc = stage_in(&bt, ws.block_table, (size_t)batch * max_blocks * 4, hin, st)) return rc;
    if (launch_step_positions((const int32_t*)sl, batch, ws.pos, ws.seq_idx, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    mla_stream_t s = stream;
    if (int rc = query_proj_impl(cfg, xs, batch, w->d_model, w->w_dq, w->w_dq ? w->d_lq : 0,
                                 w->w_uq, ws.pos, ws.q_nope, ws.q_pe, ws.q_scratch,
                                 ws.q_scratch_bytes, s, ws.split))
        return rc;
    if (int rc = append_latent_impl(cfg, xs, batch, w->d_model, w->w_dkv, ws.seq_idx, ws.pos,
                                    (const int32_t*)bt, batch, max_blocks, cache, num_blocks,
                                    nullptr, s, ws.split))
        return rc;
    if (int rc = mla_absorb_q(cfg, ws.q_nope, w->w_uk, batch, ws.q_lat, s)) return rc;
    if (int rc = mla_decode(cfg, ws.q_lat, ws.q_pe, cache, num_blocks, (const int32_t*)bt,
                            max_blocks, (const int32_t*)sl, batch, ws.o_lat, nullptr, ws.dec,
                            ws.dec_bytes, s))
        return rc;
    void* o = hout ? ws.out : out;
    if (int rc = project_out_impl(cfg, ws.o_lat, w->w_uv, batch, ws.o_v, w->w_o, w->d_model, o, s,
                                  ws.split))
        return rc;
    if (hout && cudaMemcpyAsync(out, ws.out, (size_t)batch * w->d_model * es,
                                cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}

int mla_cached_decode_step_workspace_size(const mla_config* cfg, int batch, int max_blocks,
                                          size_t* bytes) {
    if (int rc = check_cfg(cfg)) return rc;
    if (!bytes || batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    CachedWs ws;
    return cached_ws(cfg, batch, max_blocks, nullptr, &ws, bytes);
}

int mla_cached_decode_step(const mla_config* cfg, const void* q_nope, const void* q_pe,
                           const void* w_uk, const void* w_uv, const int32_t* seq_lens,
                           int batch, const void* cache, int64_t num_blocks,
                           const int32_t* block_table, int max_blocks, void* o_v, void* o_lat,
                           float* lse, int io_flags, void* workspace, size_t ws_bytes,
                           mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1 || num_blocks < 1 ||
        (io_flags & ~(MLA_IO_HOST_INPUTS | MLA_IO_HOST_OUTPUT)))
        return MLA_ERR_INVALID_ARG;
    if (!q_nope || (!q_pe && cfg->d_rope > 0) || !w_uk || !w_uv || !seq_lens || !cache ||
        !block_table || !o_v)
        return MLA_ERR_INVALID_ARG;
    CachedWs ws;
    size_t need;
    if (int rc = cached_ws(cfg, batch, max_blocks, (char*)workspace, &ws, &need)) return rc;
    if (!workspace || ws_bytes < need || ((uintptr_t)workspace & 255)) return MLA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const bool hin = io_flags & MLA_IO_HOST_INPUTS, hout = io_flags & MLA_IO_HOST_OUTPUT;
    const size_t es = dtype_size(cfg), BH = (size_t)batch * cfg->heads;
    const void* qn = q_nope;
    const void* qp = q_pe;
    const void* sl = seq_lens;
    const void* bt = block_table;
    if (int rc = stage_in(&qn, ws.q_nope, BH * cfg->d_nope * es, hin, st)) return rc;
    if (cfg->d_rope > 0)
        if (int rc = stage_in(&qp, ws.q_pe, BH * cfg->d_rope * es, hin, st)) return rc;
    if (int rc = stage_in(&sl, ws.seq_lens, (size_t)batch * 4, hin, st)) return rc;
    if (int rc = stage_in(&bt, ws.block_table, (size_t)batch * max_blocks * 4, hin, st)) return rc;
    void* ol = o_lat ? o_lat : ws.o_lat;
    float* ls = lse ? lse : ws.lse;
    void* ov = hout ? ws.o_v : o_v;
    if (int rc = mla_absorb_q(cfg, qn, w_uk, batch, ws.q_lat, stream)) return rc;
    if (int rc = mla_decode(cfg, ws.q_lat, qp, cache, num_blocks, (const int32_t*)bt, max_blocks,
                            (const int32_t*)sl, batch, ol, ls, ws.dec, ws.dec_bytes, stream))
        return rc;
    if (int rc = mla_project_out(cfg, ol, w_uv, batch, ov, nullptr, 0, nullptr, stream)) return rc;
    if (hout && cudaMemcpyAsync(o_v, ws.o_v, BH * cfg->d_v * es, cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess)
        return MLA_ERR_CUDA;
    return MLA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory where they decode: a host
// framework that owns every byte of device memory through its own pool and
// forbids direct cudaMalloc, a plugin interface that passes only input and
// output pointers, or a latency-critical loop where an allocation's implicit
// device synchronisation is not acceptable.  For them the split-KV partial
// results live in the fixed static array below instead of a workspace.  Every
// GPU that loads this library holds the array until the process exits.
// ---------------------------------------------------------------------------
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices];

// Device address of the static array for the current device, looked up once
// per device with that device current.
int noalloc_scratch(void** out) {
    int dev;
    if (int rc = current_device(&dev)) return rc;
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return MLA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_noalloc(const mla_config* cfg, const void* q_lat, const void* q_pe,
                                  const void* cache, int64_t num_blocks,
                                  const int32_t* block_table, int max_blocks,
                                  const int32_t* seq_lens, int batch, void* o_lat, float* lse,
                                  mla_stream_t stream) {
    if (int rc = check_cfg(cfg)) return rc;
    if (batch < 1 || batch > kMaxDecodeBatch || max_blocks < 1 || num_blocks < 1)
        return MLA_ERR_INVALID_ARG;
    if ((int64_t)max_blocks * cfg->block_size > (int64_t)1 << 30) return MLA_ERR_INVALID_ARG;
    if (!q_lat || (!q_pe && cfg->d_rope > 0) || !cache || !block_table || !seq_lens || !o_lat)
        return MLA_ERR_INVALID_ARG;
    // The partials of W workers need (W + batch) slots; use as many workers
    // as the array holds, up to the count mla_decode would use.
    int W;
    if (int rc = decode_workers(cfg, batch, &W)) return rc;
    while (W >= 1 && decode_ws_bytes(cfg, W, batch) > MLA_NOALLOC_SCRATCH_BYTES) --W;
    if (W < 1) return MLA_ERR_UNSUPPORTED;
    void* scratch;
    if (int rc = noalloc_scratch(&scratch)) return rc;
    int* status;
    if (int rc = status_ptr(&status)) return rc;
    // Nothing in the array has to start at zero: every partial slot the
    // merge reads is written earlier in the same call.
    DecodeArgs a{};
    a.heads = cfg->heads; a.d_latent = cfg->d_latent; a.d_rope = cfg->d_rope;
    a.block_size = cfg->block_size; a.max_blocks = max_blocks; a.batch = batch;
    a.workers = W; a.num_blocks = num_blocks; a.scale = cfg->softmax_scale;
    a.q_lat = q_lat; a.q_pe = q_pe; a.cache = cache; a.block_table = block_table;
    a.seq_lens = seq_lens; a.o_lat = o_lat; a.lse = lse; a.status = status;
    a.wait_ns = g_wait_ns;
    carve_decode_ws(a, cfg, scratch, W, batch);
    cudaStream_t st = (cudaStream_t)stream;
    const bool tc = use_tc(cfg, batch) && al16(q_lat) && al16(q_pe) && al16(cache);
    a.tile = tc ? decode_tc_tile() : kTile;
    cudaError_t e = tc ? launch_decode_tc(a, st) : launch_decode_simt(a, cfg->dtype, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_rc(launch_combine_planned(a, cfg->dtype, st));
}
