"""ctypes wrapper around the fp64 C oracle, plus the per-workload pipelines.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg.  The CUDA library never imports it, and this
module imports nothing from the CUDA library.

Inputs arrive as numpy arrays (any float dtype; bf16 inputs are passed already
widened to float32 by the caller) and are widened to float64 here, so the
oracle sees exactly the rounded values the GPU sees.
"""
import ctypes
import math

import numpy as np

from . import build as _build

_lib = None

PLANT_NONE = 0
PLANT_DROP_ROPE_TERM = 1
PLANT_TRANSPOSE_WLK = 2
PLANT_ROPE_SIGN = 3
PLANT_MASK_OFF_BY_ONE = 4
PLANT_NO_SCALE = 5
PLANT_VALUE_FROM_KEY = 6


def _L():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        lib.mla_oracle_num_threads.restype = ctypes.c_int
        lib.mla_oracle_rope.argtypes = [dp, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_int, dp]
        lib.mla_oracle_latent_rows.argtypes = [dp, ctypes.c_int, ctypes.c_int, dp, ctypes.c_int,
                                               ctypes.c_int, ip, ctypes.c_double, dp]
        lib.mla_oracle_query.argtypes = [dp, ctypes.c_int, ctypes.c_int, dp, ctypes.c_int, dp,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ip,
                                         ctypes.c_double, dp, dp]
        lib.mla_oracle_slot.restype = ctypes.c_int64
        lib.mla_oracle_slot.argtypes = [ip, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int, ctypes.c_int]
        lib.mla_oracle_scatter_rows.restype = ctypes.c_int
        lib.mla_oracle_scatter_rows.argtypes = [u8, ctypes.c_int, ctypes.c_int64, ip, ip, ip,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int64, u8]
        lib.mla_oracle_decode.restype = ctypes.c_int
        lib.mla_oracle_decode.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ip, ctypes.c_int, ip, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp,
            ctypes.c_double, dp, ctypes.c_int, ip, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp]
        lib.mla_oracle_kv_numbers_per_token.restype = ctypes.c_double
        lib.mla_oracle_kv_numbers_per_token.argtypes = [ctypes.c_int] * 3
        lib.mla_oracle_latent_numbers_per_token.restype = ctypes.c_double
        lib.mla_oracle_latent_numbers_per_token.argtypes = [ctypes.c_int] * 3
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def num_threads() -> int:
    """OpenMP threads the oracle's decode loop runs on."""
    return int(_L().mla_oracle_num_threads())


def rope(vec, pos, base=10000.0, plant=PLANT_NONE):
    """Rotary embedding of one even-length vector at position `pos`."""
    v = _f64(vec)
    out = np.empty_like(v)
    _L().mla_oracle_rope(_dp(v), v.shape[0], float(pos), float(base), int(plant), _dp(out))
    return out


def latent_rows(x, w_dkv, d_l, d_r, pos, base=10000.0):
    """Cache rows [c | RoPE(x W_KR, pos)] of new tokens x [n, d_in]."""
    x = _f64(x)
    w = _f64(w_dkv)
    pos = _i32(pos)
    n, d_in = x.shape
    assert w.shape == (d_in, d_l + d_r)
    rows = np.empty((n, d_l + d_r), dtype=np.float64)
    _L().mla_oracle_latent_rows(_dp(x), n, d_in, _dp(w), d_l, d_r, _ip(pos), float(base),
                                _dp(rows))
    return rows


def query(x, w_uq, heads, d_n, d_r, pos, w_dq=None, base=10000.0):
    """Per-head (q_nope [B,H,d_n], q_pe [B,H,d_r]) of the current tokens x [B, d_in]."""
    x = _f64(x)
    B, d_in = x.shape
    wdq = _f64(w_dq) if w_dq is not None else None
    d_lq = wdq.shape[1] if wdq is not None else d_in
    wuq = _f64(w_uq).reshape(d_lq, heads * (d_n + d_r))
    pos = _i32(pos)
    q_nope = np.empty((B, heads, d_n), dtype=np.float64)
    q_pe = np.empty((B, heads, d_r), dtype=np.float64)
    _L().mla_oracle_query(_dp(x), B, d_in, _dp(wdq), d_lq, _dp(wuq), heads, d_n, d_r,
                          _ip(pos), float(base), _dp(q_nope), _dp(q_pe))
    return q_nope, q_pe


def slot(block_table, block_size, num_blocks, b, i):
    bt = _i32(block_table)
    return int(_L().mla_oracle_slot(_ip(bt), bt.shape[1], block_size, num_blocks, b, i))


def scatter_rows(rows_u8, seq_idx, pos, block_table, block_size, cache_u8):
    """Copies each dense row (bytes) to its paged slot in cache_u8 (in place).

    rows_u8: uint8 [n_tok, row_bytes]; cache_u8: uint8 [num_blocks*block_size, row_bytes].
    Returns the number of rows skipped for an invalid block id.
    """
    rows_u8 = np.ascontiguousarray(rows_u8, dtype=np.uint8)
    assert cache_u8.flags["C_CONTIGUOUS"] and cache_u8.dtype == np.uint8
    n, row_bytes = rows_u8.shape
    num_blocks = cache_u8.shape[0] // block_size
    bt = _i32(block_table)
    u8 = ctypes.POINTER(ctypes.c_uint8)
    return int(_L().mla_oracle_scatter_rows(
        rows_u8.ctypes.data_as(u8), n, row_bytes, _ip(_i32(seq_idx)), _ip(_i32(pos)), _ip(bt),
        bt.shape[1], block_size, num_blocks, cache_u8.ctypes.data_as(u8)))


def decode(cache, block_table, seq_lens, q_nope, q_pe, w_uk, w_uv, scale, w_o=None,
           pairs=None, plant=PLANT_NONE):
    """Unmerged fp64 decode.

    cache [num_blocks, block_size, d_l + d_r] as float64, float32 or uint16/int16
    (bf16 bit patterns, read in place without a copy); block_table [B, max_blocks];
    seq_lens [B]; q_nope [B,H,d_n]; q_pe [B,H,d_r]; w_uk [H,d_l,d_n]; w_uv [H,d_l,d_v];
    w_o [H*d_v, d_model] or None; pairs: iterable of (b, h) or None for all.
    Returns dict with o_lat [B,H,d_l], o_v [B,H,d_v], lse [B,H] (NaN where not
    computed) and out [B,d_model] (only with w_o and all pairs).
    """
    cache = np.ascontiguousarray(cache)
    if cache.dtype == np.float64:
        kind = 0
    elif cache.dtype == np.float32:
        kind = 1
    elif cache.dtype in (np.uint16, np.int16):
        kind = 2
    else:
        cache = _f64(cache)
        kind = 0
    nb, bs, dr = cache.shape
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    q_nope = _f64(q_nope)
    q_pe = _f64(q_pe)
    w_uk = _f64(w_uk)
    w_uv = _f64(w_uv)
    B, H, d_n = q_nope.shape
    d_r = q_pe.shape[2]
    d_l = dr - d_r
    d_v = w_uv.shape[2]
    assert w_uk.shape == (H, d_l, d_n) and w_uv.shape == (H, d_l, d_v)
    assert bt.shape[0] == B and sl.shape == (B,)
    wo = _f64(w_o) if w_o is not None else None
    d_model = wo.shape[1] if wo is not None else 0
    if pairs is not None:
        # each (b, h) once: the C loop writes a pair's output row in place, so
        # two threads given the same pair would interleave their sums
        plist = _i32(sorted({b * H + h for (b, h) in pairs}))
        npairs = len(plist)
    else:
        plist, npairs = None, 0
    o_lat = np.full((B, H, d_l), np.nan)
    o_v = np.full((B, H, d_v), np.nan)
    lse = np.full((B, H), np.nan)
    out = np.full((B, max(d_model, 1)), np.nan)
    rc = _L().mla_oracle_decode(
        cache.ctypes.data_as(ctypes.c_void_p), kind, nb, bs, _ip(bt), bt.shape[1], _ip(sl), B, H, d_l, d_r, d_n, d_v,
        _dp(q_nope), _dp(q_pe), _dp(w_uk), _dp(w_uv), float(scale), _dp(wo), d_model,
        _ip(plist), npairs, int(plant), _dp(o_lat), _dp(o_v), _dp(lse), _dp(out))
    if rc != 0:
        raise ValueError("oracle: invalid block table or sequence length")
    res = {"o_lat": o_lat, "o_v": o_v, "lse": lse}
    if wo is not None and pairs is None:
        res["out"] = out
    return res


def decode_multi(cache, block_table, seq_lens, q_nope, q_pe, w_uk, w_uv, scale, pairs=None):
    """Decode of the last T tokens of each sequence at once.

    q_nope [B,T,H,d_n], q_pe [B,T,H,d_r]; the cache already holds the rows of
    the T new tokens.  Token j of sequence b sits at position n_b - T + j and
    attends to positions 0..n_b - T + j: the causal mask of "How DeepSeek
    Rewrote the Transformer (MLA)", section 03 ("each position attends only to
    itself and earlier ones").  Each token is therefore one unmerged decode
    over the n_b - T + 1 + j tokens before and at it, through its sequence's
    block table.  pairs: iterable of (b, j, h) or None for all.  Returns o_lat
    [B,T,H,d_l], o_v [B,T,H,d_v], lse [B,T,H].
    """
    q_nope = np.asarray(q_nope)
    q_pe = np.asarray(q_pe)
    B, T, H = q_nope.shape[:3]
    bt = np.repeat(_i32(block_table), T, axis=0)
    lens = np.repeat(_i32(seq_lens), T) - T + 1 + np.tile(np.arange(T, dtype=np.int32), B)
    rp = None if pairs is None else [(b * T + j, h) for (b, j, h) in pairs]
    r = decode(cache, bt, lens, q_nope.reshape(B * T, H, -1), q_pe.reshape(B * T, H, -1),
               w_uk, w_uv, scale, pairs=rp)
    return {"o_lat": r["o_lat"].reshape(B, T, H, -1), "o_v": r["o_v"].reshape(B, T, H, -1),
            "lse": r["lse"].reshape(B, T, H)}


def kv_numbers_per_token(kv_heads, head_dim, layers):
    return float(_L().mla_oracle_kv_numbers_per_token(kv_heads, head_dim, layers))


def latent_numbers_per_token(d_l, d_r, layers):
    return float(_L().mla_oracle_latent_numbers_per_token(d_l, d_r, layers))


def default_scale(d_n, d_r):
    """Reading of "divide by the square root of the dimension": the length of
    the dotted query/key vectors, d_n + d_r."""
    return 1.0 / math.sqrt(d_n + d_r)


# ---------------------------------------------------------------------------
# Workload pipelines.  Each takes the dict a workload generator returns
# (numpy arrays, already rounded to the workload's dtype) and composes the
# oracle steps above in the order the pages give them.
# ---------------------------------------------------------------------------

def reference_cached_decode(w, pairs=None, plant=PLANT_NONE):
    """Decode over a cache whose rows are given (shared-cache workloads).

    The query's latent-side part q_nope and rotary part q_pe are given; keys
    and values are expanded per head from the cached latents.
    """
    return decode(w["cache"], w["block_table"], w["seq_lens"], w["q_nope"], w["q_pe"],
                  w["w_uk"], w["w_uv"], w["scale"], pairs=pairs, plant=plant)


def reference_multi_decode(w, pairs=None):
    """Multi-token decode over a cache whose rows are given: q_nope and q_pe
    carry a token axis, [B,T,H,*]."""
    return decode_multi(w["cache"], w["block_table"], w["seq_lens"], w["q_nope"], w["q_pe"],
                        w["w_uk"], w["w_uv"], w["scale"], pairs=pairs)


def reference_token_decode(w, pairs=None, seqs=None, plant=PLANT_NONE):
    """Decode step for workloads that carry the current tokens' hidden states x.

    1. each new token's cache row = [x W_L | RoPE(x W_KR, pos)] written at its
       slot (earlier rows come from the given cache);
    2. query = x (W_LQ) W_UQ per head, rotary part at the query position;
    3. unmerged attention over all seq_len rows; 4. stack heads, multiply by W_O.
    seqs: restrict steps 2-4 to these sequences (results are indexed by
    position in `seqs`); pairs: (index into seqs, head) pairs, as in decode().
    Returns the decode dict plus "cache" (after the append), the new rows and
    the queries.
    """
    cfg = w["cfg"]
    d_l, d_r = cfg["d_latent"], cfg["d_rope"]
    base = cfg["rope_base"]
    cache = np.array(w["cache"], copy=True)
    nb, bs, dr = cache.shape
    rows = latent_rows(w["x_new"], w["w_dkv"], d_l, d_r, w["pos_new"], base)
    # the cache stores rows in the workload's dtype: a row written and read
    # back is the stored (rounded) value
    stored = w["store"](rows)
    flat = cache.reshape(nb * bs, dr)
    for t in range(rows.shape[0]):
        s = slot(w["block_table"], bs, nb, int(w["seq_idx_new"][t]), int(w["pos_new"][t]))
        flat[s] = stored[t]
    B = w["block_table"].shape[0]
    seqs = list(range(B)) if seqs is None else list(seqs)
    bt = np.asarray(w["block_table"])[seqs]
    sl = np.asarray(w["seq_lens"])[seqs]
    x_q = np.asarray(w["x_q"])[seqs]
    pos_q = np.asarray(w["pos_q"])[seqs]
    q_nope, q_pe = query(x_q, w["w_uq"], cfg["heads"], cfg["d_nope"], d_r, pos_q,
                         w_dq=w.get("w_dq"), base=base)
    res = decode(cache, bt, sl, q_nope, q_pe, w["w_uk"], w["w_uv"], w["scale"],
                 w_o=w.get("w_o") if pairs is None else None, pairs=pairs, plant=plant)
    res["cache"] = cache
    res["rows"] = rows
    res["q_nope"] = q_nope
    res["q_pe"] = q_pe
    return res
