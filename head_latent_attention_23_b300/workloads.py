"""Seeded synthetic inputs for MLA decode.

This module only draws random numbers and lays out input structure (sizes,
sequence lengths, page permutations).  It holds none of the attention
arithmetic, so both the CUDA library's callers and the CPU oracle's callers can
use it without sharing any computation.

Every tensor is drawn in fp32 from a CPU ``torch.Generator`` seeded with
``seed``, in the fixed order written in each function, and then rounded to the
workload dtype.  The returned dict holds the rounded tensors (torch, CPU) under
their names, plus ``cfg`` (shapes and parameters).  ``oracle_view(w)`` gives
the same values as numpy arrays for the CPU reference.

Shapes follow the DeepSeek-V2 figures quoted on the pages (128 heads of 128
dims, a 512-value latent plus a 64-value decoupled rotary key per token per
layer, hidden size 7168).  Weights are ~N(0, 1/fan_in); latents, rotary keys
and queries ~N(0, 1).
"""
import math

import numpy as np
import torch

DEEPSEEK = dict(heads=128, d_latent=512, d_rope=64, d_nope=128, d_v=128)


def _cfg(heads, d_latent, d_rope, d_nope, d_v, block_size, dtype, rope_base=10000.0,
         softmax_scale=None):
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d_nope + d_rope)
    return dict(heads=heads, d_latent=d_latent, d_rope=d_rope, d_nope=d_nope, d_v=d_v,
                block_size=block_size, dtype=dtype, rope_base=float(rope_base),
                softmax_scale=float(softmax_scale))


def torch_dtype(name):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _randn(g, shape, std, dtype):
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(torch_dtype(dtype))


def _pages(g, seq_lens, block_size, permute, extra_pages=0):
    """Block table [B, max_blocks] whose used entries are distinct page ids.

    Sequence b uses ceil(seq_len_b / block_size) pages.  With `permute` the
    page ids are a random permutation of all pages, else they are assigned in
    order.  Unused entries are -1.  Returns (block_table int32, num_blocks).
    """
    need = [(int(n) + block_size - 1) // block_size for n in seq_lens]
    total = sum(need) + extra_pages
    ids = torch.randperm(total, generator=g) if permute else torch.arange(total)
    max_blocks = max(max(need), 1)
    bt = torch.full((len(seq_lens), max_blocks), -1, dtype=torch.int32)
    k = 0
    for b, nb in enumerate(need):
        bt[b, :nb] = ids[k:k + nb].to(torch.int32)
        k += nb
    return bt, total


def cached_decode(batch, seq_lens, seed=0, dtype="bf16", block_size=64, permute=False,
                  heads=128, d_latent=512, d_rope=64, d_nope=128, d_v=128, extra_pages=0,
                  max_blocks=None):
    """Decode over an existing cache (cache rows drawn directly).

    Draw order: block-table permutation, cache pool, q_nope, q_pe, w_uk, w_uv.
    The whole pool is drawn, including slots past each sequence's end, so
    masked slots hold ordinary values that must not leak into the result.
    """
    g = torch.Generator().manual_seed(seed)
    seq_lens = [int(n) for n in seq_lens]
    assert len(seq_lens) == batch
    cfg = _cfg(heads, d_latent, d_rope, d_nope, d_v, block_size, dtype)
    bt, nblk = _pages(g, seq_lens, block_size, permute, extra_pages)
    if max_blocks is not None and max_blocks > bt.shape[1]:
        pad = torch.full((batch, max_blocks - bt.shape[1]), -1, dtype=torch.int32)
        bt = torch.cat([bt, pad], dim=1)
    cache = _randn(g, (nblk, block_size, d_latent + d_rope), 1.0, dtype)
    q_nope = _randn(g, (batch, heads, d_nope), 1.0, dtype)
    q_pe = _randn(g, (batch, heads, d_rope), 1.0, dtype)
    w_uk = _randn(g, (heads, d_latent, d_nope), 1.0 / math.sqrt(d_latent), dtype)
    w_uv = _randn(g, (heads, d_latent, d_v), 1.0 / math.sqrt(d_latent), dtype)
    return dict(cfg=cfg, kind="cached", cache=cache, block_table=bt,
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32), q_nope=q_nope, q_pe=q_pe,
                w_uk=w_uk, w_uv=w_uv, batch=batch)


def growing_scores_decode(seed=12):
    """Shared-cache decode (lengths 1000 and 600, pages permuted) whose cache
    page j of each sequence is scaled by 0.03 * 1.35^j after drawing, so the
    scores' maximum keeps rising along a sequence and an online softmax has to
    move its running maximum many times."""
    lens = [1000, 600]
    w = cached_decode(len(lens), lens, seed=seed, permute=True)
    bt = w["block_table"]
    cache = w["cache"].float()
    for b, n in enumerate(lens):
        for j in range((n + 63) // 64):
            cache[bt[b, j]] *= 0.03 * 1.35 ** j
    w["cache"] = cache.to(w["cache"].dtype)
    return w


def growing_scores_exact_query_decode(seed=12):
    """Shared-cache decode (lengths 1000 and 600, pages permuted) built so
    that the scores grow to logits of about 58 while the absorbed query stays
    exactly representable in bf16.

    Draw order: that of cached_decode(seed), then one index j(b, h) in
    [0, d_nope) per (sequence, head).  q_nope[b, h] is replaced by the unit
    vector e_j, so q_lat[b, h] = q_nope[b, h] . W_LK_h^T is column j of
    W_LK_h: a single product with 1.0, exact in any precision.  Cache page j
    of each sequence is then scaled by 1 + 1.5 j, so the running maximum of
    the scores keeps rising along a sequence (hundreds of head-tile events
    above the 2^8 lazy-rescale threshold of the tensor-core kernel)."""
    lens = [1000, 600]
    w = cached_decode(len(lens), lens, seed=seed, permute=True)
    g = torch.Generator().manual_seed(seed + 1)
    B, H, dn = w["q_nope"].shape
    idx = torch.randint(0, dn, (B, H), generator=g)
    q = torch.zeros(B, H, dn)
    q.scatter_(2, idx[..., None], 1.0)
    w["q_nope"] = q.to(w["q_nope"].dtype)
    bt = w["block_table"]
    cache = w["cache"].float()
    for b, n in enumerate(lens):
        for j in range((n + 63) // 64):
            cache[bt[b, j]] *= 1.0 + 1.5 * j
    w["cache"] = cache.to(w["cache"].dtype)
    return w


def crossing_ranges_decode(seed=31, batch=80, d_nope=64, d_v=8):
    """Shared-cache decode with many short and medium sequences (lengths
    uniform in [1, 700], one sequence of 37 tokens in the middle of the
    batch, pages permuted), so that a split of the context into equal tile
    ranges puts several sequence boundaries inside most ranges.  DeepSeek-V2
    head, latent and rotary widths; d_nope and d_v are smaller than
    DeepSeek's only to keep the unmerged CPU reference fast (the attention
    core sees the absorbed query and does not depend on them).

    Draw order: lengths, then that of cached_decode(seed)."""
    g = torch.Generator().manual_seed(seed + 104729)
    lens = torch.randint(1, 701, (batch,), generator=g).tolist()
    lens[batch // 2] = 37
    return cached_decode(batch, lens, seed=seed, permute=True, d_nope=d_nope, d_v=d_v)


def multi_token_decode(batch, seq_lens, q_tokens, seed=0, permute=True):
    """Decode of the last q_tokens tokens of each sequence at once (a chunk of
    prefill or a speculative step), over a cache whose rows are drawn: the
    cached_decode draws, then per-token queries q_nope [B,T,H,d_n] and q_pe
    [B,T,H,d_r] (unit normal) replacing the single-token ones."""
    w = cached_decode(batch, seq_lens, seed=seed, permute=permute)
    g = torch.Generator().manual_seed(seed + 7919)
    c = w["cfg"]
    w["q_nope"] = _randn(g, (batch, q_tokens, c["heads"], c["d_nope"]), 1.0, c["dtype"])
    w["q_pe"] = _randn(g, (batch, q_tokens, c["heads"], c["d_rope"]), 1.0, c["dtype"])
    w["kind"] = "multi"
    w["q_tokens"] = q_tokens
    return w


def v2_b16_ctx4k_q4(seed=0):
    """DeepSeek-V2 attention shapes, 16 sequences of 4096 tokens, the last 4
    tokens of each decoded at once (a 4-token speculative step)."""
    return multi_token_decode(16, [4096] * 16, 4, seed=seed)


def token_decode(batch, ctx, seed=0, dtype="bf16", block_size=64, permute=False,
                 heads=128, d_latent=512, d_rope=64, d_nope=128, d_v=128, d_model=7168,
                 d_lq=1536, prior_rows="random"):
    """Full decode step: the current tokens' hidden states x drive the append
    and the query; the W_O projection maps the heads back to d_model.

    prior_rows: "random" draws the ctx-1 earlier cache rows directly;
    "append" leaves the pool zero and expects every row to be appended from
    `x_ctx` (all ctx tokens per sequence).
    d_lq: query latent width (0 = no query compression; queries from x).
    Draw order: block-table permutation, pool (if random), x (ctx tokens when
    appending, else the current token), w_dkv, w_dq (if d_lq), w_uq, w_uk,
    w_uv, w_o.
    """
    g = torch.Generator().manual_seed(seed)
    cfg = _cfg(heads, d_latent, d_rope, d_nope, d_v, block_size, dtype)
    seq_lens = [ctx] * batch
    bt, nblk = _pages(g, seq_lens, block_size, permute)
    dr = d_latent + d_rope
    if prior_rows == "random":
        cache = _randn(g, (nblk, block_size, dr), 1.0, dtype)
        x = _randn(g, (batch, d_model), 1.0, dtype)
        x_new, seq_idx_new = x, torch.arange(batch, dtype=torch.int32)
        pos_new = torch.full((batch,), ctx - 1, dtype=torch.int32)
    else:
        cache = torch.zeros((nblk, block_size, dr), dtype=torch_dtype(dtype))
        x_ctx = _randn(g, (batch, ctx, d_model), 1.0, dtype)
        x_new = x_ctx.reshape(batch * ctx, d_model)
        seq_idx_new = torch.arange(batch, dtype=torch.int32).repeat_interleave(ctx)
        pos_new = torch.arange(ctx, dtype=torch.int32).repeat(batch)
        x = x_ctx[:, ctx - 1, :].contiguous()
    w_dkv = _randn(g, (d_model, dr), 1.0 / math.sqrt(d_model), dtype)
    w_dq = _randn(g, (d_model, d_lq), 1.0 / math.sqrt(d_model), dtype) if d_lq else None
    q_in = d_lq if d_lq else d_model
    w_uq = _randn(g, (q_in, heads, d_nope + d_rope), 1.0 / math.sqrt(q_in), dtype)
    w_uk = _randn(g, (heads, d_latent, d_nope), 1.0 / math.sqrt(d_latent), dtype)
    w_uv = _randn(g, (heads, d_latent, d_v), 1.0 / math.sqrt(d_latent), dtype)
    w_o = _randn(g, (heads * d_v, d_model), 1.0 / math.sqrt(heads * d_v), dtype)
    return dict(cfg=cfg, kind="token", cache=cache, block_table=bt,
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32), x_new=x_new,
                seq_idx_new=seq_idx_new, pos_new=pos_new, x_q=x,
                pos_q=torch.full((batch,), ctx - 1, dtype=torch.int32), w_dkv=w_dkv,
                w_dq=w_dq, w_uq=w_uq, w_uk=w_uk, w_uv=w_uv, w_o=w_o, batch=batch,
                d_model=d_model, d_lq=d_lq)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_f32(seed=0):
    """Tiny fp32 decode: batch 1, 8 heads, d_in 256, d_L 64, qk_nope 32,
    rope 16, v 32; 128 context tokens all written by the append step; one
    query token (the last one); unpaged cache (one 128-token block)."""
    return token_decode(1, 128, seed=seed, dtype="f32", block_size=128, heads=8,
                        d_latent=64, d_rope=16, d_nope=32, d_v=32, d_model=256, d_lq=0,
                        prior_rows="append")


def v2_b16_ctx4k(seed=0):
    """DeepSeek-V2 shapes, bf16, batch 16, every context 4096, 64-token pages
    in order."""
    return cached_decode(16, [4096] * 16, seed=seed)


def v2_ragged_b64(seed=0):
    """DeepSeek-V2 shapes, bf16, batch 64, context lengths uniform in
    [1024, 8192], pages randomly permuted."""
    g = torch.Generator().manual_seed(seed + 7919)
    lens = torch.randint(1024, 8193, (64,), generator=g).tolist()
    return cached_decode(64, lens, seed=seed, permute=True)


def v2_long_b4_ctx100k(seed=0):
    """DeepSeek-V2 shapes, bf16, batch 4, contexts of 100,000 tokens."""
    return cached_decode(4, [100000] * 4, seed=seed)


def v2_layer_b128_ctx2k(seed=0):
    """Full layer decode step, bf16: hidden 7168, latent 512 + rotary 64,
    query latent 1536, 128 heads, batch 128, contexts 2048 (2047 earlier rows
    drawn directly, the current token's row appended)."""
    return token_decode(128, 2048, seed=seed)


WORKLOADS = {
    "tiny_f32": tiny_f32,
    "v2_b16_ctx4k": v2_b16_ctx4k,
    "v2_b16_ctx4k_q4": v2_b16_ctx4k_q4,
    "v2_ragged_b64": v2_ragged_b64,
    "v2_long_b4_ctx100k": v2_long_b4_ctx100k,
    "v2_layer_b128_ctx2k": v2_layer_b128_ctx2k,
}


def round_to(dtype):
    """Returns f(float array) -> float64 array rounded through `dtype`."""
    td = torch_dtype(dtype)

    def f(a):
        return torch.from_numpy(np.asarray(a, dtype=np.float64)).to(td).to(
            torch.float64).numpy()
    return f


def store_as(dtype):
    """Returns f(float array) -> the cache's storage array (bf16 bit patterns
    as uint16, or float32) holding the values rounded to `dtype`."""
    td = torch_dtype(dtype)

    def f(a):
        t = torch.from_numpy(np.asarray(a, dtype=np.float64)).to(td)
        if td == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return f


def _np(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.float().numpy()
    return t.numpy()


def oracle_view(w):
    """The workload's tensors as numpy arrays for the CPU reference.

    bf16 values are widened to fp32 (exact).  The cache is handed over as raw
    bf16 bit patterns (uint16) to avoid a multi-GB widened copy.
    """
    cfg = w["cfg"]
    out = dict(cfg=cfg, scale=cfg["softmax_scale"], round=round_to(cfg["dtype"]),
               store=store_as(cfg["dtype"]))
    for k, v in w.items():
        if k in ("cfg", "kind", "batch", "d_model", "d_lq", "q_tokens"):
            continue
        if k == "cache" and v.dtype == torch.bfloat16:
            out[k] = v.view(torch.int16).numpy().view(np.uint16)
        elif isinstance(v, torch.Tensor):
            out[k] = _np(v)
        else:
            out[k] = v
    return out
