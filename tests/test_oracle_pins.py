"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties the oracle to what the pages or mathematics fix: a library
routine for standard attention (torch's scaled_dot_product_attention in fp64),
a 50-digit brute force, closed forms, invariants, and the byte figures the
pages print.  The last group plants a plausible mistake in the oracle and
checks that at least one pin catches it.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------------------
# RoPE: the convention is a reading (interleaved pairs, theta_j = base^(-2j/d)).
# The pins below use the complex-number form of a rotation, not the oracle's
# cos/sin formula, plus the invariants every rotary embedding has.
# ---------------------------------------------------------------------------

def _rope_complex(v, pos, base):
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[0]
    z = v[0::2] + 1j * v[1::2]
    theta = base ** (-np.arange(d // 2) * 2.0 / d)
    z = z * np.exp(1j * pos * theta)
    out = np.empty(d)
    out[0::2] = z.real
    out[1::2] = z.imag
    return out


def test_rope_matches_complex_rotation():
    r = _rng(1)
    for d in (2, 8, 16, 64):
        for pos in (0, 1, 7, 1000, 99999):
            v = r.standard_normal(d)
            # fp64 angles pos*theta carry ~pos*1e-16 rad of rounding
            assert _rel(O.rope(v, pos), _rope_complex(v, pos, 10000.0)) < 1e-13 * max(10, pos)


def test_rope_first_pair_closed_form():
    # theta_0 = 1: the first pair of e_0 turns into (cos pos, sin pos)
    for pos in (0, 1, 2, 5):
        out = O.rope([1.0, 0.0], pos)
        assert abs(out[0] - math.cos(pos)) < 1e-15 and abs(out[1] - math.sin(pos)) < 1e-15


def test_rope_invariants():
    r = _rng(2)
    d = 64
    q, k = r.standard_normal(d), r.standard_normal(d)
    # position 0 is the identity; norms are preserved
    assert np.array_equal(O.rope(q, 0), q)
    for m in (3, 50, 4095):
        assert abs(np.linalg.norm(O.rope(q, m)) - np.linalg.norm(q)) < 1e-12
    # the dot product of rotated q and k depends only on the offset m - n
    base_dot = np.dot(O.rope(q, 10), O.rope(k, 4))
    for shift in (1, 100, 5000):
        assert abs(np.dot(O.rope(q, 10 + shift), O.rope(k, 4 + shift)) - base_dot) < 1e-9


# ---------------------------------------------------------------------------
# Standard multi-head attention as a library routine.
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, scale, causal=False):
    """q [H, m, d], k [H, n, d], v [H, n, dv] -> [H, m, dv] via torch, fp64."""
    tq = torch.from_numpy(np.ascontiguousarray(q))[None]
    tk = torch.from_numpy(np.ascontiguousarray(k))[None]
    tv = torch.from_numpy(np.ascontiguousarray(v))[None]
    return F.scaled_dot_product_attention(tq, tk, tv, scale=scale, is_causal=causal)[0].numpy()


def _small_token_problem(seed, d_r, B=2, H=3, n=9, d_in=12, d_l=5, d_n=4, d_v=3, d_lq=6,
                         d_model=7, block_size=4, permute=True):
    """Tiny random problem in the layout the oracle takes: every context row is
    written from x (positions 0..n-1), the query is the last token."""
    r = _rng(seed)
    x = r.standard_normal((B, n, d_in))
    w_dkv = r.standard_normal((d_in, d_l + d_r)) / math.sqrt(d_in)
    w_dq = r.standard_normal((d_in, d_lq)) / math.sqrt(d_in) if d_lq else None
    q_in = d_lq if d_lq else d_in
    w_uq = r.standard_normal((q_in, H, d_n + d_r)) / math.sqrt(q_in)
    w_uk = r.standard_normal((H, d_l, d_n)) / math.sqrt(d_l)
    w_uv = r.standard_normal((H, d_l, d_v)) / math.sqrt(d_l)
    w_o = r.standard_normal((H * d_v, d_model)) / math.sqrt(H * d_v)
    pages_per_seq = (n + block_size - 1) // block_size
    nblk = B * pages_per_seq
    ids = r.permutation(nblk) if permute else np.arange(nblk)
    bt = ids.reshape(B, pages_per_seq).astype(np.int32)
    cache = np.zeros((nblk, block_size, d_l + d_r))
    flat = cache.reshape(-1, d_l + d_r)
    for b in range(B):
        rows = O.latent_rows(x[b], w_dkv, d_l, d_r, np.arange(n))
        for i in range(n):
            flat[O.slot(bt, block_size, nblk, b, i)] = rows[i]
    pos_q = np.full(B, n - 1, dtype=np.int32)
    q_nope, q_pe = O.query(x[:, n - 1, :], w_uq, H, d_n, d_r, pos_q, w_dq=w_dq)
    return dict(x=x, w_dkv=w_dkv, w_dq=w_dq, w_uq=w_uq, w_uk=w_uk, w_uv=w_uv, w_o=w_o,
                bt=bt, cache=cache, q_nope=q_nope, q_pe=q_pe, B=B, H=H, n=n, d_in=d_in,
                d_l=d_l, d_r=d_r, d_n=d_n, d_v=d_v, d_lq=d_lq, d_model=d_model,
                scale=O.default_scale(d_n, d_r))


def _mha_reference(p, seq_len=None, causal_rows=False):
    """Standard MHA on explicitly multiplied-out weights, with torch SDPA.

    W_K = W_L W_LK, W_V = W_L W_LV, W_Q = W_LQ W_LQQ (the factorisation on
    "Multi-Head Latent Attention (MLA)", "The construction"); the decoupled
    rotary parts, when present, are appended to each head's query and key with
    the complex-rotation RoPE above.
    """
    B, H, n = p["B"], p["H"], p["n"] if seq_len is None else seq_len
    d_l, d_r, d_n = p["d_l"], p["d_r"], p["d_n"]
    W_L = p["w_dkv"][:, :d_l]
    W_KR = p["w_dkv"][:, d_l:]
    q_in = p["d_lq"] if p["d_lq"] else p["d_in"]
    w_uq = p["w_uq"].reshape(q_in, H, d_n + d_r)
    outs, o_heads = [], []
    for b in range(B):
        X = p["x"][b, :n]
        qs, ks, vs = [], [], []
        rows_q = X if causal_rows else X[n - 1:n]
        pos_rows = np.arange(n) if causal_rows else np.array([n - 1])
        cq = rows_q @ p["w_dq"] if p["w_dq"] is not None else rows_q
        kr = np.stack([_rope_complex(X[i] @ W_KR, i, 10000.0) for i in range(n)]) \
            if d_r else np.zeros((n, 0))
        for h in range(H):
            W_K = W_L @ p["w_uk"][h]            # d_in x d_n
            W_V = W_L @ p["w_uv"][h]            # d_in x d_v
            q_h = cq @ w_uq[:, h, :d_n]
            if d_r:
                qr = np.stack([_rope_complex(cq[j] @ w_uq[:, h, d_n:], pos_rows[j], 10000.0)
                               for j in range(cq.shape[0])])
                q_h = np.concatenate([q_h, qr], axis=1)
                k_h = np.concatenate([X @ W_K, kr], axis=1)
            else:
                k_h = X @ W_K
            qs.append(q_h)
            ks.append(k_h)
            vs.append(X @ W_V)
        o = _sdpa(np.stack(qs), np.stack(ks), np.stack(vs), p["scale"], causal=causal_rows)
        o_heads.append(o)                                # [H, m, d_v]
        stacked = np.concatenate([o[h] for h in range(H)], axis=1)   # [m, H*d_v]
        outs.append(stacked @ p["w_o"])
    return np.stack(outs), np.stack(o_heads)


def _oracle_run(p, seq_lens=None, plant=O.PLANT_NONE, w_o=True):
    B = p["B"]
    sl = np.full(B, p["n"], dtype=np.int32) if seq_lens is None else np.asarray(seq_lens)
    return O.decode(p["cache"], p["bt"], sl, p["q_nope"], p["q_pe"], p["w_uk"], p["w_uv"],
                    p["scale"], w_o=p["w_o"] if w_o else None, plant=plant)


@pytest.mark.parametrize("d_lq", [6, 0])
def test_no_rope_equals_mha_with_product_weights(d_lq):
    """Without the rotary part MLA is exactly an MHA whose weights are the
    products W_L W_LK, W_L W_LV, W_LQ W_LQQ ("The RoPE problem": without
    positional embeddings MLA is exactly equivalent)."""
    p = _small_token_problem(3, d_r=0, d_lq=d_lq)
    res = _oracle_run(p)
    out, o_heads = _mha_reference(p)
    assert _rel(res["out"], out[:, 0, :]) < 1e-12
    assert _rel(res["o_v"], o_heads[:, :, 0, :]) < 1e-12


def test_decoupled_rope_equals_mha_with_appended_rotary_parts():
    p = _small_token_problem(4, d_r=4)
    res = _oracle_run(p)
    out, o_heads = _mha_reference(p)
    assert _rel(res["out"], out[:, 0, :]) < 1e-12
    assert _rel(res["o_v"], o_heads[:, :, 0, :]) < 1e-12


def test_decode_step_is_last_row_of_causal_prefill():
    """Section 04 "The KV cache": decode at step t needs only query row t, and
    row t of full causal attention equals it; rows past seq_len are masked."""
    p = _small_token_problem(5, d_r=4, B=1)
    _, o_full = _mha_reference(p, causal_rows=True)     # [1, H, n, d_v]
    for t in range(p["n"]):
        pt = dict(p)
        pt["q_nope"], pt["q_pe"] = O.query(p["x"][:, t, :], p["w_uq"], p["H"], p["d_n"],
                                           p["d_r"], np.array([t], dtype=np.int32),
                                           w_dq=p["w_dq"])
        res = _oracle_run(pt, seq_lens=[t + 1], w_o=False)
        assert _rel(res["o_v"][0], o_full[0, :, t, :]) < 1e-12


@pytest.mark.parametrize("T", [1, 2, 4])
def test_multi_token_decode_is_last_rows_of_causal_prefill(T):
    """Several new tokens decoded at once are the last T rows of full causal
    attention (torch SDPA with its causal mask over explicitly multiplied-out
    keys), sequences of different lengths in one batch."""
    p = _small_token_problem(6, d_r=4, B=2)
    n = p["n"]
    _, o_full = _mha_reference(p, causal_rows=True)     # [B, H, n, d_v]
    lens = np.array([n, n - 1], dtype=np.int32)
    qn, qp = [], []
    for b in range(p["B"]):
        pos = np.arange(lens[b] - T, lens[b], dtype=np.int32)
        a, c = O.query(p["x"][b, pos, :], p["w_uq"], p["H"], p["d_n"], p["d_r"], pos,
                       w_dq=p["w_dq"])
        qn.append(a)
        qp.append(c)
    res = O.decode_multi(p["cache"], p["bt"], lens, np.stack(qn), np.stack(qp), p["w_uk"],
                         p["w_uv"], p["scale"])
    for b in range(p["B"]):
        for j in range(T):
            t = lens[b] - T + j
            assert _rel(res["o_v"][b, j], o_full[b, :, t, :]) < 1e-12


def test_merged_weights_give_the_same_scores_and_output():
    """The two merges of "Two merges are where the compute win comes from":
    W_LQK_h = W_LQQ_h W_LK_h^T acting on latents, and W_LO_h = W_LV_h W_O_h,
    built here as explicit product matrices."""
    p = _small_token_problem(6, d_r=0)
    res = _oracle_run(p)
    H, d_l, d_n, d_v = p["H"], p["d_l"], p["d_n"], p["d_v"]
    w_uq = p["w_uq"].reshape(p["d_lq"], H, d_n)
    for b in range(p["B"]):
        x_t = p["x"][b, -1]
        c_q = x_t @ p["w_dq"]
        C = np.stack([p["cache"].reshape(-1, d_l)[O.slot(p["bt"], 4, p["cache"].shape[0], b, i)]
                      for i in range(p["n"])])
        out = np.zeros(p["d_model"])
        for h in range(H):
            W_LQK = w_uq[:, h, :] @ p["w_uk"][h].T          # d_lq x d_l
            s = (c_q @ W_LQK) @ C.T * p["scale"]
            a = np.exp(s - s.max())
            a /= a.sum()
            W_LO = p["w_uv"][h] @ p["w_o"][h * d_v:(h + 1) * d_v]   # d_l x d_model
            out += (a @ C) @ W_LO
        assert _rel(res["out"][b], out) < 1e-12


# ---------------------------------------------------------------------------
# Brute force at 50 digits (tiny: 2 heads, at most 5 tokens, dims <= 4).
# ---------------------------------------------------------------------------

def test_mpmath_brute_force():
    mpmath.mp.dps = 50
    r = _rng(7)
    H, n, d_l, d_r, d_n, d_v = 2, 5, 4, 2, 3, 4
    C = r.standard_normal((n, d_l))
    KR = r.standard_normal((n, d_r))
    qn = r.standard_normal((H, d_n))
    qp = r.standard_normal((H, d_r))
    wk = r.standard_normal((H, d_l, d_n))
    wv = r.standard_normal((H, d_l, d_v))
    scale = 0.37
    cache = np.concatenate([C, KR], axis=1)[None]        # one block of n rows
    bt = np.zeros((1, 1), dtype=np.int32)
    res = O.decode(cache, bt, [n], qn[None], qp[None], wk, wv, scale)
    for h in range(H):
        s = []
        for i in range(n):
            k = [mpmath.fsum(mpmath.mpf(C[i, l]) * mpmath.mpf(wk[h, l, j]) for l in range(d_l))
                 for j in range(d_n)]
            dot = mpmath.fsum(mpmath.mpf(qn[h, j]) * k[j] for j in range(d_n)) + \
                mpmath.fsum(mpmath.mpf(qp[h, j]) * mpmath.mpf(KR[i, j]) for j in range(d_r))
            s.append(dot * mpmath.mpf(scale))
        z = mpmath.fsum(mpmath.e ** si for si in s)
        p = [mpmath.e ** si / z for si in s]
        for j in range(d_v):
            vj = mpmath.fsum(p[i] * mpmath.fsum(mpmath.mpf(C[i, l]) * mpmath.mpf(wv[h, l, j])
                                                for l in range(d_l)) for i in range(n))
            assert abs(float(vj) - res["o_v"][0, h, j]) < 1e-12
        for l in range(d_l):
            cl = mpmath.fsum(p[i] * mpmath.mpf(C[i, l]) for i in range(n))
            assert abs(float(cl) - res["o_lat"][0, h, l]) < 1e-12
        assert abs(float(mpmath.log(z)) - res["lse"][0, h]) < 1e-12


# ---------------------------------------------------------------------------
# Special cases and invariants.
# ---------------------------------------------------------------------------

def _cached_problem(seed, B=2, H=3, n=6, d_l=8, d_r=4, d_n=5, d_v=5, bs=4):
    r = _rng(seed)
    nb = B * ((n + bs - 1) // bs)
    cache = r.standard_normal((nb, bs, d_l + d_r))
    bt = r.permutation(nb).reshape(B, -1).astype(np.int32)
    return dict(cache=cache, bt=bt, q_nope=r.standard_normal((B, H, d_n)),
                q_pe=r.standard_normal((B, H, d_r)),
                w_uk=r.standard_normal((H, d_l, d_n)) / math.sqrt(d_l),
                w_uv=r.standard_normal((H, d_l, d_v)) / math.sqrt(d_l), B=B, H=H, n=n,
                d_l=d_l, d_r=d_r, bs=bs, scale=O.default_scale(d_n, d_r))


def _dec(p, seq_lens, plant=O.PLANT_NONE):
    return O.decode(p["cache"], p["bt"], seq_lens, p["q_nope"], p["q_pe"], p["w_uk"],
                    p["w_uv"], p["scale"], plant=plant)


def _row(p, b, i):
    return p["cache"].reshape(-1, p["d_l"] + p["d_r"])[O.slot(p["bt"], p["bs"],
                                                               p["cache"].shape[0], b, i)]


def test_single_token_returns_its_value():
    """seq_len 1: the only weight is 1, so o_lat is that latent, o_v its value
    and lse its score."""
    p = _cached_problem(8)
    res = _dec(p, [1, 1])
    for b in range(p["B"]):
        row = _row(p, b, 0)
        c, kr = row[:p["d_l"]], row[p["d_l"]:]
        for h in range(p["H"]):
            assert np.allclose(res["o_lat"][b, h], c, rtol=0, atol=1e-14)
            assert np.allclose(res["o_v"][b, h], c @ p["w_uv"][h], rtol=0, atol=1e-13)
            s = (p["q_nope"][b, h] @ (c @ p["w_uk"][h]) + p["q_pe"][b, h] @ kr) * p["scale"]
            assert abs(res["lse"][b, h] - s) < 1e-12


def test_identical_rows_give_uniform_weights():
    p = _cached_problem(9)
    row = p["cache"][0, 0].copy()
    p["cache"][:] = row
    n = 6
    res = _dec(p, [n, n - 1])
    for b, m in ((0, n), (1, n - 1)):
        for h in range(p["H"]):
            assert np.allclose(res["o_lat"][b, h], row[:p["d_l"]], atol=1e-13)
            one = (p["q_nope"][b, h] @ (row[:p["d_l"]] @ p["w_uk"][h]) +
                   p["q_pe"][b, h] @ row[p["d_l"]:]) * p["scale"]
            assert abs(res["lse"][b, h] - (one + math.log(m))) < 1e-12


def test_output_is_a_convex_combination_of_visible_latents():
    """Softmax rows are non-negative and sum to 1, so every coordinate of
    o_lat lies between the smallest and largest visible latent coordinate."""
    p = _cached_problem(10, n=8)
    for lens in ([8, 3], [5, 8]):
        res = _dec(p, lens)
        for b in range(p["B"]):
            C = np.stack([_row(p, b, i)[:p["d_l"]] for i in range(lens[b])])
            lo, hi = C.min(axis=0), C.max(axis=0)
            for h in range(p["H"]):
                assert np.all(res["o_lat"][b, h] >= lo - 1e-12)
                assert np.all(res["o_lat"][b, h] <= hi + 1e-12)


def test_masked_slots_do_not_leak():
    """Rows past seq_len (same page, later slots) never affect the result."""
    p = _cached_problem(11, n=8)
    a = _dec(p, [5, 7])
    for b, n in ((0, 5), (1, 7)):
        for i in range(n, 8):
            flat = p["cache"].reshape(-1, p["d_l"] + p["d_r"])
            flat[O.slot(p["bt"], p["bs"], p["cache"].shape[0], b, i)] = 1e3
    c = _dec(p, [5, 7])
    assert np.array_equal(a["o_lat"], c["o_lat"]) and np.array_equal(a["lse"], c["lse"])


def test_page_permutation_is_invisible():
    p = _cached_problem(12, n=8)
    a = _dec(p, [8, 6])
    perm = _rng(13).permutation(p["cache"].shape[0])
    inv = np.argsort(perm)
    q = dict(p)
    q["cache"] = p["cache"][perm]          # physical page k now holds old page perm[k]
    q["bt"] = inv[p["bt"]].astype(np.int32)
    c = _dec(q, [8, 6])
    assert np.array_equal(a["o_lat"], c["o_lat"]) and np.array_equal(a["o_v"], c["o_v"])


def test_multi_token_first_token_sees_only_its_prefix():
    """Several new tokens: the first of T tokens of a sequence of n attends to
    n - T + 1 rows, so changing any of the T - 1 newest rows leaves it
    unchanged and changes the last token (the causal mask of section 03); a
    token's result equals a one-token decode of the same query over the
    sequence cut at its position, brute force by single-element loops."""
    p = _cached_problem(21, n=8)
    T, lens = 3, [8, 6]
    r = _rng(22)
    qn = r.standard_normal((p["B"], T, p["H"], p["q_nope"].shape[2]))
    qp = r.standard_normal((p["B"], T, p["H"], p["d_r"]))
    a = O.decode_multi(p["cache"], p["bt"], lens, qn, qp, p["w_uk"], p["w_uv"], p["scale"])
    q = dict(p)
    q["cache"] = p["cache"].copy()
    flat = q["cache"].reshape(-1, p["d_l"] + p["d_r"])
    for b, n in enumerate(lens):
        for i in range(n - T + 1, n):
            flat[O.slot(p["bt"], p["bs"], p["cache"].shape[0], b, i)] += 0.5
    c = O.decode_multi(q["cache"], p["bt"], lens, qn, qp, p["w_uk"], p["w_uv"], p["scale"])
    assert np.array_equal(a["o_lat"][:, 0], c["o_lat"][:, 0])
    assert not np.allclose(a["o_lat"][:, T - 1], c["o_lat"][:, T - 1])
    # token j of sequence b, head h, by hand: scores over rows 0..n-T+j
    for b, n in enumerate(lens):
        for j in range(T):
            m = n - T + 1 + j
            for h in range(p["H"]):
                qlat = p["w_uk"][h] @ qn[b, j, h]                 # [d_l]
                s = np.array([p["scale"] * (qlat @ _row(p, b, i)[:p["d_l"]] +
                                            qp[b, j, h] @ _row(p, b, i)[p["d_l"]:])
                              for i in range(m)])
                w = np.exp(s - s.max())
                w /= w.sum()
                o = sum(w[i] * _row(p, b, i)[:p["d_l"]] for i in range(m))
                assert _rel(a["o_lat"][b, j, h], o) < 1e-12


def test_index_map_golden():
    with open(os.path.join(GOLDEN, "paged_index_map.json")) as f:
        g = json.load(f)
    bt = np.array(g["block_table"], dtype=np.int32)
    for case in g["cases"]:
        assert O.slot(bt, g["block_size"], g["num_blocks"], case["b"], case["i"]) == case["row"]


def test_scatter_writes_only_its_slots():
    bs, nb, row_bytes = 4, 5, 6
    bt = np.array([[2, 0, 3], [4, 1, -1]], dtype=np.int32)
    cache = np.full((nb * bs, row_bytes), 0xAB, dtype=np.uint8)
    rows = np.arange(3 * row_bytes, dtype=np.uint8).reshape(3, row_bytes)
    skipped = O.scatter_rows(rows, [0, 1, 1], [9, 5, 8], bt, bs, cache)
    assert skipped == 1                    # (b=1, i=8) points at block -1
    expect = np.full_like(cache, 0xAB)
    expect[13] = rows[0]
    expect[5] = rows[1]
    assert np.array_equal(cache, expect)


def test_cache_byte_figures_from_the_pages():
    with open(os.path.join(GOLDEN, "cache_bytes_pages.json")) as f:
        g = json.load(f)
    H, D, nb = g["heads"]["value"], g["head_dim"]["value"], g["bytes_per_number"]["value"]
    per_layer = O.kv_numbers_per_token(H, D, 1) * nb
    layers = round(g["mha_bytes_per_token"]["value"] / per_layer)   # R1: 61 layers

    def close(x, key):
        e = g[key]
        return abs(x - e["value"]) <= e["rel_tol"] * e["value"]

    assert O.latent_numbers_per_token(g["latent"]["value"], g["rope"]["value"], 1) == \
        g["mla_numbers_per_token_per_layer"]["value"]
    mha = O.kv_numbers_per_token(H, D, layers) * nb
    gqa8 = O.kv_numbers_per_token(H // 8, D, layers) * nb
    mla = O.latent_numbers_per_token(512, 64, layers) * nb
    assert close(mha, "mha_bytes_per_token")
    assert close(gqa8, "gqa8_bytes_per_token")
    assert close(mla, "mla_bytes_per_token")
    assert close(mha / mla, "mha_over_mla")
    assert close(mha * 100000, "reads_at_100k_context_bytes")
    groups = O.latent_numbers_per_token(512, 64, 1) / O.kv_numbers_per_token(1, D, 1)
    assert close(groups, "gqa_groups_matching_mla")


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin above.
# ---------------------------------------------------------------------------

def test_planted_rope_sign_is_caught():
    v = _rng(14).standard_normal(8)
    assert _rel(O.rope(v, 5, plant=O.PLANT_ROPE_SIGN), _rope_complex(v, 5, 10000.0)) > 1e-3


@pytest.mark.parametrize("plant", [O.PLANT_DROP_ROPE_TERM, O.PLANT_TRANSPOSE_WLK,
                                   O.PLANT_NO_SCALE, O.PLANT_VALUE_FROM_KEY,
                                   O.PLANT_MASK_OFF_BY_ONE])
def test_planted_decode_mistakes_are_caught(plant):
    p = _small_token_problem(15, d_r=4, d_n=4, d_v=4)
    res = _oracle_run(p, plant=plant)
    out, o_heads = _mha_reference(p)
    assert _rel(res["o_v"], o_heads[:, :, 0, :]) > 1e-3
