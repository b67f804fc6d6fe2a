"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Metric: max|gpu - ref| / max|ref| over a whole tensor (or over the sampled
rows at full size).  Bars: 5e-3 for bf16 inputs with fp32 accumulation, 1e-5
for fp32.  Cache indexing (which slots the append writes) is bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle as O
from head_latent_attention_23_b300 import mla, workloads as W
from head_latent_attention_23_b300.runner import DecodeStep

pytestmark = pytest.mark.gpu

TOL = {"bf16": 5e-3, "f32": 1e-5}


def rel(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all()
    return float(np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30))


def host(t):
    return t.detach().float().cpu().numpy()


def run_step(w):
    step = DecodeStep(w)
    step.run()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    return step


def check_pairs(step, ref, pairs, tol):
    res = step.results()
    bi = np.array([b for b, _ in pairs])
    hi = np.array([h for _, h in pairs])
    for key in ("o_lat", "o_v", "lse"):
        g = host(res[key])[bi, hi]
        r = np.asarray(ref[key])[bi, hi]
        assert rel(g, r) <= tol, key


# ---------------------------------------------------------------- small cases

def test_tiny_f32_full_step():
    """fp32, 8 heads, 128 tokens appended from x, one query: every output."""
    w = W.tiny_f32()
    step = run_step(w)
    ref = O.reference_token_decode(W.oracle_view(w))
    tol = TOL["f32"]
    res = step.results()
    assert rel(host(step.cache).reshape(-1, 80)[:128], ref["rows"]) <= tol
    assert rel(host(res["q_nope"]), ref["q_nope"]) <= tol
    assert rel(host(res["q_pe"]), ref["q_pe"]) <= tol
    for key in ("o_lat", "o_v", "lse", "out"):
        assert rel(host(res[key]), ref[key]) <= tol, key


@pytest.mark.parametrize("lens,permute", [([1, 63, 64, 65, 200, 1000], True),
                                          ([129, 4, 777], False)])
def test_decode_small_ragged_bf16(lens, permute):
    """DeepSeek-V2 head/latent shapes, ragged lengths around the 64-token tile
    and page boundaries, all (sequence, head) pairs."""
    w = W.cached_decode(len(lens), lens, seed=11, permute=permute)
    step = run_step(w)
    ref = O.reference_cached_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key


@pytest.mark.parametrize("batch", [1, 15, 17, 64, 65])
def test_projection_modes_around_the_skinny_limit(batch):
    """The per-head absorb and value projections run transposed (weights as
    the MMA's 128-row side) up to 64 rows and tiled above; batch sizes on both
    sides of the limit and of the 16-row padding, every (sequence, head) pair
    of q_lat-dependent o_lat, lse and o_v against the oracle."""
    g = torch.Generator().manual_seed(batch)
    lens = torch.randint(1, 200, (batch,), generator=g).tolist()
    w = W.cached_decode(batch, lens, seed=60 + batch, permute=True)
    step = run_step(w)
    ref = O.reference_cached_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key


def _guarded(shape, dtype, guard=4096):
    """A tensor of `shape` inside a larger buffer whose guard bands before and
    after hold a canary pattern; returns (view, check) where check() is True
    while the bands are intact."""
    n = int(np.prod(shape))
    buf = torch.full((guard + n + guard,), -77.0, dtype=dtype, device="cuda")
    view = buf[guard:guard + n].view(*shape)
    canary = torch.full((guard,), -77.0, dtype=dtype, device="cuda")

    def check():
        torch.cuda.synchronize()
        return torch.equal(buf[:guard], canary) and torch.equal(buf[guard + n:], canary)
    return view, check


def test_outputs_stay_inside_their_buffers():
    """Canary guard bands around every output of the absorb, decode, merge,
    value projection and multi-token calls (a stand-in for a memory checker):
    the bands are intact afterwards and the outputs match the oracle."""
    lens = [1, 63, 64, 65, 200, 700]
    w = W.cached_decode(len(lens), lens, seed=70, permute=True)
    cfg = mla.config_from(w["cfg"])
    d = {k: w[k].cuda() for k in ("cache", "block_table", "seq_lens", "q_nope", "q_pe",
                                  "w_uk", "w_uv")}
    B = len(lens)
    q_lat, c1 = _guarded((B, 128, 512), torch.bfloat16)
    o_lat, c2 = _guarded((B, 128, 512), torch.bfloat16)
    lse, c3 = _guarded((B, 128), torch.float32)
    o_v, c4 = _guarded((B, 128, 128), torch.bfloat16)
    mla.absorb_q(cfg, d["q_nope"], d["w_uk"], q_lat)
    mla.decode(cfg, q_lat, d["q_pe"], d["cache"], d["block_table"], d["seq_lens"], o_lat, lse)
    mla.project_out(cfg, o_lat, d["w_uv"], o_v)
    assert c1() and c2() and c3() and c4()
    assert mla.get_status() == mla.MLA_OK
    ref = O.reference_cached_decode(W.oracle_view(w))
    assert rel(host(o_lat), ref["o_lat"]) <= TOL["bf16"]
    assert rel(host(o_v), ref["o_v"]) <= TOL["bf16"]

    T = 3
    wm = W.multi_token_decode(3, [3, 90, 200], T, seed=71)
    dm = {k: wm[k].cuda() for k in ("cache", "block_table", "seq_lens", "q_nope", "q_pe",
                                    "w_uk")}
    ql = torch.empty((3 * T, 128, 512), dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(cfg, dm["q_nope"].reshape(3 * T, 128, -1), dm["w_uk"], ql)
    om, c5 = _guarded((3, T, 128, 512), torch.bfloat16)
    lm, c6 = _guarded((3, T, 128), torch.float32)
    mla.decode_multi(cfg, ql.view(3, T, 128, 512), dm["q_pe"], dm["cache"], dm["block_table"],
                     dm["seq_lens"], om, lm)
    assert c5() and c6()
    assert mla.get_status() == mla.MLA_OK
    refm = O.reference_multi_decode(W.oracle_view(wm))
    assert rel(host(om), refm["o_lat"]) <= TOL["bf16"]


def test_seq_len_one_returns_the_cached_latent():
    w = W.cached_decode(3, [1, 1, 1], seed=5, permute=True)
    step = run_step(w)
    c = w["cache"].float().numpy()
    bt = w["block_table"].numpy()
    o = host(step.o_lat)
    for b in range(3):
        row = c[bt[b, 0], 0, :512]
        assert np.array_equal(o[b], np.broadcast_to(row, o[b].shape))


def test_masked_slots_do_not_leak():
    """Rows after seq_len in the last page hold huge values; they must not
    change the result."""
    w = W.cached_decode(2, [70, 5], seed=6)
    a = run_step(w)
    o1 = host(a.o_lat).copy()
    bt = w["block_table"].numpy()
    w["cache"][bt[0, 1], 6:] = 1e4
    w["cache"][bt[1, 0], 5:] = -1e4
    b = run_step(w)
    assert np.array_equal(o1, host(b.o_lat))


@pytest.mark.parametrize("max_pos", [256, 100000])
def test_append_indexing_is_bit_exact(max_pos):
    """The append's rows scattered by the oracle's index map reproduce the GPU
    cache byte for byte; every other slot keeps its canary.  Positions up to
    100,000 exercise the rotary angles of the long-context workloads."""
    for dtype, tol in (("bf16", TOL["bf16"]), ("f32", TOL["f32"])):
        g = torch.Generator().manual_seed(3)
        cfg = mla.config(128, 512, 64, 128, 128, 64, dtype)
        td = W.torch_dtype(dtype)
        B, n_tok, d_in = 3, 40, 320
        maxb = (max_pos + 63) // 64
        seq_idx = torch.randint(0, B, (n_tok,), generator=g).to(torch.int32)
        pos = torch.randint(0, max_pos, (n_tok,), generator=g).to(torch.int32)
        # distinct (seq, pos) so no two tokens target the same slot
        key = seq_idx.long() * 1000000 + pos.long()
        keep = torch.unique(key, return_inverse=False)
        seq_idx = (keep // 1000000).to(torch.int32)
        pos = (keep % 1000000).to(torch.int32)
        n_tok = seq_idx.numel()
        # a page per (sequence, page index) that some token uses, in a permuted
        # pool; the table's other entries point at pages no token writes
        used = sorted({(int(b), int(p) // 64) for b, p in zip(seq_idx, pos)})
        nb = len(used) + 4
        ids = torch.randperm(nb, generator=g)
        bt = torch.full((B, maxb), int(ids[-1]), dtype=torch.int32)
        for i, (b, pg) in enumerate(used):
            bt[b, pg] = int(ids[i])
        x = torch.randn(n_tok, d_in, generator=g).to(td)
        w_dkv = (torch.randn(d_in, 576, generator=g) / d_in ** 0.5).to(td)
        canary = torch.full((nb, 64, 576), 7.25, dtype=td)
        cache = canary.cuda()
        dense = torch.empty((n_tok, 576), dtype=td, device="cuda")
        mla.append_latent(cfg, x.cuda(), w_dkv.cuda(), seq_idx.cuda(), pos.cuda(), bt.cuda(),
                          cache, dense)
        torch.cuda.synchronize()
        assert mla.get_status() == mla.MLA_OK
        esz = 2 if dtype == "bf16" else 4
        expect = canary.view(torch.uint8).numpy().reshape(nb * 64, 576 * esz).copy()
        rows_u8 = dense.cpu().view(torch.uint8).numpy().reshape(n_tok, 576 * esz)
        assert O.scatter_rows(rows_u8, seq_idx.numpy(), pos.numpy(), bt.numpy(), 64,
                              expect) == 0
        got = cache.cpu().view(torch.uint8).numpy().reshape(nb * 64, 576 * esz)
        assert np.array_equal(got, expect)
        ref = O.latent_rows(x.float().numpy(), w_dkv.float().numpy(), 512, 64, pos.numpy())
        assert rel(dense.float().cpu().numpy(), ref) <= tol


def test_growing_scores_take_the_rescale_path():
    """Cache rows scaled up geometrically page by page make the score maximum
    of later tiles exceed the running one by more than the lazy-rescale
    threshold (2^8), so the kernels rescale their accumulators many times in
    the 1000-token sequence (about 80 head-tile events; logits reach ~11),
    with an ordinary (rounded) absorbed query; the result must still match
    the oracle everywhere.  The large-logit regime is covered by the next
    test, whose absorbed query is exact in bf16."""
    w = W.growing_scores_decode()      # premise checked on the CPU in test_workloads.py
    step = run_step(w)
    ref = O.reference_cached_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key


def test_large_logits_with_an_exact_query_take_hundreds_of_rescales():
    """One-hot q_nope makes q_lat = q_nope . W_LK_h^T a column of W_LK_h, exact
    in bf16, so the oracle and the GPU see the same logits; cache pages grow
    by 1 + 1.5 j, so logits reach ~58 and the running maximum moves past the
    2^8 threshold hundreds of times (both checked on the CPU in
    test_workloads.py).  Every output at the bf16 bar."""
    w = W.growing_scores_exact_query_decode()
    step = run_step(w)
    ref = O.reference_cached_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key


def test_split_ranges_crossing_sequences_all_pairs():
    """80 sequences of 1-700 tokens (one of 37 in the middle), pages permuted:
    the context is at least three 128-token tiles per split worker, and most
    workers' tile ranges hold the end of one sequence and the start of the
    next, so the kernel reloads the query and writes several partials inside
    one range.  Each row of the attention pattern sums to one over all of its
    sequence's tokens ("How DeepSeek Rewrote the Transformer (MLA)", section
    03): a split that drops or double-counts a piece fails on the pairs it
    touches, so every (sequence, head) pair of o_lat and lse is compared."""
    w = W.crossing_ranges_decode()
    cfg = mla.config_from(w["cfg"])
    d = {k: w[k].cuda() for k in ("cache", "block_table", "seq_lens", "q_nope", "q_pe",
                                  "w_uk")}
    B = w["batch"]
    q_lat = torch.empty((B, 128, 512), dtype=torch.bfloat16, device="cuda")
    o_lat = torch.empty_like(q_lat)
    lse = torch.empty((B, 128), dtype=torch.float32, device="cuda")
    mla.absorb_q(cfg, d["q_nope"], d["w_uk"], q_lat)
    mla.decode(cfg, q_lat, d["q_pe"], d["cache"], d["block_table"], d["seq_lens"], o_lat, lse)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    ref = O.reference_cached_decode(W.oracle_view(w))
    assert rel(host(o_lat), ref["o_lat"]) <= TOL["bf16"]
    assert rel(host(lse), ref["lse"]) <= TOL["bf16"]


# ---------------------------------------------------------------- several new tokens

@pytest.mark.parametrize("T,lens", [(2, [2, 3, 64, 65, 129, 700]),
                                    (4, [4, 5, 127, 128, 131, 1000, 3000])])
def test_multi_token_decode_all_pairs(T, lens):
    """The last T tokens of each sequence decoded at once, token j seeing the
    n - T + 1 + j tokens up to it (causal mask, "How DeepSeek Rewrote the
    Transformer (MLA)", section 03).  Lengths put the first new token on one
    row (n = T) and the masked edge on both sides of the 64-token page and
    128-token tile boundaries; pages permuted.  Every (sequence, token, head)
    triple of o_lat, o_v and lse."""
    w = W.multi_token_decode(len(lens), lens, T, seed=40 + T)
    step = run_step(w)
    ref = O.reference_multi_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key


def test_multi_token_decode_mask_and_single_token_equivalence():
    """Raising the newest cached row of each sequence changes the outputs of
    its last new token only; the other tokens stay bit-identical.  With one
    new token the call equals mla_decode bit for bit."""
    T, lens = 3, [3, 90, 200]
    w = W.multi_token_decode(len(lens), lens, T, seed=52)
    a = run_step(w)
    o1 = host(a.results()["o_lat"]).copy()
    bt = w["block_table"].numpy()
    for b, n in enumerate(lens):
        w["cache"][bt[b, (n - 1) // 64], (n - 1) % 64, :] *= 3.0
    o2 = host(run_step(w).results()["o_lat"])
    assert np.array_equal(o1[:, :T - 1], o2[:, :T - 1])
    for b in range(len(lens)):
        assert not np.array_equal(o1[b, T - 1], o2[b, T - 1])

    w1 = W.multi_token_decode(len(lens), lens, 1, seed=53)
    m = run_step(w1)
    cfg = mla.config_from(w1["cfg"])
    o_lat = torch.empty_like(m.o_lat)
    lse = torch.empty_like(m.lse)
    mla.decode(cfg, m.q_lat, m.q_pe.view(len(lens), 128, -1), m.cache, m.block_table,
               m.seq_lens, o_lat, lse)
    torch.cuda.synchronize()
    assert torch.equal(o_lat, m.o_lat) and torch.equal(lse, m.lse)


def test_multi_token_full_size_sampled():
    """16 sequences of 4096 tokens, the last 4 of each decoded at once: all
    tokens and heads of sequences 0, 7 and 15."""
    w = W.v2_b16_ctx4k_q4()
    step = run_step(w)
    pairs = [(b, j, h) for b in (0, 7, 15) for j in range(4) for h in range(128)]
    ref = O.reference_multi_decode(W.oracle_view(w), pairs=pairs)
    res = step.results()
    bi = np.array([p[0] for p in pairs])
    ji = np.array([p[1] for p in pairs])
    hi = np.array([p[2] for p in pairs])
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key])[bi, ji, hi], np.asarray(ref[key])[bi, ji, hi]) <= \
            TOL["bf16"], key


def _host_pinned(t):
    return t.cpu().pin_memory()


def test_layer_decode_step_single_call_matches_oracle():
    """mla_layer_decode_step (one call: query projection, append of each
    sequence's newest row, absorb, decode, W_LV and W_O) on a small full
    layer (hidden 1024, query latent 256, DeepSeek-V2 head and latent widths,
    batch 4, contexts 300), all outputs against the oracle; the host-buffer
    form of the call returns the same bytes as the device form."""
    w = W.token_decode(4, 300, seed=17, d_model=1024, d_lq=256, permute=True)
    step = DecodeStep(w)
    assert step.fused
    step.run_fused()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    ref = O.reference_token_decode(W.oracle_view(w))
    assert rel(host(step.out), ref["out"]) <= TOL["bf16"]
    got = host(step.cache).reshape(-1, 576)
    v = W.oracle_view(w)
    rows = O.latent_rows(v["x_new"], v["w_dkv"], 512, 64, v["pos_new"])
    for b in range(4):
        pg = int(v["block_table"][b, 299 // 64])
        assert rel(got[pg * 64 + 299 % 64], rows[b]) <= TOL["bf16"]
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    inputs = dict(x=_host_pinned(step.x_q), seq_lens=_host_pinned(step.seq_lens),
                  block_table=_host_pinned(step.block_table))
    step.run_fused(io_flags=mla.IO_HOST_INPUTS | mla.IO_HOST_OUTPUT, inputs=inputs, result=out_h)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    assert torch.equal(out_h, step.out.cpu())


def test_cached_decode_step_single_call_matches_oracle():
    """mla_cached_decode_step (absorb, decode, W_LV in one call) against the
    oracle, ragged lengths with permuted pages; host-buffer form equal to the
    device form."""
    w = W.cached_decode(3, [129, 1, 900], seed=19, permute=True)
    step = DecodeStep(w)
    step.run_fused()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    ref = O.reference_cached_decode(W.oracle_view(w))
    res = step.results()
    for key in ("o_lat", "o_v", "lse"):
        assert rel(host(res[key]), ref[key]) <= TOL["bf16"], key
    o_h = torch.empty(step.o_v.shape, dtype=step.o_v.dtype).pin_memory()
    inputs = {k: _host_pinned(getattr(step, k)) for k in ("q_nope", "q_pe", "seq_lens",
                                                          "block_table")}
    step.run_fused(io_flags=mla.IO_HOST_INPUTS | mla.IO_HOST_OUTPUT, inputs=inputs, result=o_h)
    torch.cuda.synchronize()
    assert torch.equal(o_h, step.o_v.cpu())


def test_invalid_block_id_is_flagged_not_read():
    w = W.cached_decode(2, [100, 100], seed=8)
    w["block_table"][1, 1] = 10 ** 6
    step = DecodeStep(w)
    step.run()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_ERR_INDEX
    assert mla.get_status() == mla.MLA_OK          # reading clears it
    # the intact sequence is still right
    ref = O.reference_cached_decode(W.oracle_view(W.cached_decode(2, [100, 100], seed=8)),
                                    pairs=[(0, h) for h in range(128)])
    assert rel(host(step.o_lat[0]), ref["o_lat"][0]) <= TOL["bf16"]


def test_combine_of_oracle_partials_equals_full_attention():
    """Two page-aligned token ranges decoded separately by the oracle, merged
    by mla_decode_combine, equal the oracle over the whole sequence.  A third,
    empty range (lse = -inf) must not contribute."""
    w = W.cached_decode(2, [256, 192], seed=9)
    v = W.oracle_view(w)
    full = O.reference_cached_decode(v)
    bt = v["block_table"]
    parts = []
    for lo_page, hi_page in ((0, 2), (2, 4)):
        sub_bt = np.full_like(bt, -1)
        lens = []
        for b in range(2):
            n_pages = (int(v["seq_lens"][b]) + 63) // 64
            hp = min(hi_page, n_pages)
            sub_bt[b, :hp - lo_page] = bt[b, lo_page:hp]
            lens.append(min(int(v["seq_lens"][b]), hp * 64) - lo_page * 64)
        parts.append(O.decode(v["cache"], sub_bt, lens, v["q_nope"], v["q_pe"], v["w_uk"],
                              v["w_uv"], v["scale"]))
    o_part = np.stack([p["o_lat"] for p in parts] + [np.zeros_like(parts[0]["o_lat"])])
    lse_part = np.stack([p["lse"] for p in parts] + [np.full_like(parts[0]["lse"], -np.inf)])
    cfg = mla.config_from(w["cfg"])
    o_lat = torch.empty((2, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 128), dtype=torch.float32, device="cuda")
    mla.decode_combine(cfg, torch.from_numpy(o_part).float().cuda(),
                       torch.from_numpy(lse_part).float().cuda(), o_lat, lse)
    torch.cuda.synchronize()
    assert rel(host(o_lat), full["o_lat"]) <= TOL["bf16"]
    assert rel(host(lse), full["lse"]) <= 1e-5


# ---------------------------------------------------------------- full size

def _checked_pairs(name, w):
    """(sequence, head) pairs compared at full size: all 128 heads of four
    sequences (batch 16 x 4096: sequences 0, 5, 10, 15, each spread over
    about five split workers whose ranges start or end inside it; ragged
    batch 64: its four shortest sequences), or four heads of every sequence
    of the 100,000-token batch (one sequence there costs the oracle minutes)."""
    lens = w["seq_lens"].tolist()
    if name == "v2_b16_ctx4k":
        seqs, heads = [0, 5, 10, 15], range(128)
    elif name == "v2_ragged_b64":
        seqs, heads = sorted(range(len(lens)), key=lambda b: lens[b])[:4], range(128)
    else:
        seqs, heads = range(len(lens)), (0, 37, 90, 127)
    return [(b, h) for b in seqs for h in heads]


@pytest.mark.parametrize("name", ["v2_b16_ctx4k", "v2_ragged_b64", "v2_long_b4_ctx100k"])
def test_full_size_cached_workloads_sampled(name):
    w = W.WORKLOADS[name]()
    step = run_step(w)
    pairs = _checked_pairs(name, w)
    ref = O.reference_cached_decode(W.oracle_view(w), pairs=pairs)
    check_pairs(step, ref, pairs, TOL["bf16"])


def test_full_layer_step_sampled():
    """hidden 7168 -> latent + rotary append, query latent 1536, 128 heads,
    batch 128, contexts 2048; out = W_O projection of all heads of one
    sequence, plus sampled (sequence, head) pairs."""
    w = W.v2_layer_b128_ctx2k()
    step = run_step(w)
    v = W.oracle_view(w)
    seqs = [0, 77]
    ref = O.reference_token_decode(v, seqs=[77])
    assert rel(host(step.out[77]), ref["out"][0]) <= TOL["bf16"]
    pairs = [(0, 0), (0, 127), (1, 5), (1, 64)]
    ref2 = O.reference_token_decode(v, seqs=seqs, pairs=pairs)
    res = step.results()
    for key in ("o_lat", "o_v"):
        g = np.stack([host(res[key][seqs[i], h]) for i, h in pairs])
        r = np.stack([ref2[key][i, h] for i, h in pairs])
        assert rel(g, r) <= TOL["bf16"], key
