"""The seeded input generators: determinism and the shapes the pages give."""
import numpy as np
import torch

from head_latent_attention_23_b300 import workloads as W


def test_seeded_and_deterministic():
    a = W.cached_decode(2, [70, 5], seed=3, permute=True)
    b = W.cached_decode(2, [70, 5], seed=3, permute=True)
    for k in ("cache", "q_nope", "q_pe", "w_uk", "w_uv", "block_table"):
        assert torch.equal(a[k], b[k])
    c = W.cached_decode(2, [70, 5], seed=4, permute=True)
    assert not torch.equal(a["cache"], c["cache"])


def test_block_table_pages_are_distinct():
    w = W.cached_decode(5, [1, 63, 64, 65, 300], seed=1, permute=True)
    bt = w["block_table"].numpy()
    used = [bt[b, :(n + 63) // 64] for b, n in enumerate([1, 63, 64, 65, 300])]
    ids = np.concatenate(used)
    assert len(set(ids.tolist())) == len(ids) == w["cache"].shape[0]
    assert (bt[0, 1:] == -1).all()


def test_named_workload_shapes():
    w = W.tiny_f32()
    assert w["cache"].dtype == torch.float32 and w["cache"].shape == (1, 128, 80)
    assert w["x_new"].shape == (128, 256) and w["w_uq"].shape == (256, 8, 48)
    v = W.oracle_view(W.cached_decode(1, [3], heads=4, d_latent=8, d_rope=4, d_nope=4, d_v=4))
    assert v["cache"].dtype == np.uint16


def test_growing_scores_inputs_cross_the_rescale_threshold_with_moderate_logits():
    """Premise of the GPU rescale test: along sequence 0 the maximum of a
    128-token tile's scores exceeds the running maximum by more than 8 (log2
    units, the kernels' lazy-rescale threshold) many times over the heads,
    while every logit stays below 15, where the bf16 tolerance holds."""
    w = W.growing_scores_decode()
    cfg = w["cfg"]
    dl, D = cfg["d_latent"], cfg["d_latent"] + cfg["d_rope"]
    n = int(w["seq_lens"][0])
    tok = torch.arange(n)
    slot = w["block_table"][0].long()[tok // 64] * 64 + tok % 64
    rows = w["cache"].reshape(-1, D)[slot].double()
    q_lat = torch.einsum("hn,hln->hl", w["q_nope"][0].double(), w["w_uk"].double())
    s = cfg["softmax_scale"] * (q_lat @ rows[:, :dl].T + w["q_pe"][0].double() @ rows[:, dl:].T)
    s2 = (s / np.log(2.0)).numpy()
    events = 0
    for h in range(s2.shape[0]):
        m = -np.inf
        for t0 in range(0, n, 128):
            mt = s2[h, t0:t0 + 128].max()
            if mt > m + 8.0:
                events += m != -np.inf
                m = mt
    assert events >= 50, events
    assert float(s.abs().max()) < 15.0


def _scores(w, b):
    """fp64 scaled scores [heads, n] of sequence b in the absorbed form."""
    cfg = w["cfg"]
    dl, D = cfg["d_latent"], cfg["d_latent"] + cfg["d_rope"]
    n = int(w["seq_lens"][b])
    tok = torch.arange(n)
    slot = w["block_table"][b].long()[tok // 64] * 64 + tok % 64
    rows = w["cache"].reshape(-1, D)[slot].double()
    q_lat = torch.einsum("hn,hln->hl", w["q_nope"][b].double(), w["w_uk"].double())
    s = cfg["softmax_scale"] * (q_lat @ rows[:, :dl].T + w["q_pe"][b].double() @ rows[:, dl:].T)
    return s, q_lat, rows


def _rescale_events(s):
    s2 = (s / np.log(2.0)).numpy()
    events = 0
    for h in range(s2.shape[0]):
        m = -np.inf
        for t0 in range(0, s2.shape[1], 128):
            mt = s2[h, t0:t0 + 128].max()
            if mt > m + 8.0:
                events += m != -np.inf
                m = mt
    return events


def test_exact_query_inputs_reach_large_logits_with_many_rescales():
    """Premise of the GPU large-logit test: the absorbed query is exact in
    bf16 (one-hot q_nope picks one column of W_LK_h), the logits reach 50 and
    more, and the 2^8 lazy-rescale threshold is crossed hundreds of times."""
    w = W.growing_scores_exact_query_decode()
    s, q_lat, _ = _scores(w, 0)
    assert torch.equal(q_lat.to(torch.bfloat16).double(), q_lat)
    assert float(s.max()) > 50.0
    assert _rescale_events(s) >= 200


def test_bf16_rounding_of_a_general_absorbed_query_moves_large_logit_outputs():
    """Why the large-logit GPU test uses an exact query: with an ordinary
    q_nope, rounding q_lat = q_nope . W_LK_h^T to bf16 (the decode call's input
    type) moves o_lat by more than the 5e-3 bf16 bar once logits approach 60,
    before any kernel arithmetic.  Absorbed-form fp64 attention with the
    exact and with the rounded query, same cache as the exact-query test."""
    w = W.growing_scores_exact_query_decode()
    g = torch.Generator().manual_seed(5)
    w["q_nope"] = torch.randn(w["q_nope"].shape, generator=g).to(torch.bfloat16)
    s, q_lat, rows = _scores(w, 0)
    cfg = w["cfg"]
    dl = cfg["d_latent"]
    qr = q_lat.to(torch.bfloat16).double()
    q_pe = w["q_pe"][0].double()
    s_r = cfg["softmax_scale"] * (qr @ rows[:, :dl].T + q_pe @ rows[:, dl:].T)
    o = torch.softmax(s, dim=1) @ rows[:, :dl]
    o_r = torch.softmax(s_r, dim=1) @ rows[:, :dl]
    assert float(s.max()) > 40.0
    assert float((o - o_r).abs().max() / o.abs().max()) > 5e-3


def test_crossing_ranges_inputs_put_sequence_ends_inside_most_ranges():
    """Premise of the GPU split-range test: with the context cut into equal
    ranges of 128-token tiles over 74 workers (two SMs each on a 148-SM
    B300), there are at least three tiles per worker and most workers' ranges
    hold parts of two or more sequences."""
    w = W.crossing_ranges_decode()
    lens = w["seq_lens"].tolist()
    pre = np.concatenate([[0], np.cumsum([(n + 127) // 128 for n in lens])])
    total, workers = int(pre[-1]), 74
    assert total >= 3 * workers
    crossing = 0
    for g in range(workers):
        lo, hi = g * total // workers, (g + 1) * total // workers
        first = np.searchsorted(pre, lo, side="right") - 1
        last = np.searchsorted(pre, hi - 1, side="right") - 1
        crossing += last > first
    assert crossing >= workers // 2
    assert 37 in lens and min(lens) >= 1


def test_multi_token_workload_adds_a_token_axis_to_the_queries():
    """Several new tokens per sequence: the shared-cache draws (same cache,
    block table and weights as cached_decode with the same seed), then
    per-token queries; deterministic in the seed."""
    w = W.multi_token_decode(3, [4, 70, 129], 4, seed=9)
    base = W.cached_decode(3, [4, 70, 129], seed=9, permute=True)
    for k in ("cache", "block_table", "w_uk", "w_uv", "seq_lens"):
        assert torch.equal(w[k], base[k])
    assert w["q_nope"].shape == (3, 4, 128, 128) and w["q_pe"].shape == (3, 4, 128, 64)
    assert w["kind"] == "multi" and w["q_tokens"] == 4
    again = W.multi_token_decode(3, [4, 70, 129], 4, seed=9)
    assert torch.equal(w["q_nope"], again["q_nope"]) and torch.equal(w["q_pe"], again["q_pe"])
    # distinct tokens get distinct queries
    assert not torch.equal(w["q_nope"][:, 0], w["q_nope"][:, 1])
    v = W.oracle_view(w)
    assert "q_tokens" not in v and v["q_nope"].shape == (3, 4, 128, 128)
    q4 = W.WORKLOADS["v2_b16_ctx4k_q4"]
    assert q4 is W.v2_b16_ctx4k_q4
