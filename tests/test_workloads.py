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
