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
