"""mla_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a framework that owns all device memory through its own pool, a
plugin interface that hands over only inputs and outputs, a loop where an
allocation's implicit synchronisation is not allowed) cannot provide
mla_decode's workspace.  The no-allocation entry point keeps the split-KV
partials in a static device array inside the library instead.  These tests
call it through the C ABI and compare it with mla_decode on the same inputs,
for two calls in a row (the second must not see the first one's leftovers),
and check that requests too large for the array are refused.
"""
import numpy as np
import pytest
import torch

from head_latent_attention_23_b300 import mla, workloads as W

pytestmark = pytest.mark.gpu

TOL = 5e-3     # bf16 inputs, fp32 accumulation: the bar the other parity tests use


def _rel(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def _inputs(lens, seed):
    w = W.cached_decode(len(lens), lens, seed=seed, permute=True)
    cfg = mla.config_from(w["cfg"])
    B = len(lens)
    g = torch.Generator().manual_seed(seed + 1)
    q_lat = (0.5 * torch.randn(B, 128, 512, generator=g)).to(torch.bfloat16).cuda()
    return cfg, dict(q_lat=q_lat, q_pe=w["q_pe"].cuda(), cache=w["cache"].cuda(),
                     block_table=w["block_table"].cuda(), seq_lens=w["seq_lens"].cuda())


def _both(cfg, t):
    B = t["q_lat"].shape[0]
    ref_o = torch.empty(B, 128, 512, dtype=torch.bfloat16, device="cuda")
    ref_l = torch.empty(B, 128, dtype=torch.float32, device="cuda")
    mla.decode(cfg, t["q_lat"], t["q_pe"], t["cache"], t["block_table"], t["seq_lens"], ref_o,
               ref_l)
    o = torch.full_like(ref_o, float("nan"))
    l = torch.full_like(ref_l, float("nan"))
    mla.decode_noalloc(cfg, t["q_lat"], t["q_pe"], t["cache"], t["block_table"], t["seq_lens"],
                       o, l)
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK
    return (o, l), (ref_o, ref_l)


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    cfg, t1 = _inputs([1, 63, 64, 65, 700], seed=21)
    (o1, l1), (r1, rl1) = _both(cfg, t1)
    assert _rel(o1, r1) <= TOL and _rel(l1, rl1) <= TOL
    cfg, t2 = _inputs([4096, 10, 300], seed=22)
    (o2, l2), (r2, rl2) = _both(cfg, t2)
    assert _rel(o2, r2) <= TOL and _rel(l2, rl2) <= TOL


def test_noalloc_with_fewer_split_ranges_than_decode_matches_decode():
    """At batch 100 the partials of mla_decode's full split (one per worker
    plus one per sequence) do not fit the array, so the no-allocation call
    cuts the context into fewer ranges: same result up to rounding."""
    g = torch.Generator().manual_seed(24)
    lens = torch.randint(1, 601, (100,), generator=g).tolist()
    cfg, t = _inputs(lens, seed=24)
    (o, l), (r, rl) = _both(cfg, t)
    assert _rel(o, r) <= TOL and _rel(l, rl) <= TOL


def test_noalloc_batch_limit_is_126_at_deepseek_shapes():
    """(1 + batch) slots of 128 heads x (512 + 1) fp32 plus 16 bytes per
    sequence fit the 32 MiB array up to batch 126: that batch runs (one split
    range) and matches mla_decode, batch 127 is refused."""
    g = torch.Generator().manual_seed(25)
    lens = torch.randint(1, 200, (126,), generator=g).tolist()
    cfg, t = _inputs(lens, seed=25)
    (o, l), (r, rl) = _both(cfg, t)
    assert _rel(o, r) <= TOL and _rel(l, rl) <= TOL
    B = 127
    q_lat = torch.zeros(B, 128, 512, dtype=torch.bfloat16, device="cuda")
    q_pe = torch.zeros(B, 128, 64, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_noalloc(cfg, q_lat, q_pe, t["cache"], bt, sl, torch.zeros_like(q_lat))
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED


def test_noalloc_refuses_batches_beyond_its_array():
    cfg, t = _inputs([5], seed=23)
    # (1 + batch) partial slots of 128 heads x 512 fp32 no longer fit 32 MiB
    B = 128
    q_lat = torch.zeros(B, 128, 512, dtype=torch.bfloat16, device="cuda")
    q_pe = torch.zeros(B, 128, 64, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    o = torch.zeros_like(q_lat)
    with pytest.raises(mla.MLAError) as e:
        mla.decode_noalloc(cfg, q_lat, q_pe, t["cache"], bt, sl, o)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED
