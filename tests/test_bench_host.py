"""Host-side arithmetic of bench.py: the algorithmic work the roofline divides
by, the peak it divides into, and when a stored DRAM-traffic figure is used."""
import hashlib
import json
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from head_latent_attention_23_b300 import workloads as W  # noqa: E402

GOLDEN = os.path.join(ROOT, "tests", "golden", "cache_bytes_pages.json")


def _cfg():
    return W.cached_decode(1, [1], seed=0)["cfg"]


def test_work_per_token_matches_the_pages_cache_row():
    """One cached token costs one cache row: 576 numbers of 2 bytes
    ("How DeepSeek Rewrote the Transformer (MLA)", section 08, 576 per token;
    16-bit entries), read once for all heads."""
    g = json.load(open(GOLDEN))
    w = {"cfg": _cfg(), "seq_lens": torch.tensor([1])}
    tokens, nbytes, flops = bench.work_per_step(w)
    assert tokens == 1
    assert nbytes == g["mla_numbers_per_token_per_layer"]["value"] * g["bytes_per_number"]["value"]
    # per head: a 576-long dot product for the score and a 512-long
    # multiply-add into the latent output, two flops per multiply-add
    heads, dl, dr = g["heads"]["value"], g["latent"]["value"], g["rope"]["value"]
    assert flops == heads * 2 * ((dl + dr) + dl) == 278_528


def test_work_of_several_new_tokens_reads_each_row_once():
    """Four new tokens per sequence: the cache bytes stay one row per cached
    token, the flops count token j of a sequence of n over n - 3 + j rows."""
    w = {"cfg": _cfg(), "seq_lens": torch.tensor([4, 10]), "q_tokens": 4}
    tokens, nbytes, flops = bench.work_per_step(w)
    assert tokens == 14
    assert nbytes == 14 * 576 * 2
    assert flops == (1 + 2 + 3 + 4 + 7 + 8 + 9 + 10) * 128 * 2 * (576 + 512)


def test_work_of_the_batch16_4k_call():
    w = {"cfg": _cfg(), "seq_lens": torch.tensor([4096] * 16)}
    tokens, nbytes, flops = bench.work_per_step(w)
    assert tokens == 65_536
    assert nbytes == 75_497_472           # 75.5 MB of cache per call
    assert flops == 18_253_611_008        # 18.25 GFLOP per call


def test_work_counts_only_real_tokens_of_ragged_batches():
    w = {"cfg": _cfg(), "seq_lens": torch.tensor([1, 63, 64, 65, 1000])}
    tokens, nbytes, _ = bench.work_per_step(w)
    assert tokens == 1193 and nbytes == 1193 * 1152


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["src"] == "fallback" and pk["hbm"] == 6400.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6504.1, "bf16_tflops": 1788.0, "bf16_tflops_sustained": 1387.0}))
    pk = bench.peaks()
    assert pk == {"hbm": 6504.1, "tc": 1788.0, "tc_sus": 1387.0, "src": "measured"}


def _write_profile(root, sha):
    csrc = root / "head_latent_attention_23_b300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "decode_tc.cu").write_bytes(b"// kernel source\n")
    (root / "profiles").mkdir()
    (root / "profiles" / "ncu_traffic.json").write_text(json.dumps(
        {"decode_tc:v2_b16_ctx4k": {"source": "decode_tc.cu", "source_sha": sha,
                       "dram_bytes_per_launch": 123}}))


def test_traffic_is_used_only_for_the_profiled_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_record("decode_tc", "v2_b16_ctx4k") is None    # no record at all
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()[:16]
    _write_profile(tmp_path, sha)
    assert bench.profile_record("decode_tc", "v2_b16_ctx4k")["dram_bytes_per_launch"] == 123
    assert bench.profile_record("decode_simt", "v2_b16_ctx4k") is None   # not that kernel
    assert bench.profile_record("decode_tc", "v2_b16_ctx4k_q4") is None  # not that workload
    (tmp_path / "head_latent_attention_23_b300" / "csrc" / "decode_tc.cu").write_bytes(
        b"// kernel source, changed\n")
    assert bench.profile_record("decode_tc", "v2_b16_ctx4k") is None    # kernel changed since


def test_committed_traffic_record_is_plausible():
    rec = bench.profile_record("decode_tc", "v2_b16_ctx4k")
    if rec is None:
        # the kernel changed since its capture: bench.py reports traffic null
        pytest.skip("profiles/ncu_traffic.json predates the current decode_tc.cu")
    # DRAM bytes per launch are at least the algorithmic cache bytes of the
    # profiled workload (batch 16 x 4096) and not far above them
    assert 75_497_472 <= rec["dram_bytes_per_launch"] <= 1.2 * 75_497_472


def test_cpu_sample_reports_parity_of_its_rows():
    """The CPU-baseline leg compares the oracle's rows of its last round with
    the same rows of the GPU's o_lat: zero error for the oracle's own full
    result, the relative error of a perturbed one."""
    import oracle as O
    w = W.cached_decode(2, [40, 7], seed=2, heads=4, d_latent=8, d_rope=4, d_nope=4, d_v=4)
    w["_name"] = "small"
    full = O.reference_cached_decode(W.oracle_view(w))["o_lat"]
    _, _, _, par = bench.cpu_sample(w, seconds_target=0.0, max_rounds=1, gpu_o_lat=full)
    assert par["max_rel_err"] == 0.0 and par["rows"] >= 1
    off = full.copy()
    off[0] *= 1.01
    _, _, _, par = bench.cpu_sample(w, seconds_target=0.0, max_rounds=1, gpu_o_lat=off)
    assert abs(par["max_rel_err"] - 0.01) < 1e-9
