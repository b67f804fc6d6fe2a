#!/usr/bin/env python3
"""Benchmark of one MLA decode step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one pass of the hot path over one batch: query absorption
(mla_absorb_q), split-KV absorbed attention + combine (mla_decode) and the
value up-projection (mla_project_out); for the full-layer workload also the
query projection and the cache append, and W_O.  Inputs are synthetic and
seeded (workloads.py).  Prints one JSON line (rank 0).

ours:       device-resident inputs; R replicas of every input tensor are
            rotated so consecutive steps never find their cache, queries or
            weights in L2 (R * bytes > 2 * L2).  Each step is the one library
            call a user makes (mla_cached_decode_step or
            mla_layer_decode_step; separate calls where a step has no
            single-call form), captured once into CUDA graphs and replayed;
            CUDA events on the launching stream time the replays; the
            mla_decode durations come from events around each call in a
            replay of the steps as separate calls; max over ranks.  e2e: the
            same call per step with pinned HOST inputs and output, the copies
            inside the call and inside the timed region, steps alternating
            over two streams (the one-stream figure is reported beside it).
reference:  the fp64 CPU oracle (unmerged MLA) on a bounded sample of the
            same workload, on the host cores.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from head_latent_attention_23_b300 import workloads as W  # noqa: E402

METRIC = "MLA decode tokens/s; latent-cache HBM GB/s & TFLOP/s as % of roofline"
UNIT = "tokens/s"
L2_BYTES = 126 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="v2_b16_ctx4k", choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_rate(local_ms, local_units, device="cpu"):
    """Whole-job rate of a weak-scaling run: the units every rank processed,
    summed, over the slowest rank's time (ms).  Returns (units per second,
    slowest ms).  With one process (or no process group) it is the local rate.
    `device` is where the reduction's tensors live: the rank's GPU under NCCL,
    the CPU under gloo."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
        u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
        local_ms, local_units = float(t.item()), float(u.item())
    return local_units / (local_ms / 1e3), local_ms


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], tc=d["bf16_tflops"], tc_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6400.0, tc=1800.0, tc_sus=1400.0, src="fallback")


def work_per_step(w):
    """Algorithmic cache bytes and flops of one decode call.

    Per (query, cached token): each head does a (d_latent + d_rope) dot
    product for the score and a d_latent axpy for the latent-space value sum.
    Each cached row (d_latent + d_rope elements) is read from HBM once per
    step, however many of the sequence's new tokens attend to it.  With T new
    tokens per sequence, token j of a sequence of n sees n - T + 1 + j rows.
    Returns (cached tokens, bytes, flops).
    """
    c = w["cfg"]
    esz = 2 if c["dtype"] == "bf16" else 4
    T = w.get("q_tokens", 1)
    lens = w["seq_lens"].long()
    rows_seen = int((lens * T - T * (T - 1) // 2).sum())
    D = c["d_latent"] + c["d_rope"]
    bytes_ = int(lens.sum()) * D * esz
    flops = rows_seen * c["heads"] * (2 * D + 2 * c["d_latent"])
    return int(lens.sum()), bytes_, flops


def profile_record(kernel_tag, workload):
    """Per-launch DRAM traffic of the decode kernel on this workload from the
    committed ncu summary, if it was taken on the current kernel source; else
    None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel_tag}:{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "head_latent_attention_23_b300", "csrc", rec["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec if h == rec["source_sha"] else None


class ClockSampler:
    """Samples SM clock and throttle reasons while the timed region runs:
    NVML when the Python binding is present, else `nvidia-smi -lms`."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.proc = None
        self._stop = threading.Event()
        self.t = None

    def _nvml_loop(self, nv, h):
        bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                "sw_power_cap": 0x4}
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksThrottleReasons(h)
                for k, b in bits.items():
                    if r & b:
                        self.reasons.add(k)
            except Exception:
                pass
            time.sleep(0.02)

    def __enter__(self):
        try:
            import pynvml as nv
            nv.nvmlInit()
            h = nv.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM)
            self.t = threading.Thread(target=self._nvml_loop, args=(nv, h), daemon=True)
            self.t.start()
            return self
        except Exception:
            pass
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.t is not None:
            self._stop.set()
            self.t.join()
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for k, v in zip(self.NAMES, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(k)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ---------------------------------------------------------------- oracle arm

def cpu_sample(w, seconds_target=12.0, max_rounds=64, gpu_o_lat=None):
    """Times the oracle (as it stands) on whole sequences' worth of heads.

    One 'round' decodes `threads` (sequence, head) pairs, one per oracle
    thread, over sequence 0's full context; rounds repeat until about
    `seconds_target` of wall time.  Returns (tokens/s, threads, description,
    parity), parity comparing the last round's o_lat rows with the same rows
    of `gpu_o_lat` (the GPU's o_lat for this workload, indexed like the
    oracle's pairs) when it is given.
    """
    import oracle as O
    v = W.oracle_view(w)
    H = w["cfg"]["heads"]
    threads = O.num_threads()
    done_heads = 0
    t0 = time.perf_counter()
    rounds = 0
    T = w.get("q_tokens", 1)
    while True:
        pairs = [(0, (done_heads + k) % H) for k in range(min(threads, H))]
        ref, keys = _oracle_pairs(O, v, w, pairs, done_heads // H, T)
        done_heads += len(pairs)
        rounds += 1
        el = time.perf_counter() - t0
        if el >= seconds_target or rounds >= max_rounds:
            break
    tokens = done_heads / H          # one decode token = all heads of one query token
    n0 = int(w["seq_lens"][0])
    desc = (f"{done_heads} (query token, head) pairs of sequence 0 (context {n0}) of "
            f"{w_name(w)}; {tokens:.3f} decode tokens in {el:.2f} s")
    parity = None
    if gpu_o_lat is not None:
        r = np.stack([ref[k] for k in keys]).astype(np.float64)
        g = np.stack([gpu_o_lat[k] for k in keys]).astype(np.float64)
        parity = {"max_rel_err": float(np.abs(g - r).max() / max(np.abs(r).max(), 1e-30)),
                  "rows": len(keys), "tolerance": 5e-3 if w["cfg"]["dtype"] == "bf16" else 1e-5,
                  "what": "o_lat rows of the timed workload's last oracle round against the GPU"}
    return tokens / el, threads, desc, parity


def _oracle_pairs(O, v, w, pairs, round_idx, T):
    """The oracle on (sequence 0, head) pairs; with several new tokens per
    sequence, on query token round_idx % T of sequence 0.  Returns a map from
    each pair's index into the full o_lat to the oracle's row, and the keys."""
    if w["kind"] == "cached":
        o = O.reference_cached_decode(v, pairs=pairs)["o_lat"]
        keys = [(0, h) for _, h in pairs]
        return {k: o[k] for k in keys}, keys
    if w["kind"] == "multi":
        j = round_idx % T
        o = O.reference_multi_decode(v, pairs=[(0, j, h) for _, h in pairs])["o_lat"]
        keys = [(0, j, h) for _, h in pairs]
        return {k: o[k] for k in keys}, keys
    o = O.reference_token_decode(v, seqs=[0], pairs=[(0, h) for _, h in pairs])["o_lat"]
    keys = [(0, h) for _, h in pairs]
    return {k: o[k] for k in keys}, keys


def w_name(w):
    return w.get("_name", "workload")


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle as O
    w = W.WORKLOADS[args.workload](args.seed)
    w["_name"] = args.workload
    v = W.oracle_view(w)
    H = w["cfg"]["heads"]
    threads = O.num_threads()
    K = args.steps if args.steps else 5
    T = w.get("q_tokens", 1)
    per = min(threads, H)     # distinct heads per step

    def step(i):
        pairs = [(0, (i * per + k) % H) for k in range(per)]
        _oracle_pairs(O, v, w, pairs, i * per // H, T)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(K):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    tokens = K * per / H
    val = tokens / el
    cfg = config_block(w, args.workload, 1, "n/a (host)")
    out = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": el / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the pages' DeepSeek-V2 figures)", "config": cfg,
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"each step: {per} (sequence 0, head) pairs "
                                   f"= {per}/{H} of one decode token"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def config_block(w, name, replicas, l2):
    c = w["cfg"]
    lens = w["seq_lens"]
    return {"workload": name, "batch": int(w["batch"]), "q_tokens": int(w.get("q_tokens", 1)),
            "heads": c["heads"],
            "d_latent": c["d_latent"], "d_rope": c["d_rope"], "d_nope": c["d_nope"],
            "d_v": c["d_v"], "block_size": c["block_size"],
            "context_min": int(lens.min()), "context_max": int(lens.max()),
            "context_total": int(lens.sum()), "parallelism": "replicas",
            "l2": l2, "input_replicas": replicas}


# ---------------------------------------------------------------- our arm

def run_ours(args):
    from head_latent_attention_23_b300 import mla
    from head_latent_attention_23_b300.runner import DecodeStep

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload](args.seed + rank)
    w["_name"] = args.workload
    tokens, cbytes, cflops = work_per_step(w)
    step_bytes = sum(t.numel() * t.element_size() for t in w.values()
                     if isinstance(t, torch.Tensor))
    R = max(1, math.ceil(2 * L2_BYTES / max(step_bytes, 1)) + 1)
    R = min(R, 8)
    steps = [DecodeStep(w, dev) for _ in range(R)]
    stream = torch.cuda.current_stream(dev)
    B = w["batch"]
    units = B * w.get("q_tokens", 1)   # query tokens decoded per step

    for i in range(max(args.warmup, 3)):
        steps[i % R].run()
    torch.cuda.synchronize()
    assert mla.get_status() == mla.MLA_OK, "device status after warm-up"

    K = args.steps
    if K is None:
        # about 1.5 s of timed steps, from one replay of a 50-step graph
        probe = capture([steps[i % R] for i in range(50)], None)
        probe.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        probe.replay()
        b.record(stream)
        torch.cuda.synchronize()
        per = a.elapsed_time(b) / 50 / 1e3
        K = int(min(max(1.5 / per, 200), 50000))
        del probe

    # The timed region replays CUDA graphs of whole steps (the library's
    # kernels, captured once), so the host's per-call overhead does not leave
    # the GPU idle between steps.  Graph A holds G consecutive steps (replicas
    # rotated), each mla_decode call bracketed by timing events; graph B holds
    # the remaining K mod G steps.
    G = min(K, 500)
    ga_steps = [steps[i % R] for i in range(G)]
    rem = K - (K // G) * G
    dec_ev = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(G)]
    # A step is timed as the one library call a user makes
    # (mla_cached_decode_step, or mla_layer_decode_step, whose batch-1
    # projections split K over all SMs), its kernels chained by programmatic
    # dependent launch; the mla_decode durations come from a replay of the
    # same steps issued as separate calls with events around mla_decode,
    # right after the timed region (an event between two kernels ends their
    # overlap, so the events stay out of the timed replays).  Steps with no
    # single-call form are timed as separate calls with the events inside.
    fused_timing = steps[0].fused
    if fused_timing:
        graph_a = capture(ga_steps, None, fused=True)
        graph_b = capture([steps[i % R] for i in range(rem)], None, fused=True) if rem else None
        graph_d = capture(ga_steps[:min(G, 100)], dec_ev[:min(G, 100)])
        dec_ev = dec_ev[:min(G, 100)]
    else:
        graph_a = capture(ga_steps, dec_ev)
        graph_b = capture([steps[i % R] for i in range(rem)], None) if rem else None
        graph_d = None
    for _ in range(2):           # graph warm-up (first replays upload the graph)
        graph_a.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(K // G):
            graph_a.replay()
        if graph_b is not None:
            graph_b.replay()
        end.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    # tokens of all ranks over the slowest rank's time
    value, total_ms = job_rate(start.elapsed_time(end), units * K, dev)
    if graph_d is not None:
        graph_d.replay()
        graph_d.replay()
        torch.cuda.synchronize()
    # the last replay of graph A (or D): one duration per mla_decode call
    dec_ms = [a.elapsed_time(b) for a, b in dec_ev]
    assert mla.get_status() == mla.MLA_OK, "device status after timed region"

    # end to end: pinned host inputs -> device, step, result -> host
    if ws > 1:
        dist.barrier()
    if steps[0].fused:
        e2e = run_e2e(steps[:2], w, dev)
    elif steps[0].kind == "multi":
        e2e = run_e2e_calls(steps[:2], units, dev)
    else:
        e2e = {"value": None, "unit": UNIT, "note": "workload appends several rows per sequence"}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    pk = peaks()
    ms_step = total_ms / K
    dec_mean_ms = statistics.mean(dec_ms)
    dec_med_ms = statistics.median(dec_ms)
    hbm_gbs = cbytes / (dec_mean_ms * 1e-3) / 1e9
    tflops = cflops / (dec_mean_ms * 1e-3) / 1e12
    t_roof = max(cbytes / (pk["hbm"] * 1e9), cflops / (pk["tc"] * 1e12))
    bound = "hbm" if cbytes / (pk["hbm"] * 1e9) >= cflops / (pk["tc"] * 1e12) else "tensor"
    path = mla.decode_path(steps[0].cfg)
    rec = profile_record("decode_tc" if path == 1 else "decode_simt", args.workload)
    roof = {
        "bound": bound,
        "achieved": hbm_gbs if bound == "hbm" else tflops,
        "peak": pk["hbm"] if bound == "hbm" else pk["tc"],
        "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
        "frac": (hbm_gbs / pk["hbm"]) if bound == "hbm" else (tflops / pk["tc"]),
        "traffic": rec["dram_bytes_per_launch"] if rec else None,
        "kernel": ("mla_decode_multi (row expansion, split-KV core + combine)"
                   if steps[0].kind == "multi" else
                   "mla_decode (split-KV core + combine)") + ", one call per step",
        "algorithmic_bytes_per_launch": cbytes,
        "algorithmic_flops_per_launch": cflops,
        "tensor_tflops": tflops,
        "tensor_frac_burst": tflops / pk["tc"],
        "tensor_frac_sustained": tflops / pk["tc_sus"],
        "roofline_frac": t_roof / (dec_mean_ms * 1e-3),
        "decode_ms_mean": dec_mean_ms, "decode_ms_median": dec_med_ms,
        "peak_source": pk["src"] + " (MEASURED_PEAKS.json burst figures)",
        "decode_path": "tcgen05" if path == 1 else "cuda-core fp32",
    }
    try:
        s0 = steps[0]
        o_host = s0.o_lat.float().cpu().numpy()
        if s0.kind == "multi":
            o_host = o_host.reshape(s0.B, s0.T, *o_host.shape[1:])
        cpu_val, cores, desc, parity = cpu_sample(w, gpu_o_lat=o_host)
        cpu = {"value": cpu_val, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc, "parity": parity}
    except Exception as e:  # the oracle is a baseline only; report why it is missing
        cpu = {"value": None, "unit": UNIT, "cores": None, "kind": "oracle",
               "sample": f"unavailable: {e}"}
    dt = w["cfg"]["dtype"]
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt,
        "data": "synthetic (seeded; shapes of the pages' DeepSeek-V2 figures)",
        "config": config_block(w, args.workload, R,
                               f"inputs rotated over {R} replicas "
                               f"({R * step_bytes / 2**20:.0f} MiB > 2 x L2)"),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * steps[0].kernels_per_step(fused=fused_timing),
        "timing": (f"CUDA graphs of {G} steps replayed {K // G} times"
                   + (f" + one of {rem} steps" if rem else "")
                   + (f"; each step one {'mla_cached_decode_step' if steps[0].kind == 'cached' else 'mla_layer_decode_step'}"
                      " call; mla_decode durations from events in a replay of the step as "
                      "separate calls" if fused_timing else
                      "; mla_decode durations from events inside the last replay")),
        "clocks": clk.summary(),
    }
    print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def capture(step_list, ev_pairs, fused=False):
    """A CUDA graph of the given steps' library calls, in order; with
    ev_pairs, timing events around each mla_decode call; with fused, each step
    as its one whole-step library call."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        # capture-time allocations: none (every buffer is owned by a step)
        with torch.cuda.graph(g, stream=side):
            cs = torch.cuda.current_stream()
            for j, s in enumerate(step_list):
                if fused:
                    s.run_fused()
                else:
                    _run_with_decode_events(s, ev_pairs[j] if ev_pairs else None, cs)
    torch.cuda.current_stream().wait_stream(side)
    return g


def _run_with_decode_events(s, evpair, stream):
    """One step, with CUDA events around its mla_decode call when evpair is
    given."""
    s.pre()
    if evpair:
        evpair[0].record(stream)
    s.decode()
    if evpair:
        evpair[1].record(stream)
    s.post()


def run_e2e(reps, w, dev, min_steps=500, min_seconds=1.0):
    """The step end to end through one public library call per step
    (mla_cached_decode_step or mla_layer_decode_step) with HOST buffers: the
    call copies the step's inputs from pinned host memory, runs the kernels
    and copies the result back, all inside the timed region.  At least
    `min_steps` steps and about `min_seconds`, whatever --steps says.

    Measured twice: one stream (each step's copies wait for the previous
    step), and two streams with one replica each, alternating, so one step's
    copies overlap the other's kernels, as a server pipelines its batches.
    Every step still copies its own inputs in and its own result out."""
    s0 = reps[0]
    if s0.kind == "cached":
        names = ["q_nope", "q_pe", "seq_lens", "block_table"]
    else:
        names = ["x", "seq_lens", "block_table"]

    def host_bufs(s):
        dev_t = dict(q_nope=s.q_nope, q_pe=s.q_pe, seq_lens=s.seq_lens,
                     block_table=s.block_table)
        if s.kind != "cached":
            dev_t["x"] = s.x_q
        result = s.o_v if s.kind == "cached" else s.out
        return ({n: dev_t[n].cpu().pin_memory() for n in names},
                torch.empty(result.shape, dtype=result.dtype).pin_memory())

    bufs = [host_bufs(s) for s in reps]
    h2d = sum(h.numel() * h.element_size() for h in bufs[0][0].values())
    d2h = bufs[0][1].numel() * bufs[0][1].element_size()
    flags = 3   # MLA_IO_HOST_INPUTS | MLA_IO_HOST_OUTPUT
    cur = torch.cuda.current_stream(dev)

    def timed(nrep, K):
        streams = [torch.cuda.Stream(dev) for _ in range(nrep)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for st in streams:
            st.wait_event(a)
        for i in range(K):
            r = i % nrep
            reps[r].run_fused(io_flags=flags, inputs=bufs[r][0], result=bufs[r][1],
                              stream=streams[r])
        for st in streams:
            cur.wait_stream(st)
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    out = {}
    for nrep in sorted({1, len(reps)}):
        timed(nrep, 5)
        per = timed(nrep, 50) / 50 / 1e3
        K = int(max(min_steps, min(min_seconds / max(per, 1e-7), 200000)))
        value, total = job_rate(timed(nrep, K), w["batch"] * K, dev)
        out[nrep] = {"value": value, "ms_per_step": total / K, "steps": K}
    best = out[max(out)]
    res = {"value": best["value"], "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": best["ms_per_step"],
           "steps": best["steps"], "streams": max(out),
           "call": "mla_cached_decode_step" if s0.kind == "cached" else "mla_layer_decode_step",
           "note": ("one library call per step with pinned host inputs and output; steps "
                    f"alternate over {max(out)} streams (one replica each) so one step's copies "
                    "overlap another's kernels; same input set every step")}
    if max(out) > 1:
        res["one_stream"] = {"value": out[1]["value"], "ms_per_step": out[1]["ms_per_step"],
                             "steps": out[1]["steps"]}
    return res


def run_e2e_calls(reps, units, dev, min_steps=500, min_seconds=1.0):
    """End to end for a step that has no single-call form (several new query
    tokens per sequence): each step copies its inputs (queries, lengths, block
    table) from pinned host memory to the device, issues the step's library
    calls and copies o_v back to pinned host memory, on one stream, inside
    the timed region.  As in run_e2e, measured on one stream and with the
    steps alternating over two streams (one replica each)."""
    names = ["q_nope", "q_pe", "seq_lens", "block_table"]
    bufs = []
    for s in reps:
        dev_t = {n: getattr(s, n) for n in names}
        bufs.append((dev_t, {n: t.cpu().pin_memory() for n, t in dev_t.items()},
                     torch.empty(s.o_v.shape, dtype=s.o_v.dtype).pin_memory()))
    h2d = sum(h.numel() * h.element_size() for h in bufs[0][1].values())
    d2h = bufs[0][2].numel() * bufs[0][2].element_size()
    cur = torch.cuda.current_stream(dev)

    def timed(nrep, K):
        streams = [torch.cuda.Stream(dev) for _ in range(nrep)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for st in streams:
            st.wait_event(a)
        for i in range(K):
            r = i % nrep
            dev_t, host_in, host_out = bufs[r]
            with torch.cuda.stream(streams[r]):
                for n in names:
                    dev_t[n].copy_(host_in[n], non_blocking=True)
                reps[r].run(streams[r])
                host_out.copy_(reps[r].o_v, non_blocking=True)
        for st in streams:
            cur.wait_stream(st)
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    out = {}
    for nrep in sorted({1, len(reps)}):
        timed(nrep, 5)
        per = timed(nrep, 50) / 50 / 1e3
        K = int(max(min_steps, min(min_seconds / max(per, 1e-7), 200000)))
        value, total = job_rate(timed(nrep, K), units * K, dev)
        out[nrep] = {"value": value, "ms_per_step": total / K, "steps": K}
    best = out[max(out)]
    res = {"value": best["value"], "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": best["ms_per_step"],
           "steps": best["steps"], "streams": max(out),
           "call": "mla_absorb_q + mla_decode_multi + mla_project_out",
           "note": ("pinned host inputs copied in and o_v copied out on the step's stream "
                    f"every step; steps alternate over {max(out)} streams (one replica each); "
                    "same input set every step")}
    if max(out) > 1:
        res["one_stream"] = {"value": out[1]["value"], "ms_per_step": out[1]["ms_per_step"],
                             "steps": out[1]["steps"]}
    return res


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
