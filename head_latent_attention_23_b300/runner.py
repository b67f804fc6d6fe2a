"""One decode step of an MLA layer, as a chain of libmla.so calls.

``DecodeStep`` uploads a workload (see ``workloads``) to the GPU once, owns the
output and scratch buffers, and ``run()`` issues the step's library calls on
one stream.  Nothing here computes: it only orders the calls.

Step for a workload whose cache rows are given (shared-cache decode):
    mla_absorb_q -> mla_decode (split-KV core + combine) -> mla_project_out
Step for several new query tokens per sequence over such a cache:
    mla_absorb_q (all tokens) -> mla_decode_multi -> mla_project_out
Step for a workload driven by hidden states x (full layer):
    mla_query_proj -> mla_append_latent -> mla_absorb_q -> mla_decode
    -> mla_project_out (with W_O)

``run_fused()`` issues the same step as one library call
(mla_cached_decode_step, or mla_layer_decode_step when each sequence gets one
new token), optionally with the per-step inputs and the result in pinned host
memory.
"""
import torch

from . import mla


class DecodeStep:
    def __init__(self, w, device="cuda"):
        self.w = w
        self.cfg_dict = w["cfg"]
        self.cfg = mla.config_from(self.cfg_dict)
        self.kind = w["kind"]
        dev = torch.device(device)
        self.device = dev
        c = self.cfg_dict
        B, H = w["batch"], c["heads"]
        dt = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32

        def up(name):
            t = w.get(name)
            return None if t is None else t.to(dev).contiguous()

        self.cache = up("cache")
        self.block_table = up("block_table")
        self.seq_lens = up("seq_lens")
        self.w_uk = up("w_uk")
        self.w_uv = up("w_uv")
        self.B = B
        self.T = w.get("q_tokens", 1)
        rows = B * self.T             # query rows: one per (sequence, new token)
        if self.kind in ("cached", "multi"):
            self.q_nope = up("q_nope")
            self.q_pe = up("q_pe")
        else:
            self.x_new = up("x_new")
            self.seq_idx_new = up("seq_idx_new")
            self.pos_new = up("pos_new")
            self.x_q = up("x_q")
            self.pos_q = up("pos_q")
            self.w_dkv = up("w_dkv")
            self.w_dq = up("w_dq")
            self.w_uq = up("w_uq")
            self.w_o = up("w_o")
            self.q_nope = torch.empty((B, H, c["d_nope"]), dtype=dt, device=dev)
            self.q_pe = torch.empty((B, H, c["d_rope"]), dtype=dt, device=dev)
            d_lq = w["d_lq"] or 0
            self.q_scratch = torch.empty(mla.query_proj_workspace_size(self.cfg, B, d_lq),
                                         dtype=torch.uint8, device=dev)
            self.out = torch.empty((B, w["d_model"]), dtype=dt, device=dev)
        self.q_lat = torch.empty((rows, H, c["d_latent"]), dtype=dt, device=dev)
        self.o_lat = torch.empty((rows, H, c["d_latent"]), dtype=dt, device=dev)
        self.lse = torch.empty((rows, H), dtype=torch.float32, device=dev)
        self.o_v = torch.empty((rows, H, c["d_v"]), dtype=dt, device=dev)
        maxb = self.block_table.shape[1]
        if self.kind == "multi":
            self.workspace = torch.empty(
                mla.decode_multi_workspace_size(self.cfg, B, self.T, maxb), dtype=torch.uint8,
                device=dev)
        else:
            self.workspace = mla.decode_workspace(self.cfg, B, dev)
        # one library call per step: the shared-cache step, or the full layer
        # step when each sequence gets exactly one new token (its newest)
        self.fused = self.kind == "cached" or (
            self.kind == "token" and w["x_new"].shape[0] == B and
            torch.equal(w["x_new"], w["x_q"]) and torch.equal(w["seq_idx_new"], torch.arange(B, dtype=torch.int32)) and
            torch.equal(w["pos_new"], w["seq_lens"] - 1))
        if self.kind == "cached":
            n = mla.cached_decode_step_workspace_size(self.cfg, B, maxb)
        elif self.fused:
            self.weights = mla.layer_weights(self.cfg, self.w_dkv, self.w_uq, self.w_uk,
                                             self.w_uv, self.w_o, w_dq=self.w_dq)
            n = mla.layer_decode_step_workspace_size(self.cfg, self.weights, B, maxb)
        else:
            n = 0
        self.step_ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)

    # the graded core: split-KV attention + combine
    def decode(self, stream=None):
        if self.kind == "multi":
            B, T, H = self.B, self.T, self.cfg_dict["heads"]
            mla.decode_multi(self.cfg, self.q_lat.view(B, T, H, -1), self.q_pe, self.cache,
                             self.block_table, self.seq_lens, self.o_lat.view(B, T, H, -1),
                             self.lse.view(B, T, H), self.workspace, stream)
        else:
            mla.decode(self.cfg, self.q_lat, self.q_pe, self.cache, self.block_table,
                       self.seq_lens, self.o_lat, self.lse, self.workspace, stream)

    def pre(self, stream=None):
        """The step's calls before mla_decode."""
        if self.kind == "token":
            mla.query_proj(self.cfg, self.x_q, self.w_uq, self.pos_q, self.q_nope, self.q_pe,
                           w_dq=self.w_dq, scratch=self.q_scratch, stream=stream)
            mla.append_latent(self.cfg, self.x_new, self.w_dkv, self.seq_idx_new, self.pos_new,
                              self.block_table, self.cache, stream=stream)
        q_nope = self.q_nope.reshape(self.q_lat.shape[0], self.q_lat.shape[1], -1)
        mla.absorb_q(self.cfg, q_nope, self.w_uk, self.q_lat, stream)

    def post(self, stream=None):
        """The step's calls after mla_decode."""
        if self.kind == "token":
            mla.project_out(self.cfg, self.o_lat, self.w_uv, self.o_v, self.w_o, self.out,
                            stream)
        else:
            mla.project_out(self.cfg, self.o_lat, self.w_uv, self.o_v, stream=stream)

    def run(self, stream=None):
        self.pre(stream)
        self.decode(stream)
        self.post(stream)

    def run_fused(self, io_flags=0, inputs=None, result=None, stream=None):
        """The step as one library call.  With io_flags, `inputs` (dict of
        pinned host tensors: q_nope, q_pe or x; seq_lens; block_table) and
        `result` (pinned host tensor for o_v or out) replace the device ones."""
        if not self.fused:
            raise ValueError("this workload appends several rows per sequence; use run()")
        t = dict(q_nope=self.q_nope, q_pe=self.q_pe, seq_lens=self.seq_lens,
                 block_table=self.block_table)
        if self.kind == "token":
            t["x"] = self.x_q
        if inputs:
            t.update(inputs)
        if self.kind == "cached":
            mla.cached_decode_step(self.cfg, t["q_nope"], t["q_pe"], self.w_uk, self.w_uv,
                                   t["seq_lens"], self.cache, t["block_table"],
                                   self.o_v if result is None else result, o_lat=self.o_lat,
                                   lse=self.lse, io_flags=io_flags, workspace=self.step_ws,
                                   stream=stream)
        else:
            mla.layer_decode_step(self.cfg, self.weights, t["x"], t["seq_lens"], self.cache,
                                  t["block_table"], self.out if result is None else result,
                                  io_flags=io_flags, workspace=self.step_ws, stream=stream)

    def kernels_per_step(self, fused=False):
        """Kernel launches one run() (or, with fused, one run_fused()) issues.
        The fused full-layer step adds the positions kernel and a split-K
        reduction after each batch-1 projection that splits K."""
        n = 1 + 2 + 1                       # absorb, decode core + combine, o_v
        if self.kind == "multi":
            n += 1                          # per-token rows of the split plan
        if self.kind == "token":
            n += 2 if self.w_dq is not None else 1   # query GEMM(s)
            n += 1                          # split/rotate kernel, or (bf16) the rotation table
                                            # for the split fused into W_UQ's epilogue
            n += 1                          # append
            n += 1                          # W_O
            if fused:
                n += 1 + self.split_reductions()
        return n

    def split_reductions(self):
        """Batch-1 projections of the fused full-layer step that the library
        splits along K (each adds one reduction kernel), by the library's rule:
        the fewest K ranges that keep 85% of the SMs' work slots busy."""
        import math
        sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        c, B = self.cfg_dict, self.B
        d_model = self.out.shape[1]
        prods = [(c["heads"] * (c["d_nope"] + c["d_rope"]), self.w_uq.shape[0]),
                 (c["d_latent"] + c["d_rope"], d_model), (d_model, c["heads"] * c["d_v"])]
        if self.w_dq is not None:
            prods.append((self.w_dq.shape[1], d_model))
        n = 0
        for N, K in prods:
            tiles = math.ceil(N / 128) * math.ceil(B / 128)
            nk = math.ceil(K / 64)
            best = 1
            for s in range(1, min(nk // 4, 32) + 1):
                waves = tiles * s / sms
                best = s
                if waves / math.ceil(waves) >= 0.85:
                    break
            n += best > 1
        return n

    def results(self):
        r = dict(o_lat=self.o_lat, lse=self.lse, o_v=self.o_v, q_lat=self.q_lat)
        if self.kind == "multi":
            r = {k: v.view(self.B, self.T, *v.shape[1:]) for k, v in r.items()}
        if self.kind == "token":
            r["out"] = self.out
            r["q_nope"] = self.q_nope
            r["q_pe"] = self.q_pe
        return r
