"""Python binding of libmla.so (argument marshalling only).

Every function here forwards to the C entry point of the same name in
``include/mla.h``: it checks that the torch tensors are CUDA, contiguous and
of the expected dtype, passes their device pointers and sizes, and raises
``MLAError`` on a non-zero status.  All arithmetic runs in the library's CUDA
kernels.  There is no fallback: if the library is missing the first call
raises.
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_TIMEOUT = 5
MLA_ERR_INDEX = 6
DTYPE_BF16 = 0
DTYPE_F32 = 1

# Every entry point declared in include/mla.h.
EXPORTS = (
    "mla_status_string", "mla_version", "mla_decode_path", "mla_get_status",
    "mla_append_latent", "mla_absorb_q", "mla_decode_workspace_size", "mla_decode",
    "mla_decode_combine", "mla_project_out", "mla_query_proj_workspace_size", "mla_query_proj",
    "mla_decode_noalloc", "mla_set_wait_limit_ns", "mla_layer_decode_step_workspace_size",
    "mla_layer_decode_step", "mla_cached_decode_step_workspace_size", "mla_cached_decode_step",
    "mla_decode_multi_workspace_size", "mla_decode_multi",
)

IO_HOST_INPUTS = 1
IO_HOST_OUTPUT = 2


class MLAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class LayerWeights(ctypes.Structure):
    """mirror of struct mla_layer_weights (device pointers)"""
    _fields_ = [("d_model", ctypes.c_int), ("d_lq", ctypes.c_int), ("w_dkv", ctypes.c_void_p),
                ("w_dq", ctypes.c_void_p), ("w_uq", ctypes.c_void_p), ("w_uk", ctypes.c_void_p),
                ("w_uv", ctypes.c_void_p), ("w_o", ctypes.c_void_p)]


class Config(ctypes.Structure):
    """mirror of struct mla_config"""
    _fields_ = [("heads", ctypes.c_int), ("d_latent", ctypes.c_int), ("d_rope", ctypes.c_int),
                ("d_nope", ctypes.c_int), ("d_v", ctypes.c_int), ("block_size", ctypes.c_int),
                ("dtype", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("rope_base", ctypes.c_double)]


def config(heads, d_latent, d_rope, d_nope, d_v, block_size, dtype, softmax_scale=None,
           rope_base=10000.0):
    if isinstance(dtype, str):
        dtype = {"bf16": DTYPE_BF16, "f32": DTYPE_F32}[dtype]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d_nope + d_rope)
    return Config(heads, d_latent, d_rope, d_nope, d_v, block_size, dtype, softmax_scale,
                  rope_base)


def config_from(cfg_dict):
    c = cfg_dict
    return config(c["heads"], c["d_latent"], c["d_rope"], c["d_nope"], c["d_v"],
                  c["block_size"], c["dtype"], c["softmax_scale"], c["rope_base"])


_lib = None


def lib():
    """The loaded libmla.so; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmla.so not found at {LIB_PATH}: build it with "
                               "`python -m head_latent_attention_23_b300.build_lib`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        CP = ctypes.POINTER(Config)
        SZ = ctypes.POINTER(ctypes.c_size_t)
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_status_string.argtypes = [I]
        L.mla_version.restype = I
        L.mla_decode_path.argtypes = [CP]
        L.mla_get_status.argtypes = [P, ctypes.POINTER(I)]
        L.mla_append_latent.argtypes = [CP, P, I, I, P, P, P, P, I, I, P, I64, P, P]
        L.mla_absorb_q.argtypes = [CP, P, P, I, P, P]
        L.mla_decode_workspace_size.argtypes = [CP, I, SZ]
        L.mla_decode.argtypes = [CP, P, P, P, I64, P, I, P, I, P, P, P, ctypes.c_size_t, P]
        L.mla_decode_combine.argtypes = [CP, P, P, I, I, P, P, P]
        L.mla_project_out.argtypes = [CP, P, P, I, P, P, I, P, P]
        L.mla_query_proj_workspace_size.argtypes = [CP, I, I, SZ]
        L.mla_query_proj.argtypes = [CP, P, I, I, P, I, P, P, P, P, P, ctypes.c_size_t, P]
        L.mla_decode_noalloc.argtypes = [CP, P, P, P, I64, P, I, P, I, P, P, P]
        L.mla_set_wait_limit_ns.argtypes = [I64]
        LW = ctypes.POINTER(LayerWeights)
        L.mla_layer_decode_step_workspace_size.argtypes = [CP, LW, I, I, SZ]
        L.mla_layer_decode_step.argtypes = [CP, LW, P, P, I, P, I64, P, I, P, I, P,
                                            ctypes.c_size_t, P]
        L.mla_cached_decode_step_workspace_size.argtypes = [CP, I, I, SZ]
        L.mla_decode_multi_workspace_size.argtypes = [CP, I, I, I, SZ]
        L.mla_decode_multi.argtypes = [CP, P, P, P, I64, P, I, P, I, I, P, P, P, ctypes.c_size_t,
                                       P]
        L.mla_cached_decode_step.argtypes = [CP, P, P, P, P, P, I, P, I64, P, I, P, P, P, I, P,
                                             ctypes.c_size_t, P]
        for name in EXPORTS:
            if name not in ("mla_status_string", "mla_version"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_string(status):
    return lib().mla_status_string(int(status)).decode()


def _check(rc, where):
    if rc != MLA_OK:
        raise MLAError(rc, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _tdtype(cfg):
    return torch.bfloat16 if cfg.dtype == DTYPE_BF16 else torch.float32


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def set_wait_limit_ns(ns):
    """mla_set_wait_limit_ns: give-up time of the decode kernel's pipeline
    waits for later calls (ns <= 0: the default, 1 s).  For tests."""
    _check(lib().mla_set_wait_limit_ns(int(ns)), "mla_set_wait_limit_ns")


def decode_path(cfg):
    return int(lib().mla_decode_path(ctypes.byref(cfg)))


def get_status(stream=None):
    v = ctypes.c_int(0)
    _check(lib().mla_get_status(_stream(stream), ctypes.byref(v)), "mla_get_status")
    return v.value


def append_latent(cfg, x, w_dkv, seq_idx, pos, block_table, cache, dense_out=None,
                  stream=None):
    dt = _tdtype(cfg)
    n_tok, d_in = x.shape
    batch, max_blocks = block_table.shape
    num_blocks = cache.shape[0]
    rc = lib().mla_append_latent(
        ctypes.byref(cfg), _ptr(x, dt, "x"), n_tok, d_in, _ptr(w_dkv, dt, "w_dkv"),
        _ptr(seq_idx, torch.int32, "seq_idx"), _ptr(pos, torch.int32, "pos"),
        _ptr(block_table, torch.int32, "block_table"), batch, max_blocks,
        _ptr(cache, dt, "cache"), num_blocks, _ptr(dense_out, dt, "dense_out"), _stream(stream))
    _check(rc, "mla_append_latent")


def absorb_q(cfg, q_nope, w_uk, q_lat, stream=None):
    dt = _tdtype(cfg)
    rc = lib().mla_absorb_q(ctypes.byref(cfg), _ptr(q_nope, dt, "q_nope"),
                            _ptr(w_uk, dt, "w_uk"), q_nope.shape[0], _ptr(q_lat, dt, "q_lat"),
                            _stream(stream))
    _check(rc, "mla_absorb_q")


def decode_workspace_size(cfg, batch):
    n = ctypes.c_size_t(0)
    _check(lib().mla_decode_workspace_size(ctypes.byref(cfg), batch, ctypes.byref(n)),
           "mla_decode_workspace_size")
    return n.value


def decode_workspace(cfg, batch, device=None):
    """A uint8 CUDA tensor big enough for mla_decode (allocated by torch)."""
    return torch.empty(decode_workspace_size(cfg, batch), dtype=torch.uint8,
                       device=device or "cuda")


def decode(cfg, q_lat, q_pe, cache, block_table, seq_lens, o_lat, lse=None, workspace=None,
           stream=None):
    dt = _tdtype(cfg)
    batch, max_blocks = block_table.shape
    if workspace is None:
        workspace = decode_workspace(cfg, batch, q_lat.device)
    rc = lib().mla_decode(
        ctypes.byref(cfg), _ptr(q_lat, dt, "q_lat"), _ptr(q_pe, dt, "q_pe"),
        _ptr(cache, dt, "cache"), cache.shape[0], _ptr(block_table, torch.int32, "block_table"),
        max_blocks, _ptr(seq_lens, torch.int32, "seq_lens"), batch, _ptr(o_lat, dt, "o_lat"),
        _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mla_decode")


def decode_noalloc(cfg, q_lat, q_pe, cache, block_table, seq_lens, o_lat, lse=None,
                   stream=None):
    """mla_decode_noalloc: mla_decode with its partials in the library's static
    device array instead of a caller workspace (for callers that cannot
    allocate).  Calls on one device must not overlap on the GPU."""
    dt = _tdtype(cfg)
    batch, max_blocks = block_table.shape
    rc = lib().mla_decode_noalloc(
        ctypes.byref(cfg), _ptr(q_lat, dt, "q_lat"), _ptr(q_pe, dt, "q_pe"),
        _ptr(cache, dt, "cache"), cache.shape[0], _ptr(block_table, torch.int32, "block_table"),
        max_blocks, _ptr(seq_lens, torch.int32, "seq_lens"), batch, _ptr(o_lat, dt, "o_lat"),
        _ptr(lse, torch.float32, "lse"), _stream(stream))
    _check(rc, "mla_decode_noalloc")


def decode_combine(cfg, o_part, lse_part, o_lat, lse=None, stream=None):
    n_splits, batch = lse_part.shape[0], lse_part.shape[1]
    rc = lib().mla_decode_combine(
        ctypes.byref(cfg), _ptr(o_part, torch.float32, "o_part"),
        _ptr(lse_part, torch.float32, "lse_part"), n_splits, batch,
        _ptr(o_lat, _tdtype(cfg), "o_lat"), _ptr(lse, torch.float32, "lse"), _stream(stream))
    _check(rc, "mla_decode_combine")


def project_out(cfg, o_lat, w_uv, o_v, w_o=None, out=None, stream=None):
    dt = _tdtype(cfg)
    d_model = w_o.shape[1] if w_o is not None else 0
    rc = lib().mla_project_out(
        ctypes.byref(cfg), _ptr(o_lat, dt, "o_lat"), _ptr(w_uv, dt, "w_uv"), o_lat.shape[0],
        _ptr(o_v, dt, "o_v"), _ptr(w_o, dt, "w_o"), d_model, _ptr(out, dt, "out"),
        _stream(stream))
    _check(rc, "mla_project_out")


def query_proj_workspace_size(cfg, batch, d_lq):
    n = ctypes.c_size_t(0)
    _check(lib().mla_query_proj_workspace_size(ctypes.byref(cfg), batch, d_lq,
                                               ctypes.byref(n)),
           "mla_query_proj_workspace_size")
    return n.value


def query_proj(cfg, x, w_uq, pos, q_nope, q_pe, w_dq=None, scratch=None, stream=None):
    dt = _tdtype(cfg)
    batch, d_in = x.shape
    d_lq = w_dq.shape[1] if w_dq is not None else 0
    if scratch is None:
        scratch = torch.empty(query_proj_workspace_size(cfg, batch, d_lq), dtype=torch.uint8,
                              device=x.device)
    rc = lib().mla_query_proj(
        ctypes.byref(cfg), _ptr(x, dt, "x"), batch, d_in, _ptr(w_dq, dt, "w_dq"), d_lq,
        _ptr(w_uq, dt, "w_uq"), _ptr(pos, torch.int32, "pos"), _ptr(q_nope, dt, "q_nope"),
        _ptr(q_pe, dt, "q_pe"), _ptr(scratch, None, "scratch"),
        scratch.numel() * scratch.element_size(), _stream(stream))
    _check(rc, "mla_query_proj")


# ---------------------------------------------------------------- whole steps

def _ptr_io(t, dtype, name, host):
    """Device pointer, or (host=True) pointer of a pinned, contiguous CPU tensor."""
    if not host:
        return _ptr(t, dtype, name)
    if t.is_cuda or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def layer_weights(cfg, w_dkv, w_uq, w_uk, w_uv, w_o, w_dq=None):
    """mla_layer_weights for device weight tensors (kept alive by the caller)."""
    dt = _tdtype(cfg)
    return LayerWeights(int(w_o.shape[1]), int(w_dq.shape[1]) if w_dq is not None else 0,
                        _ptr(w_dkv, dt, "w_dkv"), _ptr(w_dq, dt, "w_dq"), _ptr(w_uq, dt, "w_uq"),
                        _ptr(w_uk, dt, "w_uk"), _ptr(w_uv, dt, "w_uv"), _ptr(w_o, dt, "w_o"))


def layer_decode_step_workspace_size(cfg, weights, batch, max_blocks):
    n = ctypes.c_size_t(0)
    _check(lib().mla_layer_decode_step_workspace_size(ctypes.byref(cfg), ctypes.byref(weights),
                                                       batch, max_blocks, ctypes.byref(n)),
           "mla_layer_decode_step_workspace_size")
    return n.value


def layer_decode_step(cfg, weights, x, seq_lens, cache, block_table, out, io_flags=0,
                      workspace=None, stream=None):
    """mla_layer_decode_step: one full decode step (append, query, attention, W_O)."""
    dt = _tdtype(cfg)
    hin, hout = bool(io_flags & IO_HOST_INPUTS), bool(io_flags & IO_HOST_OUTPUT)
    batch, max_blocks = block_table.shape
    if workspace is None:
        workspace = torch.empty(layer_decode_step_workspace_size(cfg, weights, batch, max_blocks),
                                dtype=torch.uint8, device=cache.device)
    rc = lib().mla_layer_decode_step(
        ctypes.byref(cfg), ctypes.byref(weights), _ptr_io(x, dt, "x", hin),
        _ptr_io(seq_lens, torch.int32, "seq_lens", hin), batch, _ptr(cache, dt, "cache"),
        cache.shape[0], _ptr_io(block_table, torch.int32, "block_table", hin), max_blocks,
        _ptr_io(out, dt, "out", hout), int(io_flags), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mla_layer_decode_step")


def cached_decode_step_workspace_size(cfg, batch, max_blocks):
    n = ctypes.c_size_t(0)
    _check(lib().mla_cached_decode_step_workspace_size(ctypes.byref(cfg), batch, max_blocks,
                                                        ctypes.byref(n)),
           "mla_cached_decode_step_workspace_size")
    return n.value


def cached_decode_step(cfg, q_nope, q_pe, w_uk, w_uv, seq_lens, cache, block_table, o_v,
                       o_lat=None, lse=None, io_flags=0, workspace=None, stream=None):
    """mla_cached_decode_step: absorb, attention and value projection in one call."""
    dt = _tdtype(cfg)
    hin, hout = bool(io_flags & IO_HOST_INPUTS), bool(io_flags & IO_HOST_OUTPUT)
    batch, max_blocks = block_table.shape
    if workspace is None:
        workspace = torch.empty(cached_decode_step_workspace_size(cfg, batch, max_blocks),
                                dtype=torch.uint8, device=cache.device)
    rc = lib().mla_cached_decode_step(
        ctypes.byref(cfg), _ptr_io(q_nope, dt, "q_nope", hin), _ptr_io(q_pe, dt, "q_pe", hin),
        _ptr(w_uk, dt, "w_uk"), _ptr(w_uv, dt, "w_uv"),
        _ptr_io(seq_lens, torch.int32, "seq_lens", hin), batch, _ptr(cache, dt, "cache"),
        cache.shape[0], _ptr_io(block_table, torch.int32, "block_table", hin), max_blocks,
        _ptr_io(o_v, dt, "o_v", hout), _ptr(o_lat, dt, "o_lat"), _ptr(lse, torch.float32, "lse"),
        int(io_flags), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mla_cached_decode_step")


def decode_multi_workspace_size(cfg, batch, q_tokens, max_blocks):
    n = ctypes.c_size_t(0)
    _check(lib().mla_decode_multi_workspace_size(ctypes.byref(cfg), batch, q_tokens, max_blocks,
                                                  ctypes.byref(n)),
           "mla_decode_multi_workspace_size")
    return n.value


def decode_multi(cfg, q_lat, q_pe, cache, block_table, seq_lens, o_lat, lse=None,
                 workspace=None, stream=None):
    """mla_decode_multi: q_lat [batch][q_tokens][heads][d_latent], the last
    q_tokens tokens of each sequence with the causal mask among them."""
    dt = _tdtype(cfg)
    batch, max_blocks = block_table.shape
    q_tokens = q_lat.shape[1]
    if workspace is None:
        workspace = torch.empty(decode_multi_workspace_size(cfg, batch, q_tokens, max_blocks),
                                dtype=torch.uint8, device=q_lat.device)
    rc = lib().mla_decode_multi(
        ctypes.byref(cfg), _ptr(q_lat, dt, "q_lat"), _ptr(q_pe, dt, "q_pe"),
        _ptr(cache, dt, "cache"), cache.shape[0], _ptr(block_table, torch.int32, "block_table"),
        max_blocks, _ptr(seq_lens, torch.int32, "seq_lens"), batch, q_tokens,
        _ptr(o_lat, dt, "o_lat"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    _check(rc, "mla_decode_multi")
