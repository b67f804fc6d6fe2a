"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and rejects invalid arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from head_latent_attention_23_b300 import build_lib, mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return mla.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert sorted(mla.EXPORTS) == names


def test_status_strings(L):
    for code in range(7):
        assert mla.status_string(code) not in ("", "unknown status")
    assert mla.status_string(99) == "unknown status"
    assert L.mla_version() >= 100


def test_invalid_configs_are_rejected_on_the_host(L):
    n = ctypes.c_size_t(0)
    assert L.mla_decode_workspace_size(None, 4, ctypes.byref(n)) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_decode_path(None) == -1
    good = mla.config(128, 512, 64, 128, 128, 64, "bf16")
    bad = [
        dict(heads=0), dict(d_rope=63), dict(d_latent=0), dict(block_size=0), dict(dtype=7),
        dict(softmax_scale=float("nan")), dict(rope_base=-1.0), dict(d_nope=0),
    ]
    for kw in bad:
        c = mla.Config.from_buffer_copy(good)
        for k, v in kw.items():
            setattr(c, k, v)
        assert L.mla_decode_path(ctypes.byref(c)) == -1, kw
        assert L.mla_decode_workspace_size(ctypes.byref(c), 4, ctypes.byref(n)) == \
            mla.MLA_ERR_INVALID_ARG, kw
        assert L.mla_absorb_q(ctypes.byref(c), None, None, 1, None, None) == \
            mla.MLA_ERR_INVALID_ARG, kw


def test_bad_sizes_and_null_pointers_are_rejected(L):
    c = mla.config(128, 512, 64, 128, 128, 64, "bf16")
    cp = ctypes.byref(c)
    # batch out of range, null pointers: rejected before any CUDA call
    assert L.mla_decode(cp, None, None, None, 1, None, 1, None, 0, None, None, None, 0,
                        None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_decode(cp, None, None, None, 1, None, 1, None, 2, None, None, None, 0,
                        None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_decode_combine(cp, None, None, 0, 1, None, None, None) == \
        mla.MLA_ERR_INVALID_ARG
    assert L.mla_decode_combine(cp, None, None, 2000, 1, None, None, None) == \
        mla.MLA_ERR_INVALID_ARG
    assert L.mla_append_latent(cp, None, 1, 0, None, None, None, None, 1, 1, None, 1, None,
                               None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_append_latent(cp, None, 0, 16, None, None, None, None, 1, 1, None, 1, None,
                               None) == mla.MLA_OK          # nothing to append
    assert L.mla_project_out(cp, None, None, 2, None, None, 0, None, None) == \
        mla.MLA_ERR_INVALID_ARG
    assert L.mla_query_proj(cp, None, 2, 16, None, 0, None, None, None, None, None, 0,
                            None) == mla.MLA_ERR_INVALID_ARG


def test_step_calls_validate_on_the_host(L):
    c = mla.config(128, 512, 64, 128, 128, 64, "bf16")
    cp = ctypes.byref(c)
    n = ctypes.c_size_t(0)
    wts = mla.LayerWeights(0, 0, None, None, None, None, None, None)
    assert L.mla_layer_decode_step_workspace_size(cp, ctypes.byref(wts), 4, 8, ctypes.byref(n)) == \
        mla.MLA_ERR_INVALID_ARG
    assert L.mla_layer_decode_step_workspace_size(cp, None, 4, 8, ctypes.byref(n)) == \
        mla.MLA_ERR_INVALID_ARG
    assert L.mla_layer_decode_step(cp, ctypes.byref(wts), None, None, 4, None, 1, None, 8, None,
                                   0, None, 0, None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_cached_decode_step_workspace_size(cp, 0, 8, ctypes.byref(n)) == \
        mla.MLA_ERR_INVALID_ARG
    # unknown io flag bits and null inputs are refused before any CUDA call
    assert L.mla_cached_decode_step(cp, None, None, None, None, None, 4, None, 1, None, 8, None,
                                    None, None, 4, None, 0, None) == mla.MLA_ERR_INVALID_ARG
    assert L.mla_cached_decode_step(cp, None, None, None, None, None, 4, None, 1, None, 8, None,
                                    None, None, 0, None, 0, None) == mla.MLA_ERR_INVALID_ARG


def test_multi_token_decode_validates_on_the_host(L):
    c = mla.config(128, 512, 64, 128, 128, 64, "bf16")
    cp = ctypes.byref(c)
    n = ctypes.c_size_t(0)
    for batch, q_tokens in ((4, 0), (4, 65), (0, 2), (200, 64)):
        assert L.mla_decode_multi_workspace_size(cp, batch, q_tokens, 8, ctypes.byref(n)) == \
            mla.MLA_ERR_INVALID_ARG
        assert L.mla_decode_multi(cp, None, None, None, 1, None, 8, None, batch, q_tokens, None,
                                  None, None, 0, None) == mla.MLA_ERR_INVALID_ARG
    # a valid shape with null tensors is refused before any CUDA call
    assert L.mla_decode_multi(cp, None, None, None, 1, None, 8, None, 4, 2, None, None, None, 0,
                              None) == mla.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c_and_cpp(lang, std, tmp_path):
    """include/mla.h is a C ABI: it compiles on its own as C99 and as C++11,
    with warnings as errors, and needs no CUDA or torch header."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text('#include "mla.h"\nint probe(void) { return mla_version() > 0 ? MLA_OK : MLA_ERR_CUDA; }\n')
    r = subprocess.run([cc, "-fsyntax-only", "-Wall", "-Wextra", "-Werror", std, "-I",
                        os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
