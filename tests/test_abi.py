"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

from video_dit_long_gb300 import build as B
from video_dit_long_gb300 import k6attn as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "k6attn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(k6attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == sorted(K.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(6):
        assert lib.k6attn_status_string(s)
    assert lib.k6attn_status_string(99) == b"unknown status"


FAKE_A = ctypes.c_void_p(0x10000000)  # never dereferenced: validation fails first
FAKE_B = ctypes.c_void_p(0x20000000)


def relayout(lib, S, H, P, d=128, eb=2, direction=0, src=FAKE_A, dst=FAKE_B):
    return lib.k6attn_seq2head_relayout(src, dst, 1, S, H, d, eb, P, direction, None)


def test_relayout_rejects_indivisible_sequence(lib):
    # the pages' worked example: 3645 tokens cannot split 8 ways
    assert relayout(lib, 3645, 8, 8) == K.ERR_INVALID_ARG
    assert b"3645" in lib.k6attn_last_error()


def test_relayout_rejects_bad_arguments(lib):
    assert relayout(lib, 16, 24, 16) == K.ERR_INVALID_ARG            # H % P
    assert relayout(lib, 16, 8, 2, eb=3) == K.ERR_INVALID_ARG        # element size
    assert relayout(lib, 16, 8, 2, direction=2) == K.ERR_INVALID_ARG
    assert relayout(lib, 16, 8, 2, src=ctypes.c_void_p(0x10000008)) == K.ERR_INVALID_ARG  # misaligned
    assert relayout(lib, 16, 8, 2, src=None) == K.ERR_INVALID_ARG
    # overlapping buffers
    assert relayout(lib, 1024, 8, 2, dst=ctypes.c_void_p(0x10000000 + 4096)) == K.ERR_INVALID_ARG


def test_null_handle_is_rejected(lib):
    assert lib.k6attn_forward(None, FAKE_A, FAKE_A, FAKE_A, None, None, None, 1, FAKE_B, None, None, 0,
                              None) == K.ERR_INVALID_ARG
    assert lib.k6attn_lse_merge(None, FAKE_A, FAKE_A, 2, FAKE_B, None, None) == K.ERR_INVALID_ARG
    assert lib.k6attn_sync(None, None) == K.ERR_INVALID_ARG
    assert lib.k6attn_set_option(None, 0, 1) == K.ERR_INVALID_ARG
    assert lib.k6attn_workspace_bytes(None, 2, 1) == 0
    lib.k6attn_destroy(None)


def test_create_rejects_bad_descriptors_before_any_cuda_call(lib):
    def create(**kw):
        base = dict(B=1, H=24, d=128, dtype=K.BF16, grid_t=2, grid_h=3, grid_w=4, axis_dim=(32, 48, 48),
                    theta=10000.0, n_joint=8, joint_rope=0)
        base.update(kw)
        desc = K.Desc(base["B"], base["H"], base["d"], base["dtype"], base["grid_t"], base["grid_h"],
                      base["grid_w"], (ctypes.c_int * 3)(*base["axis_dim"]), base["theta"], base["n_joint"],
                      base["joint_rope"])
        h = ctypes.c_void_p()
        return lib.k6attn_create(ctypes.byref(desc), ctypes.byref(h))

    assert create(d=96) == K.ERR_UNSUPPORTED
    assert create(d=64, axis_dim=(16, 24, 24)) == K.ERR_UNSUPPORTED       # bf16 wants d = 128
    assert create(axis_dim=(32, 48, 40)) == K.ERR_INVALID_ARG              # sum != d
    assert create(axis_dim=(33, 47, 48)) == K.ERR_INVALID_ARG              # odd
    assert create(grid_t=0) == K.ERR_INVALID_ARG
    assert create(n_joint=-1) == K.ERR_INVALID_ARG
    assert create(theta=0.0) == K.ERR_INVALID_ARG
    assert create(joint_rope=2) == K.ERR_INVALID_ARG
    assert create(dtype=7) == K.ERR_INVALID_ARG


def test_load_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(K, "_lib", None)
    monkeypatch.setattr(K._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(OSError):
        K.load(build_if_missing=False)
