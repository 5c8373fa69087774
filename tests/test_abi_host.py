"""Host-side checks of the C ABI: the library loads, exports every symbol include/msa.h
declares, and rejects bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from block_sparse_gqa_02_gb300 import _lib
from block_sparse_gqa_02_gb300._lib import (MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED,
                                            make_shape)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "msa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_abi_version(lib):
    assert lib.msa_abi_version() == 2
    assert lib.msa_debug_build() == 0          # the release build


def test_status_strings(lib):
    for code in range(6):
        assert lib.msa_status_string(code).startswith(b"MSA_")


def _good_prefill():
    return make_shape(1, 1024, 1024, 16, 4, 64, 64, 64, 4, 64, "f32")


def _good_decode():
    return make_shape(8, 1, 1 << 20, 64, 4, 128, 128, 128, 64, 1, "bf16")


FAKE = 1 << 20          # a 16-byte aligned non-null pointer value; never dereferenced here


def call_index(lib, shape, a=FAKE, b=FAKE, c=FAKE):
    return lib.msa_index_scores(ctypes.byref(shape), a, b, c, None)


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, MSA_ERR_INVALID_ARG),
    ("seq_q", 0, MSA_ERR_INVALID_ARG),
    ("n_heads_q", 6, MSA_ERR_INVALID_ARG),          # not a multiple of 4 KV heads
    ("block_size", 0, MSA_ERR_INVALID_ARG),
    ("top_k", 0, MSA_ERR_INVALID_ARG),
    ("q_tile", 48, MSA_ERR_INVALID_ARG),            # block 64 % 48 != 0
    ("seq_k", 1000, MSA_ERR_INVALID_ARG),           # prefill with seq_q != seq_k
    ("dtype", 7, MSA_ERR_INVALID_ARG),
    ("head_dim", 96, MSA_ERR_UNSUPPORTED),
    ("index_dim", 32, MSA_ERR_UNSUPPORTED),
    ("sm_scale", -1.0, MSA_ERR_INVALID_ARG),
    ("index_scale", float("inf"), MSA_ERR_INVALID_ARG),
])
def test_bad_shape_rejected(lib, field, value, status):
    s = _good_prefill()
    setattr(s, field, value)
    assert call_index(lib, s) == status
    assert lib.msa_last_error() != b""


def test_too_many_blocks(lib):
    s = make_shape(1, 1 << 22, 1 << 22, 16, 4, 64, 64, 64, 4, 64, "bf16")  # 65536 blocks
    assert call_index(lib, s) == MSA_ERR_UNSUPPORTED


def test_grid_limits(lib):
    # 65536 query tiles (q_tile 1), and batch * n_heads_kv beyond a grid dimension
    s = make_shape(1, 65536, 65536, 16, 4, 64, 64, 64, 4, 1, "bf16")
    assert call_index(lib, s) == MSA_ERR_UNSUPPORTED
    assert b"query tiles" in lib.msa_last_error()
    s = make_shape(16384, 1024, 1024, 32, 8, 64, 64, 64, 4, 64, "bf16")
    assert call_index(lib, s) == MSA_ERR_UNSUPPORTED
    assert b"n_heads_kv" in lib.msa_last_error()


def test_null_and_misaligned_pointers(lib):
    s = _good_prefill()
    assert call_index(lib, s, a=None) == MSA_ERR_INVALID_ARG
    assert b"idx_q" in lib.msa_last_error()
    assert call_index(lib, s, b=FAKE + 4) == MSA_ERR_INVALID_ARG
    assert b"aligned" in lib.msa_last_error()
    assert lib.msa_block_topk(ctypes.byref(s), FAKE, None, None) == MSA_ERR_INVALID_ARG
    assert lib.msa_sparse_prefill(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None, None, 0,
                                  None) == MSA_ERR_INVALID_ARG
    # lse misaligned (nullable but, when given, must be aligned)
    assert lib.msa_sparse_prefill(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, None,
                                  0, None) == MSA_ERR_INVALID_ARG


def test_decode_checks(lib):
    d = _good_decode()
    need = lib.msa_workspace_bytes(ctypes.byref(d), 1)
    assert need > 0
    # workspace too small / missing
    assert lib.msa_sparse_decode(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                 need - 16, None) == MSA_ERR_INVALID_ARG
    assert b"workspace" in lib.msa_last_error()
    assert lib.msa_sparse_decode(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                                 need, None) == MSA_ERR_INVALID_ARG
    # a prefill shape is not a decode shape
    p = _good_prefill()
    assert lib.msa_sparse_decode(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                 1 << 30, None) == MSA_ERR_INVALID_ARG
    # and decode shapes go to msa_sparse_decode
    assert lib.msa_sparse_prefill(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0,
                                  None) == MSA_ERR_INVALID_ARG


def test_workspace_bytes(lib):
    d = _good_decode()
    n = lib.msa_workspace_bytes(ctypes.byref(d), 1)
    # partial outputs and lse, fp32, per (sequence, query head, split)
    slots = n // ((128 + 1) * 4)
    assert slots * (128 + 1) * 4 == n
    assert slots % (8 * 64) == 0 and 1 <= slots // (8 * 64) <= 64
    assert lib.msa_workspace_bytes(ctypes.byref(_good_prefill()), 0) == 0
    bad = _good_decode()
    bad.batch = 0
    assert lib.msa_workspace_bytes(ctypes.byref(bad), 1) == 0


def test_python_binding_raises(lib):
    s = _good_prefill()
    with pytest.raises(_lib.MsaError) as ei:
        _lib.msa_index_scores(s, None, FAKE, FAKE, stream=0)
    assert ei.value.status == MSA_ERR_INVALID_ARG


def test_index_kl_tensor_core_covers_the_longest_accepted_sequence(lib):
    """The tensor-core index KL keeps a key block's query-tile list in 16-bit entries; the
    shape check accepts at most 65535 query tiles a sequence, so the longest accepted prefill
    still takes that path, and one tile more is refused before anything runs."""
    t = 65535 * 64
    longest = make_shape(1, t, t, 32, 4, 128, 128, 128, 16, 64, "bf16")
    assert lib.msa_workspace_bytes(ctypes.byref(longest), 3) > 0
    past = make_shape(1, t + 64, t + 64, 32, 4, 128, 128, 128, 16, 64, "bf16")
    assert lib.msa_workspace_bytes(ctypes.byref(past), 3) == 0
    assert b"query tiles" in lib.msa_last_error()


def test_training_workspace_and_checks(lib):
    """The tensor-core backward and index KL need a workspace (sized by which = 2 / 3) and
    refuse a missing or short one; CUDA-core shapes need none."""
    tc = make_shape(1, 4096, 4096, 32, 4, 128, 128, 128, 16, 64, "bf16")
    simt = make_shape(1, 1024, 1024, 16, 4, 64, 64, 64, 4, 64, "f32")
    for which in (2, 3):
        need = lib.msa_workspace_bytes(ctypes.byref(tc), which)
        assert need > 0 and need % 16 == 0
        assert lib.msa_workspace_bytes(ctypes.byref(simt), which) == 0
        assert lib.msa_workspace_bytes(ctypes.byref(_good_decode()), which) == 0
    need = lib.msa_workspace_bytes(ctypes.byref(tc), 2)
    args = [FAKE] * 10
    assert lib.msa_sparse_prefill_backward(ctypes.byref(tc), *args, None, need,
                                           None) == MSA_ERR_INVALID_ARG
    assert b"workspace" in lib.msa_last_error()
    assert lib.msa_sparse_prefill_backward(ctypes.byref(tc), *args, FAKE, need - 16,
                                           None) == MSA_ERR_INVALID_ARG
    need = lib.msa_workspace_bytes(ctypes.byref(tc), 3)
    args = [FAKE] * 9
    assert lib.msa_index_kl_loss(ctypes.byref(tc), *args, FAKE, need - 16,
                                 None) == MSA_ERR_INVALID_ARG
    assert b"workspace" in lib.msa_last_error()
    # decode shapes are not training shapes
    d = _good_decode()
    assert lib.msa_sparse_prefill_backward(ctypes.byref(d), *([FAKE] * 10), FAKE, 1 << 30,
                                           None) == MSA_ERR_INVALID_ARG
