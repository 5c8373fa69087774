"""ctypes binding of libmsa.so: the C ABI in include/msa.h, argument marshalling only.

Every computation runs in the library's CUDA kernels.  Tensors are passed as raw device
pointers (``tensor.data_ptr()``) together with the current torch CUDA stream; a missing
library or CUDA device raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

(MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_CUDA, MSA_ERR_TIMEOUT,
 MSA_ERR_BOUNDS) = range(6)
MSA_F32, MSA_BF16 = 0, 1
_DTYPE_CODES = {"f32": MSA_F32, "bf16": MSA_BF16}

# Every function include/msa.h declares, with its ctypes signature.
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t


class MsaShape(ctypes.Structure):
    """Mirror of ``msa_shape``."""
    _fields_ = [("batch", _i32), ("seq_q", _i32), ("seq_k", _i32), ("n_heads_q", _i32),
                ("n_heads_kv", _i32), ("head_dim", _i32), ("index_dim", _i32),
                ("block_size", _i32), ("top_k", _i32), ("q_tile", _i32), ("dtype", _i32),
                ("sm_scale", ctypes.c_float), ("index_scale", ctypes.c_float)]

    @property
    def n_blocks(self) -> int:
        return -(-self.seq_k // self.block_size)

    @property
    def n_rows(self) -> int:
        return -(-self.seq_q // self.q_tile)

    def __repr__(self):
        return "MsaShape(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_SHAPE_P = ctypes.POINTER(MsaShape)
SIGNATURES = {
    "msa_index_scores": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp]),
    "msa_block_topk": (_i32, [_SHAPE_P, _vp, _vp, _vp]),
    "msa_index_topk_fused": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp]),
    "msa_block_topk_shared": (_i32, [_SHAPE_P, _vp, _vp, _vp]),
    "msa_sparse_prefill": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "msa_sparse_decode": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "msa_sparse_prefill_backward": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _sz, _vp]),
    "msa_index_kl_loss": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                 _sz, _vp]),
    "msa_sparse_decode_static": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "msa_index_scores_paged": (_i32, [_SHAPE_P, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "msa_block_topk_ragged": (_i32, [_SHAPE_P, _vp, _vp, _vp, _vp]),
    "msa_sparse_decode_paged": (_i32, [_SHAPE_P, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp, _sz, _vp]),
    "msa_workspace_bytes": (_sz, [_SHAPE_P, ctypes.c_int]),
    "msa_get_device_status": (_i32, [_vp]),
    "msa_status_string": (ctypes.c_char_p, [_i32]),
    "msa_last_error": (ctypes.c_char_p, []),
    "msa_abi_version": (_i32, []),
    "msa_debug_build": (_i32, []),
    "msa_debug_set_fault": (_i32, [_i32]),
}

_lock = threading.Lock()
_libs = {}                 # variant -> loaded library
# The variant the calls below go through: "release" (libmsa.so), or "debug"
# (libmsa_debug.so, built with the device-side index checks) when the environment sets
# MSA_LIBRARY_VARIANT=debug.  A process loads one variant: the two libraries export the same
# symbols and device variables.
_active = os.environ.get("MSA_LIBRARY_VARIANT", "release")


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({detail})")


def library_path(variant: str = "release") -> str:
    name = "libmsa.so" if variant == "release" else f"libmsa_{variant}.so"
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), name)


def load(build_if_missing: bool = True, variant: str | None = None):
    """The loaded library of `variant` (default: the process's variant, see
    MSA_LIBRARY_VARIANT), built in-tree with nvcc on first use if needed."""
    variant = _active if variant is None else variant
    if variant not in ("release", "debug"):
        raise ValueError(f"unknown MSA library variant {variant!r}")
    with _lock:
        if _libs and variant not in _libs:
            raise RuntimeError(f"the {next(iter(_libs))} MSA library is already loaded in this "
                               f"process; run the {variant} variant in a process of its own")
        if variant not in _libs:
            path = library_path(variant)
            if build_if_missing:
                from . import build as _build
                path = _build.build(variant=variant)
            if not os.path.exists(path):
                raise RuntimeError(f"MSA CUDA library missing at {path}; run the build first")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _libs[variant] = lib
        return _libs[variant]


def _ptr(x):
    """Device pointer of a tensor (must be contiguous), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("MSA tensors must be contiguous")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != MSA_OK:
        lib = load()
        detail = (lib.msa_last_error() or b"").decode() or \
            (lib.msa_status_string(status) or b"").decode()
        raise MsaError(status, where, detail)


def make_shape(batch, seq_q, seq_k, n_heads_q, n_heads_kv, head_dim, index_dim, block_size,
               top_k, q_tile, dtype="bf16", sm_scale=0.0, index_scale=0.0) -> MsaShape:
    code = _DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return MsaShape(batch, seq_q, seq_k, n_heads_q, n_heads_kv, head_dim, index_dim,
                    block_size, top_k, q_tile, code, sm_scale, index_scale)


def shape_from_config(cfg, **override) -> MsaShape:
    kw = dict(batch=cfg.batch, seq_q=cfg.seq_q, seq_k=cfg.seq_k, n_heads_q=cfg.n_heads_q,
              n_heads_kv=cfg.n_heads_kv, head_dim=cfg.head_dim, index_dim=cfg.index_dim,
              block_size=cfg.block_size, top_k=cfg.top_k, q_tile=cfg.q_tile, dtype=cfg.dtype)
    kw.update(override)
    return make_shape(**kw)


# ------------------------------------------------------------- the C-ABI calls

def msa_index_scores(shape: MsaShape, idx_q, idx_k, block_scores, stream=None):
    _check(load().msa_index_scores(ctypes.byref(shape), _ptr(idx_q), _ptr(idx_k),
                                   _ptr(block_scores), _stream(stream)), "msa_index_scores")


def msa_block_topk(shape: MsaShape, block_scores, sel, stream=None):
    _check(load().msa_block_topk(ctypes.byref(shape), _ptr(block_scores), _ptr(sel),
                                 _stream(stream)), "msa_block_topk")


def msa_block_topk_shared(shape: MsaShape, block_scores, sel, stream=None):
    """Ablation: one selection per row from the KV heads' summed scores, shared by all heads."""
    _check(load().msa_block_topk_shared(ctypes.byref(shape), _ptr(block_scores), _ptr(sel),
                                        _stream(stream)), "msa_block_topk_shared")


def msa_index_topk_fused(shape: MsaShape, idx_q, idx_k, sel, block_scores=None, stream=None):
    _check(load().msa_index_topk_fused(ctypes.byref(shape), _ptr(idx_q), _ptr(idx_k),
                                       _ptr(block_scores), _ptr(sel), _stream(stream)),
           "msa_index_topk_fused")


def msa_sparse_prefill(shape: MsaShape, q, k, v, sel, out, lse=None, workspace=None,
                       ws_bytes=0, stream=None):
    _check(load().msa_sparse_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(sel),
                                     _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                     _stream(stream)), "msa_sparse_prefill")


def msa_sparse_prefill_backward(shape: MsaShape, q, k, v, sel, out, lse, dout, dq, dk, dv,
                                workspace=None, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().msa_sparse_prefill_backward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(sel), _ptr(out), _ptr(lse), _ptr(dout),
                                              _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                              ws_bytes, _stream(stream)),
           "msa_sparse_prefill_backward")


def msa_index_kl_loss(shape: MsaShape, q, k, lse, idx_q, idx_k, sel, loss, d_idx_q, d_idx_k,
                      workspace=None, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().msa_index_kl_loss(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(lse),
                                    _ptr(idx_q), _ptr(idx_k), _ptr(sel), _ptr(loss),
                                    _ptr(d_idx_q), _ptr(d_idx_k), _ptr(workspace), ws_bytes,
                                    _stream(stream)),
           "msa_index_kl_loss")


def msa_sparse_decode(shape: MsaShape, q, k_cache, v_cache, sel, out, lse=None, workspace=None,
                      ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().msa_sparse_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(sel), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                    _stream(stream)), "msa_sparse_decode")


def msa_sparse_decode_static(shape: MsaShape, q, k_cache, v_cache, sel, out, lse=None,
                             stream=None):
    """msa_sparse_decode without a caller workspace: for callers that cannot allocate
    device memory where decode runs, the library's own static device scratch is used."""
    _check(load().msa_sparse_decode_static(ctypes.byref(shape), _ptr(q), _ptr(k_cache),
                                           _ptr(v_cache), _ptr(sel), _ptr(out), _ptr(lse),
                                           _stream(stream)), "msa_sparse_decode_static")


def msa_index_scores_paged(shape: MsaShape, seq_lens, block_table, n_phys, idx_q, idx_k_pool,
                           block_scores, stream=None):
    _check(load().msa_index_scores_paged(ctypes.byref(shape), _ptr(seq_lens), _ptr(block_table),
                                         int(n_phys), _ptr(idx_q), _ptr(idx_k_pool),
                                         _ptr(block_scores), _stream(stream)),
           "msa_index_scores_paged")


def msa_block_topk_ragged(shape: MsaShape, seq_lens, block_scores, sel, stream=None):
    _check(load().msa_block_topk_ragged(ctypes.byref(shape), _ptr(seq_lens), _ptr(block_scores),
                                        _ptr(sel), _stream(stream)), "msa_block_topk_ragged")


def msa_sparse_decode_paged(shape: MsaShape, seq_lens, block_table, n_phys, q, k_pool, v_pool,
                            sel, out, lse=None, workspace=None, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().msa_sparse_decode_paged(ctypes.byref(shape), _ptr(seq_lens), _ptr(block_table),
                                          int(n_phys), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                          _ptr(sel), _ptr(out), _ptr(lse), _ptr(workspace),
                                          ws_bytes, _stream(stream)), "msa_sparse_decode_paged")


def msa_workspace_bytes(shape: MsaShape, which: int) -> int:
    return int(load().msa_workspace_bytes(ctypes.byref(shape), which))


def msa_get_device_status(stream=None):
    _check(load().msa_get_device_status(_stream(stream)), "msa_get_device_status")


def msa_abi_version() -> int:
    return int(load().msa_abi_version())


def msa_debug_set_fault(mode: int):
    """Test hook: mode 1 makes tensor-core prefill launches time out (see include/msa.h)."""
    _check(load().msa_debug_set_fault(mode), "msa_debug_set_fault")
