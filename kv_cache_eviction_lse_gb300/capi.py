"""Thin Python binding of the kvs C ABI (include/kvs.h): argument marshalling only.

Every function has the name and argument order of its C counterpart.  Tensor
arguments are CUDA tensors (or None for an optional/NULL pointer); they are passed as
raw device pointers.  ``stream`` defaults to torch's current CUDA stream.  A non-zero
status raises :class:`KvsError` carrying the library's message.  Nothing is computed
here: every step runs in the library's CUDA kernels.  The library must have been built
(``kv_cache_eviction_lse_gb300.build``); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libkvs.so")

KVS_OK, KVS_ERR_ARG, KVS_ERR_SHAPE, KVS_ERR_ALIGN, KVS_ERR_UNSUPPORTED, KVS_ERR_CAPACITY, \
    KVS_ERR_CUDA, KVS_ERR_DEVICE = range(8)
KVS_THRESHOLD, KVS_TOPK = 0, 1
STATUS_NAMES = ["KVS_OK", "KVS_ERR_ARG", "KVS_ERR_SHAPE", "KVS_ERR_ALIGN", "KVS_ERR_UNSUPPORTED",
                "KVS_ERR_CAPACITY", "KVS_ERR_CUDA", "KVS_ERR_DEVICE"]


class KvsError(RuntimeError):
    def __init__(self, status: int, message: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("D_h", ctypes.c_int32)]

    def __repr__(self):
        return f"Dims(L={self.L}, H_q={self.H_q}, H_kv={self.H_kv}, d={self.d}, D_h={self.D_h})"


def dims(L, H_q, H_kv, d, D_h=0) -> Dims:
    return Dims(L, H_q, H_kv, d, D_h)


if not os.path.exists(LIB_PATH):
    raise ImportError(f"kvs CUDA library not built ({LIB_PATH} missing); run "
                      "`python -m kv_cache_eviction_lse_gb300.build` (needs nvcc)")
_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int32
_F = ctypes.c_float
_S = ctypes.c_size_t
_D = ctypes.POINTER(Dims)

_SIGS = {
    "kvs_version": ([], ctypes.c_char_p),
    "kvs_last_error": ([], ctypes.c_char_p),
    "kvs_launch_count": ([], ctypes.c_uint64),
    "kvs_device_error": ([ctypes.POINTER(ctypes.c_int32), _I, _P], ctypes.c_int),
    "kvs_lse": ([_D, _P, _I, _P, _I, _P, _I, _P, _P], ctypes.c_int),
    "kvs_score_max_workspace_size": ([_D, _I, _I], _S),
    "kvs_score_max": ([_D, _P, _I, _P, _I, _P, _P, _P, _I, _P, _P, _S, _P], ctypes.c_int),
    "kvs_score_future_sum_workspace_size": ([_D, _I], ctypes.c_size_t),
    "kvs_score_future_sum": ([_D, _P, _P, _I, _P, _I, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "kvs_vnorm_workspace_size": ([_D], _S),
    "kvs_vnorm": ([_D, _P, _I, _P, _P, _P, _S, _P], ctypes.c_int),
    "kvs_vnorm_noalloc": ([_D, _P, _I, _P, _P, _P], ctypes.c_int),
    "kvs_value_refit_workspace_size": ([_D, _I, _I], ctypes.c_size_t),
    "kvs_value_refit": ([_D, _P, _I, _P, _P, _I, _P, _I, _F, _P, _P, ctypes.c_size_t, _P],
                        ctypes.c_int),
    "kvs_decode_step": ([_D, _I, _I, _P, _P, _P, _P, _P, _P, _P, _F, _I, _P, _P, _I, _P, _P, _I,
                         _P, _I, _P], ctypes.c_int),
    "kvs_attn_fwd": ([_D, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _P], ctypes.c_int),
    "kvs_surrogate": ([_D, _P, _I, _P, _P, _P, _F, _I, _P, _P, _P], ctypes.c_int),
    "kvs_surrogate_mlp": ([_D, _P, _I, _I, _P, _P, _P, _P, _P, _F, _I, _P, _P, _P], ctypes.c_int),
    "kvs_prune_mask": ([_D, _P, _I, _I, _F, _I, _I, _P, _P, _P], ctypes.c_int),
    "kvs_compact_workspace_size": ([_D, _I], _S),
    "kvs_compact_paged": ([_D, _P, _P, _I, _P, _I, _P, _P, _I, _P, _I, _P, _P, _P, _S, _P],
                          ctypes.c_int),
    "kvs_prune_quantile": ([_D, _P, _I, _F, _I, _P, _P, _P, _P], ctypes.c_int),
    "kvs_prune_topk_multi": ([_D, _P, _I, _I, _P, _I, _P, _P, _P], ctypes.c_int),
    "kvs_compact_multi_workspace_size": ([_D, _I, _I], _S),
    "kvs_compact_paged_multi": ([_D, _P, _P, _I, _I, _P, _I, _P, _P, _I, _P, _I, _P, _P, _P, _S,
                                 _P], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

EXPORTED = tuple(_SIGS)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("kvs: tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("kvs: tensor arguments must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != KVS_OK:
        raise KvsError(status, _lib.kvs_last_error().decode())


def _d(dm: Dims):
    return ctypes.byref(dm)


def kvs_version() -> str:
    return _lib.kvs_version().decode()


def kvs_last_error() -> str:
    return _lib.kvs_last_error().decode()


def kvs_launch_count() -> int:
    return int(_lib.kvs_launch_count())


def kvs_device_error(clear: bool = True, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(_lib.kvs_device_error(ctypes.byref(code), int(clear), _stream(stream)))
    return code.value


def kvs_lse(dm, q, n_q, k_ctx, T, k_tail, n_tail, lse, stream=None):
    _check(_lib.kvs_lse(_d(dm), _ptr(q), n_q, _ptr(k_ctx), T, _ptr(k_tail), n_tail, _ptr(lse),
                        _stream(stream)))


def kvs_score_max_workspace_size(dm, n_q, with_h) -> int:
    return _lib.kvs_score_max_workspace_size(_d(dm), n_q, int(with_h))


def kvs_score_max(dm, q, n_q, k_ctx, T, lse, vnorm, h, accumulate, log_score, ws, ws_bytes,
                  stream=None):
    _check(_lib.kvs_score_max(_d(dm), _ptr(q), n_q, _ptr(k_ctx), T, _ptr(lse), _ptr(vnorm),
                              _ptr(h), int(accumulate), _ptr(log_score), _ptr(ws), ws_bytes,
                              _stream(stream)))


def kvs_score_future_sum_workspace_size(dm, T):
    return int(_lib.kvs_score_future_sum_workspace_size(_d(dm), T))


def kvs_score_future_sum(dm, q, k, T, lse, w, score, ws, ws_bytes, stream=None):
    _check(_lib.kvs_score_future_sum(_d(dm), _ptr(q), _ptr(k), T, _ptr(lse), w, _ptr(score),
                                     _ptr(ws), ws_bytes, _stream(stream)))


def kvs_vnorm_workspace_size(dm) -> int:
    return _lib.kvs_vnorm_workspace_size(_d(dm))


def kvs_vnorm(dm, v, T, w_o, vnorm, ws, ws_bytes, stream=None):
    _check(_lib.kvs_vnorm(_d(dm), _ptr(v), T, _ptr(w_o), _ptr(vnorm), _ptr(ws), ws_bytes,
                          _stream(stream)))


def kvs_vnorm_noalloc(dm, v, T, w_o, vnorm, stream=None):
    """kvs_vnorm without a workspace argument: uses the library's built-in device
    scratch (for callers that cannot allocate device memory; see include/kvs.h)."""
    _check(_lib.kvs_vnorm_noalloc(_d(dm), _ptr(v), T, _ptr(w_o), _ptr(vnorm), _stream(stream)))


def kvs_attn_fwd(dm, q, n_q, k_ctx, v_ctx, T, k_tail, v_tail, n_tail, o, lse, stream=None):
    _check(_lib.kvs_attn_fwd(_d(dm), _ptr(q), n_q, _ptr(k_ctx), _ptr(v_ctx), T, _ptr(k_tail),
                             _ptr(v_tail), n_tail, _ptr(o), _ptr(lse), _stream(stream)))


def kvs_value_refit_workspace_size(dm, n_q, k):
    return int(_lib.kvs_value_refit_workspace_size(_d(dm), n_q, k))


def kvs_value_refit(dm, q, n_q, k_ctx, v_ctx, T, k_kept, k, lambda_rel, v_fit, ws, ws_bytes,
                    stream=None):
    _check(_lib.kvs_value_refit(_d(dm), _ptr(q), n_q, _ptr(k_ctx), _ptr(v_ctx), T, _ptr(k_kept),
                                k, float(lambda_rel), _ptr(v_fit), _ptr(ws), ws_bytes,
                                _stream(stream)))


def kvs_decode_step(dm, B, w, pos, new_score, new_k, new_v, ring_score, ring_k, ring_v, tau,
                    page_size, k_pages, v_pages, capacity_pages, next_page, block_table,
                    max_pages, seq_lens, advance_pos=True, stream=None):
    _check(_lib.kvs_decode_step(_d(dm), B, w, _ptr(pos), _ptr(new_score), _ptr(new_k),
                                _ptr(new_v), _ptr(ring_score), _ptr(ring_k), _ptr(ring_v),
                                float(tau), page_size, _ptr(k_pages), _ptr(v_pages),
                                capacity_pages, _ptr(next_page), _ptr(block_table), max_pages,
                                _ptr(seq_lens), 1 if advance_pos else 0, _stream(stream)))


def kvs_surrogate(dm, h, T, W, b, score, tau=0.0, w=0, mask=None, keep=None, stream=None):
    _check(_lib.kvs_surrogate(_d(dm), _ptr(h), T, _ptr(W), _ptr(b), _ptr(score), float(tau), w,
                              _ptr(mask), _ptr(keep), _stream(stream)))


def kvs_surrogate_mlp(dm, h, T, D_mid, W1, b1, W2, b2, score, tau=0.0, w=0, mask=None, keep=None,
                      stream=None):
    _check(_lib.kvs_surrogate_mlp(_d(dm), _ptr(h), T, D_mid, _ptr(W1), _ptr(b1), _ptr(W2),
                                  _ptr(b2), _ptr(score), float(tau), w, _ptr(mask), _ptr(keep),
                                  _stream(stream)))


def kvs_prune_mask(dm, score, T, mode, tau, k, w, mask, keep, stream=None):
    _check(_lib.kvs_prune_mask(_d(dm), _ptr(score), T, mode, float(tau), k, w, _ptr(mask),
                               _ptr(keep), _stream(stream)))


def kvs_prune_quantile(dm, score, T, q, w, tau, mask, keep, stream=None):
    _check(_lib.kvs_prune_quantile(_d(dm), _ptr(score), T, float(q), w, _ptr(tau), _ptr(mask),
                                   _ptr(keep), _stream(stream)))


def kvs_prune_topk_multi(dm, score, T, ks, w, masks, keeps, stream=None):
    """ks: a sequence of budgets (marshalled into a host int32 array)."""
    arr = (ctypes.c_int32 * max(1, len(ks)))(*[int(k) for k in ks])
    _check(_lib.kvs_prune_topk_multi(_d(dm), _ptr(score), T, len(ks), ctypes.cast(arr, _P), w,
                                     _ptr(masks),
                                     _ptr(keeps), _stream(stream)))


def kvs_compact_multi_workspace_size(dm, T, n_masks) -> int:
    return _lib.kvs_compact_multi_workspace_size(_d(dm), T, n_masks)


def kvs_compact_paged_multi(dm, k, v, T, n_masks, masks, page_size, k_pages, v_pages,
                            capacity_pages, block_table, max_pages, seq_lens, needed_pages, ws,
                            ws_bytes, stream=None):
    _check(_lib.kvs_compact_paged_multi(_d(dm), _ptr(k), _ptr(v), T, n_masks, _ptr(masks),
                                        page_size, _ptr(k_pages), _ptr(v_pages), capacity_pages,
                                        _ptr(block_table), max_pages, _ptr(seq_lens),
                                        _ptr(needed_pages), _ptr(ws), ws_bytes, _stream(stream)))


def kvs_compact_workspace_size(dm, T) -> int:
    return _lib.kvs_compact_workspace_size(_d(dm), T)


def kvs_compact_paged(dm, k, v, T, mask, page_size, k_pages, v_pages, capacity_pages,
                      block_table, max_pages, seq_lens, needed_pages, ws, ws_bytes, stream=None):
    _check(_lib.kvs_compact_paged(_d(dm), _ptr(k), _ptr(v), T, _ptr(mask), page_size,
                                  _ptr(k_pages), _ptr(v_pages), capacity_pages, _ptr(block_table),
                                  max_pages, _ptr(seq_lens), _ptr(needed_pages), _ptr(ws),
                                  ws_bytes, _stream(stream)))
