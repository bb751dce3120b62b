"""Thin Python binding of the GB300 paged GQA decode library (libpaged_decode.so).

Every function here only marshals arguments: it checks the torch tensors'
dtype, device and layout, passes their device pointers and the current CUDA
stream to the C ABI declared in ``include/paged_decode.h``, and raises
:class:`PagedDecodeError` on a non-OK status. All computation runs in the
library's CUDA kernels; there is no fallback. PyTorch provides device memory
and streams only.

Names follow the C ABI: ``pa_reshape_and_cache``, ``pa_decode``,
``quest_update_meta``, ``quest_reshape_and_cache`` (both write steps in one
launch), ``quest_rebuild_meta``, ``quest_select_topk``,
``quest_sparse_decode``; ``pa_decode_multi`` for several query rows per
sequence; the ``*_fp8`` variants for an 8-bit (E4M3) cache; plus the
workspace-size queries and checks.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpaged_decode.so")

PA_OK = 0
_lib = None
_lock = threading.Lock()

__all__ = [
    "PagedDecodeError", "load_library", "pa_status_string", "pa_reshape_and_cache",
    "pa_decode_workspace_size", "pa_decode", "pa_decode_budget", "quest_update_meta", "quest_reshape_and_cache",
    "quest_rebuild_meta",
    "quest_select_workspace_size", "quest_select_topk", "quest_sparse_decode", "quest_sparse_decode_budget",
    "quest_decode_workspace_size", "quest_decode", "quest_decode_fp8",
    "pa_decode_multi_workspace_size", "pa_decode_multi",
    "pa_reshape_and_cache_fp8", "quest_update_meta_fp8", "quest_reshape_and_cache_fp8",
    "quest_rebuild_meta_fp8", "quest_select_topk_fp8", "pa_decode_fp8", "pa_decode_fp8_budget",
    "quest_sparse_decode_fp8",
    "quest_sparse_decode_fp8_budget",
    "pa_reshape_and_cache_fp8_block", "quest_reshape_and_cache_fp8_block", "quest_select_topk_fp8_block",
    "pa_decode_fp8_block", "pa_decode_fp8_block_budget", "quest_sparse_decode_fp8_block", "quest_decode_fp8_block",
    "pa_reshape_and_decode", "quest_reshape_and_decode",
    "pa_workspace_status", "pa_check_metadata", "Workspace",
]


class PagedDecodeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == -4 and _lib is not None:
            detail = f" (cuda error {_lib.pa_last_cuda_error()})"
        super().__init__(f"{fn} failed: {pa_status_string(status)}{detail}")


def load_library(path: Optional[str] = None):
    """Load libpaged_decode.so (built in-tree by ``paged_gqa_decode_reshape_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with "
                              "`python -m paged_gqa_decode_reshape_gb300.build`")
        L = ctypes.CDLL(p)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        L.pa_status_string.argtypes = [i32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_last_cuda_error.argtypes = []
        L.pa_last_cuda_error.restype = i32
        L.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, vp]
        L.pa_reshape_and_cache.restype = i32
        L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        L.pa_decode_workspace_size.restype = sz
        L.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32,
                                vp, sz, vp]
        L.pa_decode.restype = i32
        L.pa_decode_budget.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32,
                                       i32, vp, sz, vp]
        L.pa_decode_budget.restype = i32
        L.quest_update_meta.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i64, vp]
        L.quest_update_meta.restype = i32
        L.quest_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, vp]
        L.quest_reshape_and_cache.restype = i32
        L.quest_rebuild_meta.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64, vp]
        L.quest_rebuild_meta.restype = i32
        L.quest_select_workspace_size.argtypes = [i32, i32, i32]
        L.quest_select_workspace_size.restype = sz
        L.quest_select_topk.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64,
                                        i32, vp, sz, vp]
        L.quest_select_topk.restype = i32
        L.quest_sparse_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                          i32, i64, f32, vp, sz, vp]
        L.quest_sparse_decode.restype = i32
        L.quest_sparse_decode_budget.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                                 i32, i64, f32, i32, vp, sz, vp]
        L.quest_sparse_decode_budget.restype = i32
        L.quest_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.quest_decode_workspace_size.restype = sz
        L.quest_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64,
                                   i32, f32, i32, vp, sz, vp]
        L.quest_decode.restype = i32
        L.quest_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                       i32, i64, i32, f32, i32, vp, sz, vp]
        L.quest_decode_fp8.restype = i32
        L.pa_workspace_status.argtypes = [vp, vp]
        L.pa_workspace_status.restype = i32
        L.pa_check_metadata.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i64, vp]
        L.pa_check_metadata.restype = i32
        L.pa_decode_multi_workspace_size.argtypes = [i32, i32, i32, i32]
        L.pa_decode_multi_workspace_size.restype = sz
        L.pa_decode_multi.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
                                      i64, f32, vp, sz, vp]
        L.pa_decode_multi.restype = i32
        L.pa_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i64, vp]
        L.pa_reshape_and_cache_fp8.restype = i32
        L.quest_update_meta_fp8.argtypes = [vp, vp, vp, vp, i64, vp, i32, i32, i32, i64, vp]
        L.quest_update_meta_fp8.restype = i32
        L.quest_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i32,
                                                  i32, i64, vp]
        L.quest_reshape_and_cache_fp8.restype = i32
        L.quest_rebuild_meta_fp8.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64, vp]
        L.quest_rebuild_meta_fp8.restype = i32
        L.quest_select_topk_fp8.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                            i64, i32, vp, sz, vp]
        L.quest_select_topk_fp8.restype = i32
        L.pa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                    i64, f32, vp, sz, vp]
        L.pa_decode_fp8.restype = i32
        L.quest_sparse_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32,
                                              i32, i32, i32, i64, f32, vp, sz, vp]
        L.quest_sparse_decode_fp8.restype = i32
        L.quest_sparse_decode_fp8_budget.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32,
                                                     i32, i32, i32, i64, f32, i32, vp, sz, vp]
        L.quest_sparse_decode_fp8_budget.restype = i32
        L.pa_reshape_and_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                            i32, i64, f32, vp, sz, vp]
        L.pa_reshape_and_decode.restype = i32
        L.quest_reshape_and_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                               i32, i32, i64, i32, f32, i32, vp, sz, vp]
        L.quest_reshape_and_decode.restype = i32
        L.pa_reshape_and_cache_fp8_block.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i64, vp]
        L.pa_reshape_and_cache_fp8_block.restype = i32
        L.quest_reshape_and_cache_fp8_block.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, i32, i32,
                                                        i32, i64, vp]
        L.quest_reshape_and_cache_fp8_block.restype = i32
        L.quest_select_topk_fp8_block.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                                  i64, i32, vp, sz, vp]
        L.quest_select_topk_fp8_block.restype = i32
        L.pa_decode_fp8_block.argtypes = L.pa_decode_fp8.argtypes
        L.pa_decode_fp8_block.restype = i32
        L.pa_decode_fp8_budget.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                           i64, f32, i32, vp, sz, vp]
        L.pa_decode_fp8_budget.restype = i32
        L.pa_decode_fp8_block_budget.argtypes = L.pa_decode_fp8_budget.argtypes
        L.pa_decode_fp8_block_budget.restype = i32
        L.quest_sparse_decode_fp8_block.argtypes = L.quest_sparse_decode_fp8_budget.argtypes
        L.quest_sparse_decode_fp8_block.restype = i32
        L.quest_decode_fp8_block.argtypes = L.quest_decode_fp8.argtypes
        L.quest_decode_fp8_block.restype = i32
        _lib = L
        return _lib


def pa_status_string(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


# ------------------------------------------------------------------ helpers


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn: str, status: int):
    if status != PA_OK:
        raise PagedDecodeError(fn, status)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


class Workspace:
    """A zero-filled device scratch buffer, grown on demand, per device.

    The decode kernels leave their workspace zeroed after every call, so one
    buffer serves every sequential call on one stream. Calls that may overlap
    in time (several streams) need separate Workspace objects."""

    def __init__(self):
        self._buf = {}

    def get(self, device: torch.device, nbytes: int) -> torch.Tensor:
        key = device.index if device.index is not None else torch.cuda.current_device()
        buf = self._buf.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._buf[key] = buf
        return buf


_default_ws = Workspace()
_default_sel_ws = Workspace()


# --------------------------------------------------------------- entry points


def pa_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    """Scatter this step's K/V rows [T, Hkv, D] into the paged caches [NB, BS, Hkv, D]."""
    L = load_library()
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.bfloat16, 4, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    T = slot_mapping.shape[0]
    if value_cache.shape != key_cache.shape or key.shape != (T, Hkv, D) or value.shape != key.shape:
        raise ValueError("shape mismatch between key/value and the caches")
    _check("pa_reshape_and_cache",
           L.pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                  _ptr(slot_mapping), T, Hkv, D, BS, NB, _stream(dev)))


def pa_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load_library().pa_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim))


def quest_select_workspace_size(batch: int, num_kv_heads: int, max_blocks_per_seq: int) -> int:
    return int(load_library().quest_select_workspace_size(batch, num_kv_heads, max_blocks_per_seq))


def _attention_checks(out, query, key_cache, value_cache, block_tables, context_lens):
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.bfloat16, 4, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = query.shape
    NB, BS, Hkv, D2 = key_cache.shape
    if D != D2 or value_cache.shape != key_cache.shape or out.shape != query.shape:
        raise ValueError("shape mismatch between query/out and the caches")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    return dev, B, Hq, Hkv, D, BS, NB, block_tables.shape[1]


def pa_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
              value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
              scale: float, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dense GQA paged decode attention; writes out [B, Hq, D] (bf16)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks(out, query, key_cache, value_cache,
                                                        block_tables, context_lens)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode",
           L.pa_decode(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                       _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D, BS, NB,
                       float(scale), _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return out


def pa_decode_budget(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                     value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                     scale: float, max_ctas: int, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pa_decode on at most max_ctas CTAs (0: one per SM), leaving the other
    SMs to work on another stream."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks(out, query, key_cache, value_cache,
                                                        block_tables, context_lens)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_budget",
           L.pa_decode_budget(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                              _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D, BS, NB,
                              float(scale), int(max_ctas), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(dev)))
    return out


def quest_sparse_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                        value_cache: torch.Tensor, block_tables: torch.Tensor,
                        context_lens: torch.Tensor, selected: torch.Tensor, scale: float,
                        workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest sparse attention over selected [B, Hkv, topk] logical blocks; writes out."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks(out, query, key_cache, value_cache,
                                                        block_tables, context_lens)
    _need(selected, "selected", torch.int32, 3, dev)
    if selected.shape[:2] != (B, Hkv):
        raise ValueError("selected must be [B, Hkv, topk]")
    topk = selected.shape[2]
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("quest_sparse_decode",
           L.quest_sparse_decode(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                 _ptr(block_tables), MBS, _ptr(context_lens), _ptr(selected), topk,
                                 B, Hq, Hkv, D, BS, NB, float(scale), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(dev)))
    return out


def quest_sparse_decode_budget(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                               value_cache: torch.Tensor, block_tables: torch.Tensor,
                               context_lens: torch.Tensor, selected: torch.Tensor, scale: float,
                               max_ctas: int, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """quest_sparse_decode launching at most max_ctas CTAs (0: the default)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks(out, query, key_cache, value_cache,
                                                        block_tables, context_lens)
    _need(selected, "selected", torch.int32, 3, dev)
    if selected.shape[:2] != (B, Hkv):
        raise ValueError("selected must be [B, Hkv, topk]")
    topk = selected.shape[2]
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("quest_sparse_decode_budget",
           L.quest_sparse_decode_budget(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                        _ptr(block_tables), MBS, _ptr(context_lens), _ptr(selected), topk,
                                        B, Hq, Hkv, D, BS, NB, float(scale), int(max_ctas), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(dev)))
    return out


def quest_update_meta(kmin: torch.Tensor, kmax: torch.Tensor, key: torch.Tensor,
                      slot_mapping: torch.Tensor, block_size: int) -> None:
    """Fold this step's new keys into the per-block min/max metadata [NB, Hkv, D]."""
    L = load_library()
    _need(kmin, "kmin", torch.bfloat16, 3)
    dev = kmin.device
    _need(kmax, "kmax", torch.bfloat16, 3, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, Hkv, D = kmin.shape
    T = slot_mapping.shape[0]
    if kmax.shape != kmin.shape or key.shape != (T, Hkv, D):
        raise ValueError("shape mismatch between key and the metadata")
    _check("quest_update_meta",
           L.quest_update_meta(_ptr(kmin), _ptr(kmax), _ptr(key), _ptr(slot_mapping), T, Hkv, D,
                               int(block_size), NB, _stream(dev)))


def quest_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, kmin: torch.Tensor, kmax: torch.Tensor,
                            slot_mapping: torch.Tensor) -> None:
    """The write path in one launch: pa_reshape_and_cache then quest_update_meta."""
    L = load_library()
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.bfloat16, 4, dev)
    _need(kmin, "kmin", torch.bfloat16, 3, dev)
    _need(kmax, "kmax", torch.bfloat16, 3, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    T = slot_mapping.shape[0]
    if (value_cache.shape != key_cache.shape or key.shape != (T, Hkv, D) or value.shape != key.shape
            or kmin.shape != (NB, Hkv, D) or kmax.shape != kmin.shape):
        raise ValueError("shape mismatch between key/value, the caches and the metadata")
    _check("quest_reshape_and_cache",
           L.quest_reshape_and_cache(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                     _ptr(kmin), _ptr(kmax), _ptr(slot_mapping), T, Hkv, D, BS, NB,
                                     _stream(dev)))


def quest_rebuild_meta(kmin: torch.Tensor, kmax: torch.Tensor, key_cache: torch.Tensor,
                       block_tables: torch.Tensor, context_lens: torch.Tensor) -> None:
    """Recompute the metadata of every block the sequences use from the cache."""
    L = load_library()
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    dev = key_cache.device
    _need(kmin, "kmin", torch.bfloat16, 3, dev)
    _need(kmax, "kmax", torch.bfloat16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    B, MBS = block_tables.shape
    if kmin.shape != (NB, Hkv, D) or kmax.shape != kmin.shape:
        raise ValueError("metadata must be [NB, Hkv, D]")
    _check("quest_rebuild_meta",
           L.quest_rebuild_meta(_ptr(kmin), _ptr(kmax), _ptr(key_cache), _ptr(block_tables), MBS,
                                _ptr(context_lens), B, Hkv, D, BS, NB, _stream(dev)))


def quest_select_topk(selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                      kmax: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                      block_size: int, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Score every logical block and write the top-K per (b, kvh) into selected [B, Hkv, topk]."""
    L = load_library()
    _need(kmin, "kmin", torch.bfloat16, 3)
    dev = kmin.device
    _need(kmax, "kmax", torch.bfloat16, 3, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(selected, "selected", torch.int32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = query.shape
    NB, Hkv, D2 = kmin.shape
    MBS = block_tables.shape[1]
    if D != D2 or selected.shape[:2] != (B, Hkv):
        raise ValueError("shape mismatch in quest_select_topk")
    topk = selected.shape[2]
    need = quest_select_workspace_size(B, Hkv, MBS)
    ws = workspace if workspace is not None else _default_sel_ws.get(dev, need)
    _check("quest_select_topk",
           L.quest_select_topk(_ptr(selected), _ptr(query), _ptr(kmin), _ptr(kmax),
                               _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                               int(block_size), NB, topk, _ptr(ws), ws.numel() * ws.element_size(),
                               _stream(dev)))
    return selected


def pa_workspace_status(workspace: torch.Tensor) -> int:
    """Status word of a decode workspace (synchronises the current stream)."""
    return int(load_library().pa_workspace_status(_ptr(workspace), _stream(workspace.device)))


def default_workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """The binding's shared decode workspace for `device` (zero-filled, >= nbytes)."""
    return _default_ws.get(device, nbytes)


def pa_check_metadata(slot_mapping: Optional[torch.Tensor], block_tables: Optional[torch.Tensor],
                      context_lens: Optional[torch.Tensor], block_size: int, num_blocks: int,
                      device: Optional[torch.device] = None) -> list:
    """Count malformed metadata on the device: [slots past the pool, bad context_lens,
    table entries outside the pool, repeated slots]."""
    L = load_library()
    ref = next(t for t in (slot_mapping, block_tables, context_lens) if t is not None)
    dev = device or ref.device
    counts = torch.empty(4, dtype=torch.int32, device=dev)
    T = slot_mapping.shape[0] if slot_mapping is not None else 0
    B = context_lens.shape[0] if context_lens is not None else 0
    MBS = block_tables.shape[1] if block_tables is not None else 0
    _check("pa_check_metadata",
           L.pa_check_metadata(_ptr(counts), _ptr(slot_mapping), T, _ptr(block_tables), MBS,
                               _ptr(context_lens), B, int(block_size), int(num_blocks), _stream(dev)))
    return counts.cpu().tolist()


# ------------------------------------------------- 8-bit (E4M3) KV cache
#
# Caches and metadata are uint8 tensors holding E4M3 codes; k_scale / v_scale
# are float32 [Hkv] tensors on the same device (see include/paged_decode.h).
# key_cache is [NB, BS, Hkv, D]; value_cache is [NB, Hkv, D, BS] (per block
# and KV head a dim-by-token byte matrix, tokens of a row in the order
# 0 1 8 9 2 3 10 11 ...), BS = 16.


def _scales(k_scale, v_scale, Hkv, dev):
    _need(k_scale, "k_scale", torch.float32, 1, dev)
    if v_scale is not None:
        _need(v_scale, "v_scale", torch.float32, 1, dev)
    if k_scale.shape[0] != Hkv or (v_scale is not None and v_scale.shape[0] != Hkv):
        raise ValueError("scales must be [num_kv_heads]")


def pa_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                             value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                             k_scale: torch.Tensor, v_scale: torch.Tensor) -> None:
    """Quantise this step's K/V rows [T, Hkv, D] (bf16) into 8-bit caches [NB, BS, Hkv, D]."""
    L = load_library()
    _need(key_cache, "key_cache", torch.uint8, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.uint8, 4, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    T = slot_mapping.shape[0]
    if value_cache.shape != (NB, Hkv, D, BS) or key.shape != (T, Hkv, D) or value.shape != key.shape:
        raise ValueError("shape mismatch between key/value and the caches")
    _scales(k_scale, v_scale, Hkv, dev)
    _check("pa_reshape_and_cache_fp8",
           L.pa_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                      _ptr(slot_mapping), T, _ptr(k_scale), _ptr(v_scale), Hkv, D, BS,
                                      NB, _stream(dev)))


def quest_update_meta_fp8(kmin: torch.Tensor, kmax: torch.Tensor, key: torch.Tensor,
                          slot_mapping: torch.Tensor, k_scale: torch.Tensor, block_size: int) -> None:
    """Fold this step's quantised keys into the 8-bit metadata [NB, Hkv, D]."""
    L = load_library()
    _need(kmin, "kmin", torch.uint8, 3)
    dev = kmin.device
    _need(kmax, "kmax", torch.uint8, 3, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, Hkv, D = kmin.shape
    T = slot_mapping.shape[0]
    if kmax.shape != kmin.shape or key.shape != (T, Hkv, D):
        raise ValueError("shape mismatch between key and the metadata")
    _scales(k_scale, None, Hkv, dev)
    _check("quest_update_meta_fp8",
           L.quest_update_meta_fp8(_ptr(kmin), _ptr(kmax), _ptr(key), _ptr(slot_mapping), T,
                                   _ptr(k_scale), Hkv, D, int(block_size), NB, _stream(dev)))


def quest_reshape_and_cache_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                                value_cache: torch.Tensor, kmin: torch.Tensor, kmax: torch.Tensor,
                                slot_mapping: torch.Tensor, k_scale: torch.Tensor,
                                v_scale: torch.Tensor) -> None:
    """The 8-bit write path in one launch: pa_reshape_and_cache_fp8 then quest_update_meta_fp8."""
    L = load_library()
    _need(key_cache, "key_cache", torch.uint8, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.uint8, 4, dev)
    _need(kmin, "kmin", torch.uint8, 3, dev)
    _need(kmax, "kmax", torch.uint8, 3, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    T = slot_mapping.shape[0]
    if (value_cache.shape != (NB, Hkv, D, BS) or key.shape != (T, Hkv, D) or value.shape != key.shape
            or kmin.shape != (NB, Hkv, D) or kmax.shape != kmin.shape):
        raise ValueError("shape mismatch between key/value, the caches and the metadata")
    _scales(k_scale, v_scale, Hkv, dev)
    _check("quest_reshape_and_cache_fp8",
           L.quest_reshape_and_cache_fp8(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                         _ptr(kmin), _ptr(kmax), _ptr(slot_mapping), T, _ptr(k_scale),
                                         _ptr(v_scale), Hkv, D, BS, NB, _stream(dev)))


def quest_rebuild_meta_fp8(kmin: torch.Tensor, kmax: torch.Tensor, key_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor) -> None:
    """Recompute the 8-bit metadata of every block the sequences use from the 8-bit cache."""
    L = load_library()
    _need(key_cache, "key_cache", torch.uint8, 4)
    dev = key_cache.device
    _need(kmin, "kmin", torch.uint8, 3, dev)
    _need(kmax, "kmax", torch.uint8, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    B, MBS = block_tables.shape
    if kmin.shape != (NB, Hkv, D) or kmax.shape != kmin.shape:
        raise ValueError("metadata must be [NB, Hkv, D]")
    _check("quest_rebuild_meta_fp8",
           L.quest_rebuild_meta_fp8(_ptr(kmin), _ptr(kmax), _ptr(key_cache), _ptr(block_tables), MBS,
                                    _ptr(context_lens), B, Hkv, D, BS, NB, _stream(dev)))


def quest_select_topk_fp8(selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                          kmax: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                          block_size: int, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest selection on 8-bit metadata; writes selected [B, Hkv, topk]."""
    L = load_library()
    _need(kmin, "kmin", torch.uint8, 3)
    dev = kmin.device
    _need(kmax, "kmax", torch.uint8, 3, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(selected, "selected", torch.int32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = query.shape
    NB, Hkv, D2 = kmin.shape
    MBS = block_tables.shape[1]
    if D != D2 or selected.shape[:2] != (B, Hkv):
        raise ValueError("shape mismatch in quest_select_topk_fp8")
    topk = selected.shape[2]
    need = quest_select_workspace_size(B, Hkv, MBS)
    ws = workspace if workspace is not None else _default_sel_ws.get(dev, need)
    _check("quest_select_topk_fp8",
           L.quest_select_topk_fp8(_ptr(selected), _ptr(query), _ptr(kmin), _ptr(kmax),
                                   _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                                   int(block_size), NB, topk, _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(dev)))
    return selected


def _attention_checks_fp8(out, query, key_cache, value_cache, block_tables, context_lens,
                          k_scale, v_scale, per_block=False):
    _need(key_cache, "key_cache", torch.uint8, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.uint8, 4, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = query.shape
    NB, BS, Hkv, D2 = key_cache.shape
    if D != D2 or value_cache.shape != (NB, Hkv, D, BS) or out.shape != query.shape:
        raise ValueError("shape mismatch between query/out and the caches")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens batch mismatch")
    if per_block:
        _block_scales(k_scale, v_scale, NB, Hkv, dev)
    else:
        _scales(k_scale, v_scale, Hkv, dev)
    return dev, B, Hq, Hkv, D, BS, NB, block_tables.shape[1]


def pa_decode_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                  value_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                  workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dense GQA paged decode attention over 8-bit caches; writes out [B, Hq, D] (bf16)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache,
                                                            block_tables, context_lens, k_scale, v_scale)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_fp8",
           L.pa_decode_fp8(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(k_scale),
                           _ptr(v_scale), _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                           BS, NB, float(scale), _ptr(ws), ws.numel() * ws.element_size(),
                           _stream(dev)))
    return out


def pa_decode_fp8_budget(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                         block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, max_ctas: int,
                         workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pa_decode_fp8 on at most max_ctas CTAs (0: one per SM)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache,
                                                            block_tables, context_lens, k_scale, v_scale)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_fp8_budget",
           L.pa_decode_fp8_budget(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(k_scale),
                                  _ptr(v_scale), _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                                  BS, NB, float(scale), int(max_ctas), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(dev)))
    return out


def quest_sparse_decode_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor,
                            selected: torch.Tensor, scale: float,
                            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest sparse attention over 8-bit caches and the selected [B, Hkv, topk] blocks."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache,
                                                            block_tables, context_lens, k_scale, v_scale)
    _need(selected, "selected", torch.int32, 3, dev)
    if selected.shape[:2] != (B, Hkv):
        raise ValueError("selected must be [B, Hkv, topk]")
    topk = selected.shape[2]
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("quest_sparse_decode_fp8",
           L.quest_sparse_decode_fp8(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), MBS,
                                     _ptr(context_lens), _ptr(selected), topk, B, Hq, Hkv, D, BS, NB,
                                     float(scale), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(dev)))
    return out


def quest_sparse_decode_fp8_budget(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                                   block_tables: torch.Tensor, context_lens: torch.Tensor,
                                   selected: torch.Tensor, scale: float, max_ctas: int,
                                   workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """quest_sparse_decode_fp8 launching at most max_ctas CTAs (0: the default)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache,
                                                            block_tables, context_lens, k_scale, v_scale)
    _need(selected, "selected", torch.int32, 3, dev)
    if selected.shape[:2] != (B, Hkv):
        raise ValueError("selected must be [B, Hkv, topk]")
    topk = selected.shape[2]
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("quest_sparse_decode_fp8_budget",
           L.quest_sparse_decode_fp8_budget(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                            _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), MBS,
                                            _ptr(context_lens), _ptr(selected), topk, B, Hq, Hkv, D, BS, NB,
                                            float(scale), int(max_ctas), _ptr(ws), ws.numel() * ws.element_size(),
                                            _stream(dev)))
    return out


# ------------------------------------------------------ multi-token rows


def pa_decode_multi_workspace_size(total_q: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load_library().pa_decode_multi_workspace_size(total_q, num_q_heads, num_kv_heads, head_dim))


def pa_decode_multi(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                    value_cache: torch.Tensor, block_tables: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    context_lens: torch.Tensor, scale: float,
                    workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode attention of multi-token query rows [total_q, Hq, D] with right-aligned
    causal masks; cu_seqlens_q [B+1] int32 gives each sequence's rows."""
    L = load_library()
    _need(key_cache, "key_cache", torch.bfloat16, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.bfloat16, 4, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(out, "out", torch.bfloat16, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    total_q, Hq, D = query.shape
    NB, BS, Hkv, D2 = key_cache.shape
    B = context_lens.shape[0]
    if D != D2 or value_cache.shape != key_cache.shape or out.shape != query.shape:
        raise ValueError("shape mismatch between query/out and the caches")
    if block_tables.shape[0] != B or cu_seqlens_q.shape[0] != B + 1:
        raise ValueError("block_tables / cu_seqlens_q / context_lens batch mismatch")
    need = pa_decode_multi_workspace_size(max(total_q, 1), Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_multi",
           L.pa_decode_multi(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                             _ptr(block_tables), block_tables.shape[1], _ptr(cu_seqlens_q),
                             _ptr(context_lens), B, total_q, Hq, Hkv, D, BS, NB, float(scale), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(dev)))
    return out


def quest_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                max_blocks_per_seq: int) -> int:
    return int(load_library().quest_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                          max_blocks_per_seq))


def _quest_decode(fn, what, out, selected, query, kmin, kmax, key_cache, value_cache, block_tables,
                  context_lens, topk, scale, max_ctas, workspace, scales, checks):
    dev, B, Hq, Hkv, D, BS, NB, MBS = checks
    _need(selected, "selected", torch.int32, 3, dev)
    if tuple(selected.shape) != (B, Hkv, int(topk)):
        raise ValueError("selected must be [B, Hkv, topk]")
    if tuple(kmin.shape) != (NB, Hkv, D) or tuple(kmax.shape) != (NB, Hkv, D):
        raise ValueError("kmin / kmax must be [NB, Hkv, D]")
    need = quest_decode_workspace_size(B, Hq, Hkv, D, MBS)
    if need == 0:
        raise PagedDecodeError(f"{what}: unsupported shape")
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check(what, fn(_ptr(out), _ptr(selected), _ptr(query), _ptr(kmin), _ptr(kmax), _ptr(key_cache),
                    _ptr(value_cache), *scales, _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D, BS,
                    NB, int(topk), float(scale), int(max_ctas), _ptr(ws), ws.numel() * ws.element_size(),
                    _stream(dev)))
    return out


def quest_decode(out: torch.Tensor, selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                 kmax: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, topk: int, scale: float,
                 max_ctas: int = 0, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest scores, then top-K and sparse attention in one launch; writes selected and out."""
    L = load_library()
    checks = _attention_checks(out, query, key_cache, value_cache, block_tables, context_lens)
    _need(kmin, "kmin", torch.bfloat16, 3, checks[0])
    _need(kmax, "kmax", torch.bfloat16, 3, checks[0])
    return _quest_decode(L.quest_decode, "quest_decode", out, selected, query, kmin, kmax, key_cache,
                         value_cache, block_tables, context_lens, topk, scale, max_ctas, workspace, (), checks)


def quest_decode_fp8(out: torch.Tensor, selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                     kmax: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                     k_scale: torch.Tensor, v_scale: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, topk: int, scale: float, max_ctas: int = 0,
                     workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """quest_decode over 8-bit caches (E4M3 metadata, K and V codes with per-KV-head scales)."""
    L = load_library()
    checks = _attention_checks_fp8(out, query, key_cache, value_cache, block_tables, context_lens, k_scale,
                                   v_scale)
    _need(kmin, "kmin", torch.uint8, 3, checks[0])
    _need(kmax, "kmax", torch.uint8, 3, checks[0])
    return _quest_decode(L.quest_decode_fp8, "quest_decode_fp8", out, selected, query, kmin, kmax, key_cache,
                         value_cache, block_tables, context_lens, topk, scale, max_ctas, workspace,
                         (_ptr(k_scale), _ptr(v_scale)), checks)


# ------------------------------------- 8-bit cache with per-block scales


def _block_scales(k_bscale, v_bscale, NB, Hkv, dev):
    _need(k_bscale, "k_bscale", torch.float32, 2, dev)
    if v_bscale is not None:
        _need(v_bscale, "v_bscale", torch.float32, 2, dev)
    if tuple(k_bscale.shape) != (NB, Hkv) or (v_bscale is not None and tuple(v_bscale.shape) != (NB, Hkv)):
        raise ValueError("per-block scales must be [num_blocks, num_kv_heads]")


def _write_fp8_block(fn, what, key, value, key_cache, value_cache, slot_mapping, k_bscale, v_bscale,
                     meta=None):
    _need(key_cache, "key_cache", torch.uint8, 4)
    dev = key_cache.device
    _need(value_cache, "value_cache", torch.uint8, 4, dev)
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    NB, BS, Hkv, D = key_cache.shape
    T = slot_mapping.shape[0]
    if value_cache.shape != (NB, Hkv, D, BS) or key.shape != (T, Hkv, D) or value.shape != key.shape:
        raise ValueError("shape mismatch between key/value and the caches")
    _block_scales(k_bscale, v_bscale, NB, Hkv, dev)
    m = ()
    if meta is not None:
        for t, n in zip(meta, ("kmin", "kmax")):
            _need(t, n, torch.uint8, 3, dev)
            if tuple(t.shape) != (NB, Hkv, D):
                raise ValueError("metadata must be [NB, Hkv, D]")
        m = (_ptr(meta[0]), _ptr(meta[1]))
    _check(what, fn(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), *m, _ptr(slot_mapping), T,
                    _ptr(k_bscale), _ptr(v_bscale), Hkv, D, BS, NB, _stream(dev)))


def pa_reshape_and_cache_fp8_block(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                                   k_bscale: torch.Tensor, v_bscale: torch.Tensor) -> None:
    """Quantise this step's K/V rows into 8-bit caches with per-block power-of-two scales
    k_bscale / v_bscale [NB, Hkv] (fp32, updated in place; 0 marks an empty block)."""
    L = load_library()
    _write_fp8_block(L.pa_reshape_and_cache_fp8_block, "pa_reshape_and_cache_fp8_block", key, value,
                     key_cache, value_cache, slot_mapping, k_bscale, v_bscale)


def quest_reshape_and_cache_fp8_block(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                                      value_cache: torch.Tensor, kmin: torch.Tensor, kmax: torch.Tensor,
                                      slot_mapping: torch.Tensor, k_bscale: torch.Tensor,
                                      v_bscale: torch.Tensor) -> None:
    """pa_reshape_and_cache_fp8_block and the Quest metadata update in one launch."""
    L = load_library()
    _write_fp8_block(L.quest_reshape_and_cache_fp8_block, "quest_reshape_and_cache_fp8_block", key, value,
                     key_cache, value_cache, slot_mapping, k_bscale, v_bscale, meta=(kmin, kmax))


def quest_select_topk_fp8_block(selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                                kmax: torch.Tensor, k_bscale: torch.Tensor, block_tables: torch.Tensor,
                                context_lens: torch.Tensor, block_size: int,
                                workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest selection on 8-bit metadata of a cache with per-block scales."""
    L = load_library()
    _need(kmin, "kmin", torch.uint8, 3)
    dev = kmin.device
    _need(kmax, "kmax", torch.uint8, 3, dev)
    _need(query, "query", torch.bfloat16, 3, dev)
    _need(selected, "selected", torch.int32, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    B, Hq, D = query.shape
    NB, Hkv, D2 = kmin.shape
    MBS = block_tables.shape[1]
    if D != D2 or selected.shape[:2] != (B, Hkv):
        raise ValueError("shape mismatch in quest_select_topk_fp8_block")
    _block_scales(k_bscale, None, NB, Hkv, dev)
    topk = selected.shape[2]
    need = quest_select_workspace_size(B, Hkv, MBS)
    ws = workspace if workspace is not None else _default_sel_ws.get(dev, need)
    _check("quest_select_topk_fp8_block",
           L.quest_select_topk_fp8_block(_ptr(selected), _ptr(query), _ptr(kmin), _ptr(kmax), _ptr(k_bscale),
                                         _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                                         int(block_size), NB, topk, _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(dev)))
    return selected


def pa_decode_fp8_block(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                        value_cache: torch.Tensor, k_bscale: torch.Tensor, v_bscale: torch.Tensor,
                        block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                        workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dense GQA paged decode over 8-bit caches with per-block scales [NB, Hkv]."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache, block_tables,
                                                            context_lens, k_bscale, v_bscale, per_block=True)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_fp8_block",
           L.pa_decode_fp8_block(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(k_bscale),
                                 _ptr(v_bscale), _ptr(block_tables), MBS, _ptr(context_lens), B, Hq, Hkv, D,
                                 BS, NB, float(scale), _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return out


def pa_decode_fp8_block_budget(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                               value_cache: torch.Tensor, k_bscale: torch.Tensor, v_bscale: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                               max_ctas: int, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """pa_decode_fp8_block on at most max_ctas CTAs (0: one per SM)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache, block_tables,
                                                            context_lens, k_bscale, v_bscale, per_block=True)
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_decode_fp8_block_budget",
           L.pa_decode_fp8_block_budget(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                        _ptr(k_bscale), _ptr(v_bscale), _ptr(block_tables), MBS,
                                        _ptr(context_lens), B, Hq, Hkv, D, BS, NB, float(scale), int(max_ctas),
                                        _ptr(ws), ws.numel() * ws.element_size(), _stream(dev)))
    return out


def quest_sparse_decode_fp8_block(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                  value_cache: torch.Tensor, k_bscale: torch.Tensor, v_bscale: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  selected: torch.Tensor, scale: float, max_ctas: int = 0,
                                  workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quest sparse attention over 8-bit caches with per-block scales (max_ctas 0: the default)."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks_fp8(out, query, key_cache, value_cache, block_tables,
                                                            context_lens, k_bscale, v_bscale, per_block=True)
    _need(selected, "selected", torch.int32, 3, dev)
    if selected.shape[:2] != (B, Hkv):
        raise ValueError("selected must be [B, Hkv, topk]")
    topk = selected.shape[2]
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("quest_sparse_decode_fp8_block",
           L.quest_sparse_decode_fp8_block(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache),
                                           _ptr(k_bscale), _ptr(v_bscale), _ptr(block_tables), MBS,
                                           _ptr(context_lens), _ptr(selected), topk, B, Hq, Hkv, D, BS, NB,
                                           float(scale), int(max_ctas), _ptr(ws), ws.numel() * ws.element_size(),
                                           _stream(dev)))
    return out


def quest_decode_fp8_block(out: torch.Tensor, selected: torch.Tensor, query: torch.Tensor, kmin: torch.Tensor,
                           kmax: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                           k_bscale: torch.Tensor, v_bscale: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, topk: int, scale: float, max_ctas: int = 0,
                           workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """quest_decode over 8-bit caches with per-block scales."""
    L = load_library()
    checks = _attention_checks_fp8(out, query, key_cache, value_cache, block_tables, context_lens, k_bscale,
                                   v_bscale, per_block=True)
    _need(kmin, "kmin", torch.uint8, 3, checks[0])
    _need(kmax, "kmax", torch.uint8, 3, checks[0])
    return _quest_decode(L.quest_decode_fp8_block, "quest_decode_fp8_block", out, selected, query, kmin, kmax,
                         key_cache, value_cache, block_tables, context_lens, topk, scale, max_ctas, workspace,
                         (_ptr(k_bscale), _ptr(v_bscale)), checks)


# ------------------------------------- the step's write folded into decode


def _step_tokens(key, value, slot_mapping, B, Hkv, D, dev):
    _need(key, "key", torch.bfloat16, 3, dev)
    _need(value, "value", torch.bfloat16, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, dev)
    if tuple(key.shape) != (B, Hkv, D) or value.shape != key.shape or slot_mapping.shape[0] != B:
        raise ValueError("key / value must be [B, Hkv, D] and slot_mapping [B]: one new token per sequence")


def pa_reshape_and_decode(out: torch.Tensor, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                          slot_mapping: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                          block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                          kmin: Optional[torch.Tensor] = None, kmax: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Each sequence's new token written at position ctx_b - 1 (when slot_mapping[b] is that
    slot; also into kmin / kmax when given), then dense decode, in one launch."""
    L = load_library()
    dev, B, Hq, Hkv, D, BS, NB, MBS = _attention_checks(out, query, key_cache, value_cache, block_tables,
                                                        context_lens)
    _step_tokens(key, value, slot_mapping, B, Hkv, D, dev)
    if (kmin is None) != (kmax is None):
        raise ValueError("kmin and kmax go together")
    if kmin is not None:
        for t, n in ((kmin, "kmin"), (kmax, "kmax")):
            _need(t, n, torch.bfloat16, 3, dev)
            if tuple(t.shape) != (NB, Hkv, D):
                raise ValueError("kmin / kmax must be [NB, Hkv, D]")
    need = pa_decode_workspace_size(B, Hq, Hkv, D)
    ws = workspace if workspace is not None else _default_ws.get(dev, need)
    _check("pa_reshape_and_decode",
           L.pa_reshape_and_decode(_ptr(out), _ptr(query), _ptr(key), _ptr(value), _ptr(slot_mapping),
                                   _ptr(key_cache), _ptr(value_cache), _ptr(kmin), _ptr(kmax), _ptr(block_tables),
                                   MBS, _ptr(context_lens), B, Hq, Hkv, D, BS, NB, float(scale), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(dev)))
    return out


def quest_reshape_and_decode(out: torch.Tensor, selected: torch.Tensor, query: torch.Tensor, key: torch.Tensor,
                             value: torch.Tensor, slot_mapping: torch.Tensor, kmin: torch.Tensor,
                             kmax: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor, topk: int, scale: float,
                             max_ctas: int = 0, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The step's write and metadata update folded into the score launch, then the
    fused top-K and sparse decode: quest_reshape_and_cache + quest_decode in two launches."""
    L = load_library()
    checks = _attention_checks(out, query, key_cache, value_cache, block_tables, context_lens)
    dev, B, Hq, Hkv, D = checks[:5]
    _step_tokens(key, value, slot_mapping, B, Hkv, D, dev)
    _need(kmin, "kmin", torch.bfloat16, 3, dev)
    _need(kmax, "kmax", torch.bfloat16, 3, dev)
    fn = lambda *a: L.quest_reshape_and_decode(a[0], a[1], a[2], _ptr(key), _ptr(value), _ptr(slot_mapping),
                                               *a[3:])
    return _quest_decode(fn, "quest_reshape_and_decode", out, selected, query, kmin, kmax, key_cache,
                         value_cache, block_tables, context_lens, topk, scale, max_ctas, workspace, (), checks)
