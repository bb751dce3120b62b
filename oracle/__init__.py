"""CPU oracle for the paged decode path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded C implementation (``oracle.c``) of what the
path computes, loaded with ctypes. It is the checker the CUDA library is
compared against and shares no code with it. Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg (and its
``--impl reference`` arm) may import this package; the product path never does.

Every function takes and returns host numpy arrays; bf16 data is carried as
``uint16`` bit patterns. Attention outputs are float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    """Compile a C oracle source into the shared library ``out`` (gcc, no FMA contraction)."""
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def load(path: str):
    """Load a compiled oracle library and declare the signatures of its entry points."""
    L = ctypes.CDLL(path)
    vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    L.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64]
    L.oracle_reshape_and_cache.restype = i64
    L.oracle_quest_update_meta.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i64]
    L.oracle_quest_update_meta.restype = i64
    L.oracle_quest_rebuild_meta.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64]
    L.oracle_quest_rebuild_meta.restype = i32
    att = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f64]
    L.oracle_paged_attention.argtypes = att + [vp, i64]
    L.oracle_paged_attention.restype = i32
    L.oracle_paged_attention_online.argtypes = att + [i64]
    L.oracle_paged_attention_online.restype = i32
    L.oracle_paged_attention_split.argtypes = att + [i32]
    L.oracle_paged_attention_split.restype = i32
    L.oracle_sparse_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32,
                                          i32, i32, i32, i32, i32, i64, f64, vp, i64]
    L.oracle_sparse_attention.restype = i32
    score = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64]
    L.oracle_quest_scores_kernel_order.argtypes = score
    L.oracle_quest_scores_kernel_order.restype = i32
    L.oracle_quest_scores_plain.argtypes = [vp] + score
    L.oracle_quest_scores_plain.restype = i32
    L.oracle_quest_scores_plain_fp8.argtypes = [vp] + score
    L.oracle_quest_scores_plain_fp8.restype = i32
    L.oracle_quest_topk.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32]
    L.oracle_quest_topk.restype = i32
    L.oracle_quest_topk_f64.argtypes = [vp, vp, i32, vp, i32, i32, i32, i32]
    L.oracle_quest_topk_f64.restype = i32
    L.oracle_e4m3_encode_array.argtypes = [vp, vp, i64]
    L.oracle_e4m3_encode_array.restype = None
    L.oracle_e4m3_decode_array.argtypes = [vp, vp, i64]
    L.oracle_e4m3_decode_array.restype = None
    L.oracle_reshape_and_cache_fp8.argtypes = [vp, vp, vp, vp, vp, i64, vp, vp, i32, i32, i32, i64]
    L.oracle_reshape_and_cache_fp8.restype = i64
    L.oracle_quest_update_meta_fp8.argtypes = [vp, vp, vp, vp, i64, vp, i32, i32, i32, i64]
    L.oracle_quest_update_meta_fp8.restype = i64
    L.oracle_quest_rebuild_meta_fp8.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64]
    L.oracle_quest_rebuild_meta_fp8.restype = i32
    L.oracle_attention_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32,
                                       i32, i32, i32, i32, i32, i64, f64, vp, i64]
    L.oracle_attention_fp8.restype = i32
    L.oracle_quest_scores_kernel_order_fp8.argtypes = score
    L.oracle_quest_scores_kernel_order_fp8.restype = i32
    L.oracle_reshape_and_cache_fp8_block.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                                     i64]
    L.oracle_reshape_and_cache_fp8_block.restype = i64
    L.oracle_attention_fp8_block.argtypes = L.oracle_attention_fp8.argtypes
    L.oracle_attention_fp8_block.restype = i32
    bscore = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64]
    L.oracle_quest_scores_kernel_order_fp8_block.argtypes = bscore
    L.oracle_quest_scores_kernel_order_fp8_block.restype = i32
    L.oracle_quest_scores_plain_fp8_block.argtypes = [vp] + bscore
    L.oracle_quest_scores_plain_fp8_block.restype = i32
    L.oracle_paged_attention_multi.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32,
                                               i32, i32, i32, i64, f64, vp, i64]
    L.oracle_paged_attention_multi.restype = i32
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc: int, what: str):
    if rc == -1:
        raise ValueError(f"oracle {what}: block table entry outside the pool")
    if rc == -2:
        raise ValueError(f"oracle {what}: invalid sizes")
    if rc != 0:
        raise RuntimeError(f"oracle {what}: status {rc}")


# ----------------------------------------------------------------- cache


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping) -> int:
    """Scatter new K/V rows into the caches IN PLACE; returns #out-of-pool slots."""
    assert key_cache.dtype == np.uint16 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.uint16 and value_cache.flags.c_contiguous
    NB, BS, Hkv, D = key_cache.shape
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    slots = _c(slot_mapping, np.int64)
    return int(lib().oracle_reshape_and_cache(_p(key), _p(value), _p(key_cache), _p(value_cache),
                                              _p(slots), slots.shape[0], Hkv, D, BS, NB))


def quest_update_meta(kmin, kmax, key, slot_mapping, BS: int) -> int:
    """Incremental Quest metadata update IN PLACE; returns #out-of-pool slots."""
    assert kmin.dtype == np.uint16 and kmin.flags.c_contiguous
    assert kmax.dtype == np.uint16 and kmax.flags.c_contiguous
    NB, Hkv, D = kmin.shape
    key = _c(key, np.uint16)
    slots = _c(slot_mapping, np.int64)
    return int(lib().oracle_quest_update_meta(_p(kmin), _p(kmax), _p(key), _p(slots),
                                              slots.shape[0], Hkv, D, BS, NB))


def quest_rebuild_meta(key_cache, block_tables, context_lens, kmin=None, kmax=None):
    """Metadata of every block a sequence uses, from the cache. Returns (kmin, kmax).

    Blocks no sequence uses keep the values passed in (zeros by default)."""
    NB, BS, Hkv, D = key_cache.shape
    if kmin is None:
        kmin = np.zeros((NB, Hkv, D), dtype=np.uint16)
    if kmax is None:
        kmax = np.zeros((NB, Hkv, D), dtype=np.uint16)
    kc = _c(key_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    rc = lib().oracle_quest_rebuild_meta(_p(kmin), _p(kmax), _p(kc), _p(bt), bt.shape[1], _p(ctx),
                                         bt.shape[0], Hkv, D, BS, NB)
    _check(rc, "quest_rebuild_meta")
    return kmin, kmax


# ------------------------------------------------------------- attention


def _att_args(q, key_cache, value_cache, block_tables, context_lens):
    q = _c(q, np.uint16)
    kc = _c(key_cache, np.uint16)
    vc = _c(value_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, BS, Hkv, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape and bt.shape[0] == B and ctx.shape == (B,)
    return q, kc, vc, bt, ctx, B, Hq, Hkv, D, BS, NB


def _rows_arg(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
    return r, r.shape[0]


def paged_attention(q, key_cache, value_cache, block_tables, context_lens, scale, rows=None):
    """Dense GQA paged decode attention, two-pass softmax in fp64.

    Returns [B, Hq, D] float64, or [len(rows), D] for the listed (b, h) pairs."""
    q, kc, vc, bt, ctx, B, Hq, Hkv, D, BS, NB = _att_args(q, key_cache, value_cache,
                                                          block_tables, context_lens)
    r, nr = _rows_arg(rows)
    out = np.zeros((nr, D) if r is not None else (B, Hq, D), dtype=np.float64)
    rc = lib().oracle_paged_attention(_p(out), _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(ctx),
                                      B, Hq, Hkv, D, BS, NB, float(scale), _p(r), nr)
    _check(rc, "paged_attention")
    return out


def paged_attention_online(q, key_cache, value_cache, block_tables, context_lens, scale, chunk):
    """Dense attention via the online-softmax recurrence (``chunk`` tokens per update)."""
    q, kc, vc, bt, ctx, B, Hq, Hkv, D, BS, NB = _att_args(q, key_cache, value_cache,
                                                          block_tables, context_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = lib().oracle_paged_attention_online(_p(out), _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1],
                                             _p(ctx), B, Hq, Hkv, D, BS, NB, float(scale), int(chunk))
    _check(rc, "paged_attention_online")
    return out


def paged_attention_split(q, key_cache, value_cache, block_tables, context_lens, scale, num_splits):
    """Dense attention via split-KV partials and their log-sum-exp combine."""
    q, kc, vc, bt, ctx, B, Hq, Hkv, D, BS, NB = _att_args(q, key_cache, value_cache,
                                                          block_tables, context_lens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = lib().oracle_paged_attention_split(_p(out), _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1],
                                            _p(ctx), B, Hq, Hkv, D, BS, NB, float(scale),
                                            int(num_splits))
    _check(rc, "paged_attention_split")
    return out


def sparse_attention(q, key_cache, value_cache, block_tables, context_lens, selected, scale,
                     rows=None):
    """Quest sparse attention over the selected logical blocks (fp64)."""
    q, kc, vc, bt, ctx, B, Hq, Hkv, D, BS, NB = _att_args(q, key_cache, value_cache,
                                                          block_tables, context_lens)
    sel = _c(selected, np.int32)
    assert sel.shape[:2] == (B, Hkv)
    topk = sel.shape[2]
    r, nr = _rows_arg(rows)
    out = np.zeros((nr, D) if r is not None else (B, Hq, D), dtype=np.float64)
    rc = lib().oracle_sparse_attention(_p(out), _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(ctx),
                                       _p(sel), topk, B, Hq, Hkv, D, BS, NB, float(scale),
                                       _p(r), nr)
    _check(rc, "sparse_attention")
    return out


# ----------------------------------------------------------------- Quest


def _score_args(q, kmin, kmax, block_tables, context_lens, meta_dtype):
    q = _c(q, np.uint16)
    kmin = _c(kmin, meta_dtype)
    kmax = _c(kmax, meta_dtype)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, Hkv, D2 = kmin.shape
    assert D == D2 and kmax.shape == kmin.shape
    return q, kmin, kmax, bt, ctx, (B, Hq, Hkv, D, NB, bt.shape[1])


def _scores_plain(fn, q, kmin, kmax, block_tables, context_lens, BS, meta_dtype, with_abs):
    q, kmin, kmax, bt, ctx, (B, Hq, Hkv, D, NB, MBS) = _score_args(q, kmin, kmax, block_tables,
                                                                   context_lens, meta_dtype)
    out = np.empty((B, Hkv, MBS), dtype=np.float64)
    absum = np.empty((B, Hkv, MBS), dtype=np.float64)
    rc = fn(_p(out), _p(absum), _p(q), _p(kmin), _p(kmax), _p(bt), MBS, _p(ctx), B, Hq, Hkv, D, BS, NB)
    _check(rc, "quest_scores")
    return (out, absum) if with_abs else out


def quest_scores(q, kmin, kmax, block_tables, context_lens, BS: int, with_abs: bool = False):
    """Quest block scores as the method defines them, [B, Hkv, MBS] float64:
    sum over the GQA group of sum_d max(q*min, q*max), written out term by
    term in fp64 (-inf past each sequence's blocks). with_abs: also return
    A = sum_h sum_d |q| * max(|min|, |max|) per block (scales any
    floating-point evaluation's rounding error)."""
    return _scores_plain(lib().oracle_quest_scores_plain, q, kmin, kmax, block_tables, context_lens, BS,
                         np.uint16, with_abs)


def quest_scores_kernel_order(q, kmin, kmax, block_tables, context_lens, BS: int):
    """The same block scores evaluated in fp32 in the CUDA kernel's fixed
    order (a bit-exact reproduction of the kernel's arithmetic), [B, Hkv, MBS]
    float32."""
    q, kmin, kmax, bt, ctx, (B, Hq, Hkv, D, NB, MBS) = _score_args(q, kmin, kmax, block_tables,
                                                                   context_lens, np.uint16)
    out = np.empty((B, Hkv, MBS), dtype=np.float32)
    rc = lib().oracle_quest_scores_kernel_order(_p(out), _p(q), _p(kmin), _p(kmax), _p(bt), MBS, _p(ctx),
                                                B, Hq, Hkv, D, BS, NB)
    _check(rc, "quest_scores_kernel_order")
    return out


def quest_topk(scores, context_lens, BS: int, topk: int):
    """Top-K logical blocks per (b, kvh): [B, Hkv, topk] int32, ascending, -1
    padded; ties to the lower block index. Scores float32 or float64."""
    f64 = np.asarray(scores).dtype == np.float64
    s = _c(scores, np.float64 if f64 else np.float32)
    ctx = _c(context_lens, np.int32)
    B, Hkv, MBS = s.shape
    out = np.empty((B, Hkv, topk), dtype=np.int32)
    fn = lib().oracle_quest_topk_f64 if f64 else lib().oracle_quest_topk
    rc = fn(_p(out), _p(s), MBS, _p(ctx), B, Hkv, BS, int(topk))
    _check(rc, "quest_topk")
    return out


def quest_select(q, kmin, kmax, block_tables, context_lens, BS: int, topk: int):
    """The selection the method defines: top-K of the plain fp64 scores."""
    return quest_topk(quest_scores(q, kmin, kmax, block_tables, context_lens, BS),
                      context_lens, BS, topk)


def quest_select_kernel_order(q, kmin, kmax, block_tables, context_lens, BS: int, topk: int):
    """Top-K of the fp32 kernel-order scores (the CUDA path's exact set)."""
    return quest_topk(quest_scores_kernel_order(q, kmin, kmax, block_tables, context_lens, BS),
                      context_lens, BS, topk)


# ------------------------------------------------------- fp8 (E4M3) cache


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of every fp32 value (ties to even, +-448 saturation, NaN -> 0x7F)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_p(x), _p(out), x.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    """Value of every E4M3 code (float64, NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_p(c), _p(out), c.size)
    return out


def reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale) -> int:
    """Quantise and scatter new K/V rows into uint8 E4M3 caches IN PLACE; returns #out-of-pool slots.

    key_cache is [NB, BS, Hkv, D]; value_cache is [NB, Hkv, D, BS] with the
    tokens of each 16-byte row in the order 0 1 8 9 2 3 10 11 ... (BS = 16)."""
    assert key_cache.dtype == np.uint8 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.uint8 and value_cache.flags.c_contiguous
    NB, BS, Hkv, D = key_cache.shape
    assert value_cache.shape == (NB, Hkv, D, BS) and BS == 16
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    slots = _c(slot_mapping, np.int64)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    assert ks.shape == (Hkv,) and vs.shape == (Hkv,)
    return int(lib().oracle_reshape_and_cache_fp8(_p(key), _p(value), _p(key_cache), _p(value_cache),
                                                  _p(slots), slots.shape[0], _p(ks), _p(vs), Hkv, D, BS,
                                                  NB))


def reshape_and_cache_fp8_block(key, value, key_cache, value_cache, slot_mapping, k_bscale, v_bscale,
                                kmin=None, kmax=None) -> int:
    """Quantise and scatter new K/V rows into uint8 E4M3 caches with per-block
    power-of-two scales, IN PLACE (caches, k_bscale / v_bscale [NB, Hkv]
    float32, and the E4M3 metadata kmin / kmax [NB, Hkv, D] when given);
    returns #out-of-pool slots. A scale of 0 marks a block that holds nothing."""
    for a in (key_cache, value_cache):
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    NB, BS, Hkv, D = key_cache.shape
    assert value_cache.shape == (NB, Hkv, D, BS) and BS == 16
    for a in (k_bscale, v_bscale):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.shape == (NB, Hkv)
    if kmin is not None:
        for a in (kmin, kmax):
            assert a.dtype == np.uint8 and a.flags.c_contiguous and a.shape == (NB, Hkv, D)
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    slots = _c(slot_mapping, np.int64)
    return int(lib().oracle_reshape_and_cache_fp8_block(_p(key), _p(value), _p(key_cache), _p(value_cache),
                                                        _p(kmin), _p(kmax), _p(k_bscale), _p(v_bscale),
                                                        _p(slots), slots.shape[0], Hkv, D, BS, NB))


def quest_update_meta_fp8(kmin, kmax, key, slot_mapping, k_scale, BS: int) -> int:
    """Incremental Quest metadata (E4M3 codes) update IN PLACE; returns #out-of-pool slots."""
    assert kmin.dtype == np.uint8 and kmin.flags.c_contiguous
    assert kmax.dtype == np.uint8 and kmax.flags.c_contiguous
    NB, Hkv, D = kmin.shape
    key = _c(key, np.uint16)
    slots = _c(slot_mapping, np.int64)
    ks = _c(k_scale, np.float32)
    return int(lib().oracle_quest_update_meta_fp8(_p(kmin), _p(kmax), _p(key), _p(slots),
                                                  slots.shape[0], _p(ks), Hkv, D, BS, NB))


def quest_rebuild_meta_fp8(key_cache, block_tables, context_lens, kmin=None, kmax=None):
    """E4M3 metadata of every block a sequence uses, from an E4M3 cache. Returns (kmin, kmax)."""
    NB, BS, Hkv, D = key_cache.shape
    if kmin is None:
        kmin = np.zeros((NB, Hkv, D), dtype=np.uint8)
    if kmax is None:
        kmax = np.zeros((NB, Hkv, D), dtype=np.uint8)
    kc = _c(key_cache, np.uint8)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    rc = lib().oracle_quest_rebuild_meta_fp8(_p(kmin), _p(kmax), _p(kc), _p(bt), bt.shape[1],
                                             _p(ctx), bt.shape[0], Hkv, D, BS, NB)
    _check(rc, "quest_rebuild_meta_fp8")
    return kmin, kmax


def attention_fp8(q, key_cache, value_cache, k_scale, v_scale, block_tables, context_lens, scale,
                  selected=None, rows=None):
    """Dense (selected None) or Quest sparse attention over E4M3 caches, fp64
    (value_cache in the [NB, Hkv, D, 16] layout of reshape_and_cache_fp8).
    k_scale / v_scale: [Hkv] per-KV-head scales, or [NB, Hkv] per-block scales."""
    q = _c(q, np.uint16)
    kc = _c(key_cache, np.uint8)
    vc = _c(value_cache, np.uint8)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32)
    ctx = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, BS, Hkv, D2 = kc.shape
    per_block = ks.ndim == 2
    want = (NB, Hkv) if per_block else (Hkv,)
    assert D == D2 and vc.shape == (NB, Hkv, D, BS) and ks.shape == want and vs.shape == want
    sel, topk = None, 0
    if selected is not None:
        sel = _c(selected, np.int32)
        assert sel.shape[:2] == (B, Hkv)
        topk = sel.shape[2]
    r, nr = _rows_arg(rows)
    out = np.zeros((nr, D) if r is not None else (B, Hq, D), dtype=np.float64)
    fn = lib().oracle_attention_fp8_block if per_block else lib().oracle_attention_fp8
    rc = fn(_p(out), _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt), bt.shape[1], _p(ctx), _p(sel), topk,
            B, Hq, Hkv, D, BS, NB, float(scale), _p(r), nr)
    _check(rc, "attention_fp8")
    return out


def _bscale_arg(k_bscale, NB, Hkv):
    if k_bscale is None:
        return None
    ks = _c(k_bscale, np.float32)
    assert ks.shape == (NB, Hkv)
    return ks


def quest_scores_fp8(q, kmin, kmax, block_tables, context_lens, BS: int, with_abs: bool = False,
                     k_bscale=None):
    """Plain fp64 Quest scores over E4M3 metadata (min/max = decoded codes).
    With per-KV-head scales (k_bscale None) the K scale, a positive factor of
    a whole row, is left out; with per-block scales k_bscale [NB, Hkv] each
    block's score carries its own K scale."""
    if k_bscale is None:
        return _scores_plain(lib().oracle_quest_scores_plain_fp8, q, kmin, kmax, block_tables,
                             context_lens, BS, np.uint8, with_abs)
    q, kmin, kmax, bt, ctx, (B, Hq, Hkv, D, NB, MBS) = _score_args(q, kmin, kmax, block_tables,
                                                                   context_lens, np.uint8)
    ks = _bscale_arg(k_bscale, NB, Hkv)
    out = np.empty((B, Hkv, MBS), dtype=np.float64)
    absum = np.empty((B, Hkv, MBS), dtype=np.float64)
    rc = lib().oracle_quest_scores_plain_fp8_block(_p(out), _p(absum), _p(q), _p(kmin), _p(kmax), _p(ks),
                                                   _p(bt), MBS, _p(ctx), B, Hq, Hkv, D, BS, NB)
    _check(rc, "quest_scores_fp8 (per-block scales)")
    return (out, absum) if with_abs else out


def quest_scores_kernel_order_fp8(q, kmin, kmax, block_tables, context_lens, BS: int, k_bscale=None):
    """fp32 kernel-order scores over E4M3 metadata, [B, Hkv, MBS] float32
    (times the block's K scale when per-block scales k_bscale are given)."""
    q, kmin, kmax, bt, ctx, (B, Hq, Hkv, D, NB, MBS) = _score_args(q, kmin, kmax, block_tables,
                                                                   context_lens, np.uint8)
    out = np.empty((B, Hkv, MBS), dtype=np.float32)
    if k_bscale is None:
        rc = lib().oracle_quest_scores_kernel_order_fp8(_p(out), _p(q), _p(kmin), _p(kmax), _p(bt), MBS,
                                                        _p(ctx), B, Hq, Hkv, D, BS, NB)
    else:
        ks = _bscale_arg(k_bscale, NB, Hkv)
        rc = lib().oracle_quest_scores_kernel_order_fp8_block(_p(out), _p(q), _p(kmin), _p(kmax), _p(ks),
                                                              _p(bt), MBS, _p(ctx), B, Hq, Hkv, D, BS, NB)
    _check(rc, "quest_scores_kernel_order_fp8")
    return out


def quest_select_fp8(q, kmin, kmax, block_tables, context_lens, BS: int, topk: int, k_bscale=None):
    """Top-K of the plain fp64 scores over E4M3 metadata."""
    return quest_topk(quest_scores_fp8(q, kmin, kmax, block_tables, context_lens, BS, k_bscale=k_bscale),
                      context_lens, BS, topk)


def quest_select_kernel_order_fp8(q, kmin, kmax, block_tables, context_lens, BS: int, topk: int,
                                  k_bscale=None):
    """Top-K of the fp32 kernel-order scores over E4M3 metadata."""
    return quest_topk(quest_scores_kernel_order_fp8(q, kmin, kmax, block_tables, context_lens, BS,
                                                    k_bscale=k_bscale),
                      context_lens, BS, topk)


def paged_attention_multi(q, key_cache, value_cache, block_tables, cu_seqlens_q, context_lens, scale,
                          rows=None):
    """Dense attention of multi-token query rows with right-aligned causal masks.

    q: [total_q, Hq, D] bf16 bits; cu_seqlens_q: [B+1]. Returns [total_q, Hq, D]
    float64 (or [len(rows), D] for the listed (row, head) pairs)."""
    q = _c(q, np.uint16)
    kc = _c(key_cache, np.uint16)
    vc = _c(value_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    ctx = _c(context_lens, np.int32)
    total_q, Hq, D = q.shape
    NB, BS, Hkv, D2 = kc.shape
    B = ctx.shape[0]
    assert D == D2 and vc.shape == kc.shape and bt.shape[0] == B and cu.shape == (B + 1,)
    r, nr = _rows_arg(rows)
    out = np.zeros((nr, D) if r is not None else (total_q, Hq, D), dtype=np.float64)
    rc = lib().oracle_paged_attention_multi(_p(out), _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cu),
                                            _p(ctx), B, total_q, Hq, Hkv, D, BS, NB, float(scale), _p(r), nr)
    _check(rc, "paged_attention_multi")
    return out
