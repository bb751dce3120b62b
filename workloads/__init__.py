"""Seeded synthetic inputs for the paged GQA decode / ReshapeAndCache / Quest path.

This module only draws inputs. It holds none of the path's arithmetic (no
cache scatter, no attention, no Quest scoring or selection): both the CPU
oracle's tests and the CUDA path's tests and benchmark take their inputs from
here, so neither side can lean on the other.

Shapes follow the workloads described on the pages:

* "Ascend Kernel-to-Serving Pipeline", section "ReshapeAndCache": new K/V rows
  are contiguous ``[T, Hkv, D]`` and land in the paged cache through
  ``slot_mapping``; a negative slot means the token is skipped.
* "Ascend Kernel-to-Serving Pipeline", section "GQA Paged Attention":
  ``block_tables`` maps logical to physical blocks, ``context_lens`` gives each
  sequence's length, the last block may be partial.
* "18 e2e inference serving" (TileLang tutorial), section 2.6: the cache of one
  layer is ``[physical_block, block_size, kv_head, head_dim]`` and
  ``block_table[seq][logical_block] = physical_block``.
* Same tutorial, section 2.4/2.5: Qwen2.5-7B attention shape, 28 query heads,
  4 KV heads, head_dim 128, bf16.

bf16 values are carried as ``uint16`` bit patterns (numpy has no bf16 type).

Recipe (all draws from ``numpy.random.default_rng`` streams spawned from one
``SeedSequence(seed)``, in a fixed order, so a seed fixes every byte):

* context lengths per config (uniform, log-normal clipped, or fixed);
* a physical pool of exactly ``sum(ceil(ctx/BS))`` blocks (or the stated pool
  size), assigned to logical blocks by a seeded permutation;
* Q, cached K/V and the new tokens' K/V ~ N(0, 1) drawn in float32 and rounded
  to bf16 (round to nearest even);
* the step's new token of sequence b sits at position ``ctx_b - 1``; its cache
  slot is left as poison when the step writes it, and pre-filled when the
  step's slot is negative (padding), so the cache is fully defined;
* cache slots at positions ``>= ctx_b`` and pool blocks that no sequence uses
  hold a bf16 NaN in correctness mode (``poison=True``) and N(0, 1) otherwise;
* Quest planting (when the config asks for it): a seeded 5 % (at least one) of
  each sequence's logical blocks get ``3 * q_hat`` added to every K row, where
  ``q_hat`` is the unit vector of the mean of the GQA group's query vectors;
  the addition is done in float32 on the bf16 value and rounded back to bf16.
"""

from __future__ import annotations

import concurrent.futures
import math
import os
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

BF16_NAN = np.uint16(0x7FC0)

# Draw K/V in chunks of this many physical blocks so that the byte stream of a
# seed does not depend on the machine's memory.
_CHUNK_BLOCKS = 1024


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); finite inputs."""
    u = np.array(x, dtype=np.float32, copy=True, order="C").view(np.uint32)
    b = np.right_shift(u, 16)
    np.bitwise_and(b, 1, out=b)
    b += np.uint32(0x7FFF)
    u += b
    return np.right_shift(u, 16).astype(np.uint16)


def _draw_pool(seed_seq: np.random.SeedSequence, n: int, inner: tuple) -> np.ndarray:
    """n x inner bf16 values ~ N(0, 1).

    The leading dimension is cut into chunks of _CHUNK_BLOCKS; chunk c draws
    from its own stream spawned from `seed_seq`, so the result depends only
    on the seed (not on how many threads fill the chunks)."""
    out = np.empty((n,) + tuple(inner), dtype=np.uint16)
    starts = list(range(0, n, _CHUNK_BLOCKS))
    seeds = seed_seq.spawn(len(starts))

    def fill(i):
        c0 = starts[i]
        c1 = min(n, c0 + _CHUNK_BLOCKS)
        rng = np.random.default_rng(seeds[i])
        out[c0:c1] = f32_to_bf16_bits(rng.standard_normal((c1 - c0,) + tuple(inner), dtype=np.float32))

    workers = max(1, min(len(starts), os.cpu_count() or 1))
    if workers == 1:
        for i in range(len(starts)):
            fill(i)
    else:
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, range(len(starts))))
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One decode step's inputs, all host numpy arrays."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    NB: int
    MBS: int
    topk: int
    scale: float
    context_lens: np.ndarray      # int32 [B]
    block_tables: np.ndarray      # int32 [B, MBS]; entries past a sequence's blocks are -1
    q: np.ndarray                 # uint16 (bf16) [B, Hq, D]
    key_cache: np.ndarray         # uint16 (bf16) [NB, BS, Hkv, D], state before the step's write
    value_cache: np.ndarray       # uint16 (bf16) [NB, BS, Hkv, D]
    key: np.ndarray               # uint16 (bf16) [T, Hkv, D], this step's new tokens
    value: np.ndarray             # uint16 (bf16) [T, Hkv, D]
    slot_mapping: np.ndarray      # int64 [T]; negative = padding, skipped
    token_seq: np.ndarray         # int32 [T], the sequence each new token belongs to
    planted: Optional[np.ndarray] = None   # bool [B, MBS] planted logical blocks (Quest configs)
    poison: bool = True
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def num_blocks(self) -> np.ndarray:
        """ceil(ctx / BS) per sequence (int64)."""
        c = self.context_lens.astype(np.int64)
        return (c + self.BS - 1) // self.BS


# --------------------------------------------------------------------------
# context-length draws
# --------------------------------------------------------------------------

def _ctx_uniform(rng, B, lo, hi):
    return rng.integers(lo, hi + 1, size=B, dtype=np.int64)


def _ctx_lognormal(rng, B, mean, sigma, lo, hi):
    mu = math.log(mean) - sigma * sigma / 2.0
    x = rng.lognormal(mean=mu, sigma=sigma, size=B)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


# --------------------------------------------------------------------------
# generic builder
# --------------------------------------------------------------------------

def build_workload(name: str, *, B: int, Hq: int, Hkv: int, D: int, BS: int,
                   ctx: np.ndarray, seed_seq: np.random.SeedSequence,
                   topk: int, scale: float, pool_blocks: Optional[int] = None,
                   pad_tokens: Optional[np.ndarray] = None,
                   pad_fraction: float = 0.0, plant: bool = False,
                   poison: bool = True) -> Workload:
    """Draw one step's inputs.

    ``pad_tokens``: explicit sequence indices whose new-token slot is -1.
    ``pad_fraction``: else a seeded fraction of the B new tokens get slot -1.
    """
    assert Hq % Hkv == 0
    (s_perm, s_q, s_k, s_v, s_new, s_pad, s_plant) = seed_seq.spawn(7)
    ctx = np.asarray(ctx, dtype=np.int64)
    assert ctx.shape == (B,) and (ctx >= 1).all()
    nb = (ctx + BS - 1) // BS
    used = int(nb.sum())
    NB = used if pool_blocks is None else int(pool_blocks)
    assert NB >= used
    MBS = int(nb.max())

    # physical assignment: seeded permutation of the pool
    perm = np.random.default_rng(s_perm).permutation(NB).astype(np.int32)
    bt = np.full((B, MBS), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        bt[b, : nb[b]] = perm[off: off + nb[b]]
        off += nb[b]

    # queries
    q = f32_to_bf16_bits(np.random.default_rng(s_q).standard_normal((B, Hq, D), dtype=np.float32))

    # cache pools (N(0,1) everywhere, then poison and planting)
    kc = _draw_pool(s_k, NB, (BS, Hkv, D))
    vc = _draw_pool(s_v, NB, (BS, Hkv, D))

    # the step's new tokens: one per sequence, at position ctx-1
    T = B
    rng_new = np.random.default_rng(s_new)
    key = f32_to_bf16_bits(rng_new.standard_normal((T, Hkv, D), dtype=np.float32))
    value = f32_to_bf16_bits(rng_new.standard_normal((T, Hkv, D), dtype=np.float32))
    token_seq = np.arange(B, dtype=np.int32)
    pos = ctx - 1
    phys_new = bt[np.arange(B), pos // BS].astype(np.int64)
    slot = phys_new * BS + pos % BS

    rng_pad = np.random.default_rng(s_pad)
    padded = np.zeros(B, dtype=bool)
    if pad_tokens is not None:
        padded[np.asarray(pad_tokens, dtype=np.int64)] = True
    elif pad_fraction > 0.0:
        npad = int(round(pad_fraction * B))
        padded[rng_pad.choice(B, size=npad, replace=False)] = True
    slot = np.where(padded, -1, slot).astype(np.int64)

    # planting (before poison so that poison stays poison)
    planted = None
    if plant:
        rng_plant = np.random.default_rng(s_plant)
        planted = np.zeros((B, MBS), dtype=bool)
        G = Hq // Hkv
        qf = bf16_bits_to_f32(q).reshape(B, Hkv, G, D)
        qmean = qf.mean(axis=2)                                    # [B, Hkv, D]
        qhat = qmean / np.linalg.norm(qmean, axis=-1, keepdims=True)
        add = (3.0 * qhat).astype(np.float32)                     # [B, Hkv, D]
        for b in range(B):
            n_plant = max(1, int(math.ceil(0.05 * nb[b])))
            js = rng_plant.choice(nb[b], size=n_plant, replace=False)
            planted[b, js] = True
            for j in js:
                p = bt[b, j]
                kf = bf16_bits_to_f32(kc[p])                          # [BS, Hkv, D]
                kc[p] = f32_to_bf16_bits(kf + add[b][None, :, :])
            jn = pos[b] // BS
            if planted[b, jn]:
                key[b] = f32_to_bf16_bits(bf16_bits_to_f32(key[b]) + add[b])

    if poison:
        # slots at positions >= ctx in each sequence's last block
        for b in range(B):
            p_last = bt[b, nb[b] - 1]
            first_invalid = int(ctx[b] - (nb[b] - 1) * BS)
            kc[p_last, first_invalid:] = BF16_NAN
            vc[p_last, first_invalid:] = BF16_NAN
        # pool blocks no sequence uses
        if NB > used:
            unused = perm[used:]
            kc[unused] = BF16_NAN
            vc[unused] = BF16_NAN
        # the new token's slot is poison until the step writes it
        for b in range(B):
            if not padded[b]:
                p = phys_new[b]
                o = int(pos[b] % BS)
                kc[p, o] = BF16_NAN
                vc[p, o] = BF16_NAN

    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, NB=NB, MBS=MBS,
                    topk=topk, scale=scale, context_lens=ctx.astype(np.int32),
                    block_tables=bt, q=q, key_cache=kc, value_cache=vc, key=key,
                    value=value, slot_mapping=slot, token_seq=token_seq,
                    planted=planted, poison=poison,
                    meta={"padded": padded})


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

WORKLOADS = ("tiny", "dense_b32", "quest_8k", "long_40k", "mixed_b128")


def make(name: str, *, poison: bool = True, seed: Optional[int] = None,
         batch: Optional[int] = None, ctx_scale: float = 1.0,
         topk: Optional[int] = None) -> Workload:
    """Build one of the named workloads.

    ``batch`` and ``ctx_scale`` shrink a workload for fast elementwise parity
    (same recipe, fewer and shorter sequences) and ``topk`` overrides the
    selection size; leave them at their defaults for the full sizes.
    """
    w = _make(name, poison=poison, seed=seed, batch=batch, ctx_scale=ctx_scale)
    if topk is not None:
        w.topk = int(topk)
    return w


def _make(name: str, *, poison: bool, seed: Optional[int], batch: Optional[int],
          ctx_scale: float) -> Workload:
    if name == "tiny":
        # batch 2, Hq 4, Hkv 1, D 64, ctx {37, 100}, pool of 16 blocks, topk 3,
        # the second sequence's new-token slot is -1
        s = 0 if seed is None else seed
        return build_workload(name, B=2, Hq=4, Hkv=1, D=64, BS=16,
                              ctx=np.array([37, 100]), seed_seq=np.random.SeedSequence(s),
                              topk=3, scale=1.0 / math.sqrt(64), pool_blocks=16,
                              pad_tokens=np.array([1]), poison=poison)

    qwen = dict(Hq=28, Hkv=4, D=128, BS=16, scale=1.0 / math.sqrt(128))
    if name == "dense_b32":
        s = 1 if seed is None else seed
        ss = np.random.SeedSequence(s)
        s_ctx, s_rest = ss.spawn(2)
        B = 32 if batch is None else batch
        lo, hi = int(1024 * ctx_scale), int(8192 * ctx_scale)
        ctx = _ctx_uniform(np.random.default_rng(s_ctx), B, max(1, lo), max(1, hi))
        return build_workload(name, B=B, ctx=ctx, seed_seq=s_rest, topk=64, poison=poison, **qwen)
    if name == "quest_8k":
        s = 2 if seed is None else seed
        ss = np.random.SeedSequence(s)
        s_ctx, s_rest = ss.spawn(2)
        B = 16 if batch is None else batch
        ctx = _ctx_lognormal(np.random.default_rng(s_ctx), B, 8192 * ctx_scale, 0.5,
                             max(1, int(2048 * ctx_scale)), max(1, int(16384 * ctx_scale)))
        topk = 64 if ctx_scale == 1.0 else max(1, int(64 * ctx_scale))
        return build_workload(name, B=B, ctx=ctx, seed_seq=s_rest, topk=topk,
                              plant=True, poison=poison, **qwen)
    if name == "long_40k":
        s = 3 if seed is None else seed
        ss = np.random.SeedSequence(s)
        _, s_rest = ss.spawn(2)
        B = 4 if batch is None else batch
        ctx = np.full(B, max(1, int(40960 * ctx_scale)), dtype=np.int64)
        topk = 128 if ctx_scale == 1.0 else max(1, int(128 * ctx_scale))
        return build_workload(name, B=B, ctx=ctx, seed_seq=s_rest, topk=topk,
                              plant=True, poison=poison, **qwen)
    if name == "mixed_b128":
        s = 4 if seed is None else seed
        ss = np.random.SeedSequence(s)
        s_ctx, s_rest = ss.spawn(2)
        B = 128 if batch is None else batch
        ctx = _ctx_uniform(np.random.default_rng(s_ctx), B, 16, max(16, int(32768 * ctx_scale)))
        topk = 64 if ctx_scale == 1.0 else max(1, int(64 * ctx_scale))
        return build_workload(name, B=B, ctx=ctx, seed_seq=s_rest, topk=topk,
                              pad_fraction=0.1, poison=poison, **qwen)
    raise ValueError(f"unknown workload {name!r}; choose from {WORKLOADS}")


def random_selection(w: Workload, seed: int) -> np.ndarray:
    """A fixed, seeded block selection in the Quest output format.

    ``[B, Hkv, topk]`` int32: distinct logical block indices below
    ``ceil(ctx/BS)``, ascending, padded with -1. Used to check sparse attention
    on a selection that does not come from the scoring kernels.
    """
    rng = np.random.default_rng(seed)
    nb = w.num_blocks()
    sel = np.full((w.B, w.Hkv, w.topk), -1, dtype=np.int32)
    for b in range(w.B):
        k = min(w.topk, int(nb[b]))
        for h in range(w.Hkv):
            js = np.sort(rng.choice(int(nb[b]), size=k, replace=False))
            sel[b, h, :k] = js
    return sel


def fp8_scales(Hkv: int):
    """Per-KV-head scales for an 8-bit (E4M3) cache of these workloads:
    k_scale[h] = (6 + h/2) / 448, v_scale[h] = (5 + h/2) / 448, so that
    |x| up to about 6 (N(0, 1) values plus the planted signal) maps inside
    the format's finite range without saturating. A fixed calibration (an
    input of the cache), float32 [Hkv] each."""
    h = np.arange(Hkv, dtype=np.float32)
    return ((6.0 + h / 2) / 448.0).astype(np.float32), ((5.0 + h / 2) / 448.0).astype(np.float32)
