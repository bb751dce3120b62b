"""Pins for the CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: hand-worked slot arithmetic, a library softmax-attention routine
(``torch.nn.functional.scaled_dot_product_attention``) on contiguous layouts,
closed forms, invariances, brute force on tiny inputs, and exact integer
cases. A plausible slip in the oracle (a dropped term, a wrong sign, a swapped
index, a wrong head mapping or mask) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

import workloads
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers


def bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def rand_bf16(rng, shape, scale=1.0):
    return bf16(rng.standard_normal(shape).astype(np.float32) * scale)


def contiguous_paged(rng, B, Hkv, D, BS, ctx, permute=True, extra_blocks=0, poison=False):
    """Contiguous per-sequence K/V, and the same data laid out as a paged pool.

    Logical block j of sequence b holds positions j*BS..j*BS+BS-1 of that
    sequence. With permute=False the pool is the identity layout (sequence
    b's blocks are pool blocks b*MBS .. b*MBS+MBS-1), so the pool is a plain
    reshape of the contiguous arrays. With permute=True the pool blocks are
    relabelled by a random permutation (a pure relabelling of the same data).
    """
    ctx = np.asarray(ctx)
    MBS = int(max(1, max((c + BS - 1) // BS for c in ctx)))
    Kc = rand_bf16(rng, (B, MBS * BS, Hkv, D))
    Vc = rand_bf16(rng, (B, MBS * BS, Hkv, D))
    NB = B * MBS + extra_blocks
    kc = np.zeros((NB, BS, Hkv, D), dtype=np.uint16)
    vc = np.zeros((NB, BS, Hkv, D), dtype=np.uint16)
    kc[: B * MBS] = Kc.reshape(B * MBS, BS, Hkv, D)
    vc[: B * MBS] = Vc.reshape(B * MBS, BS, Hkv, D)
    bt = np.arange(B * MBS, dtype=np.int32).reshape(B, MBS)
    if poison:
        for b in range(B):
            flat_k = kc[: B * MBS].reshape(B, MBS * BS, Hkv, D)
            flat_v = vc[: B * MBS].reshape(B, MBS * BS, Hkv, D)
            flat_k[b, ctx[b]:] = 0x7FC0
            flat_v[b, ctx[b]:] = 0x7FC0
        kc[B * MBS:] = 0x7FC0
        vc[B * MBS:] = 0x7FC0
    if permute:
        perm = rng.permutation(NB)
        kc2 = np.empty_like(kc)
        vc2 = np.empty_like(vc)
        kc2[perm] = kc
        vc2[perm] = vc
        kc, vc = kc2, vc2
        bt = perm[bt].astype(np.int32)
    return Kc, Vc, kc, vc, bt, MBS


def sdpa_reference(q, Kc, Vc, ctx, scale):
    """Library softmax attention (fp64) on contiguous K/V, GQA via enable_gqa."""
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        n = int(ctx[b])
        if n == 0:
            continue
        qq = torch.from_numpy(bf16_bits_to_f32(q[b]).astype(np.float64))[:, None, :]    # [Hq,1,D]
        kk = torch.from_numpy(bf16_bits_to_f32(Kc[b, :n]).astype(np.float64)).permute(1, 0, 2)
        vv = torch.from_numpy(bf16_bits_to_f32(Vc[b, :n]).astype(np.float64)).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            qq[None], kk[None], vv[None], scale=scale, enable_gqa=True)
        out[b] = o[0, :, 0, :].numpy()
    return out


# ------------------------------------------------------------ slot math


def test_reshape_slot_math_golden(oracle_lib):
    rows = []
    with open(os.path.join(GOLDEN, "slot_math.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    BS, NB, Hkv, D = 16, 16, 2, 8
    T = len(rows)
    slots = np.array([int(r[0]) for r in rows], dtype=np.int64)
    rng = np.random.default_rng(0)
    key = rand_bf16(rng, (T, Hkv, D))
    value = rand_bf16(rng, (T, Hkv, D))
    kc0 = rand_bf16(rng, (NB, BS, Hkv, D))
    vc0 = rand_bf16(rng, (NB, BS, Hkv, D))
    kc, vc = kc0.copy(), vc0.copy()
    assert oracle_lib.reshape_and_cache(key, value, kc, vc, slots) == 0
    touched = np.zeros((NB, BS), dtype=bool)
    for t, r in enumerate(rows):
        if r[1] == "skip":
            continue
        blk, off = int(r[1]), int(r[2])
        np.testing.assert_array_equal(kc[blk, off], key[t])
        np.testing.assert_array_equal(vc[blk, off], value[t])
        touched[blk, off] = True
    # every other cache byte unchanged (skipped tokens wrote nothing)
    np.testing.assert_array_equal(kc[~touched], kc0[~touched])
    np.testing.assert_array_equal(vc[~touched], vc0[~touched])


def test_reshape_out_of_pool_slot_is_not_written(oracle_lib):
    rng = np.random.default_rng(1)
    NB, BS, Hkv, D = 4, 16, 1, 8
    kc0 = rand_bf16(rng, (NB, BS, Hkv, D))
    kc, vc = kc0.copy(), kc0.copy()
    key = rand_bf16(rng, (2, Hkv, D))
    n = oracle_lib.reshape_and_cache(key, key, kc, vc, np.array([NB * BS, NB * BS + 5]))
    assert n == 2
    np.testing.assert_array_equal(kc, kc0)


# ------------------------------------------------------- dense attention


@pytest.mark.parametrize("B,Hq,Hkv,D,BS,ctx", [
    (2, 4, 1, 64, 16, [37, 100]),        # the tiny workload's shape
    (3, 4, 4, 4, 2, [1, 2, 5]),          # G = 1 (MHA), ctx 1 and one full block
    (2, 6, 2, 8, 4, [3, 13]),            # G = 3, ragged last blocks
    (2, 28, 4, 16, 16, [16, 17]),        # G = 7, exactly one block and one past it
    (1, 8, 1, 32, 8, [64]),              # G = 8, whole blocks only
])
@pytest.mark.parametrize("permute", [False, True])
def test_dense_matches_library_sdpa(oracle_lib, B, Hq, Hkv, D, BS, ctx, permute):
    rng = np.random.default_rng(B * 1000 + Hq * 10 + D)
    Kc, Vc, kc, vc, bt, MBS = contiguous_paged(rng, B, Hkv, D, BS, ctx, permute=permute,
                                               extra_blocks=3, poison=True)
    q = rand_bf16(rng, (B, Hq, D))
    scale = 1.0 / math.sqrt(D)
    ctx_a = np.array(ctx, dtype=np.int32)
    got = oracle_lib.paged_attention(q, kc, vc, bt, ctx_a, scale)
    want = sdpa_reference(q, Kc, Vc, ctx_a, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dense_relabelling_pool_is_invariant(oracle_lib):
    rng = np.random.default_rng(7)
    ctx = np.array([37, 100, 5], dtype=np.int32)
    Kc, Vc, kc, vc, bt, _ = contiguous_paged(rng, 3, 2, 16, 16, ctx, permute=False)
    q = rand_bf16(rng, (3, 6, 16))
    a = oracle_lib.paged_attention(q, kc, vc, bt, ctx, 0.25)
    perm = rng.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    b = oracle_lib.paged_attention(q, kc2, vc2, perm[bt].astype(np.int32), ctx, 0.25)
    np.testing.assert_array_equal(a, b)


def test_dense_closed_forms(oracle_lib):
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D, BS = 2, 4, 2, 8, 4
    ctx = np.array([7, 1], dtype=np.int32)
    Kc, Vc, kc, vc, bt, MBS = contiguous_paged(rng, B, Hkv, D, BS, ctx, poison=True)
    q = rand_bf16(rng, (B, Hq, D))
    # (a) every valid V row equal to one vector -> output is that vector
    const = rand_bf16(rng, (Hkv, D))
    vc_c = vc.copy()
    for b in range(B):
        for t in range(ctx[b]):
            vc_c[bt[b, t // BS], t % BS] = const
    out = oracle_lib.paged_attention(q, kc, vc_c, bt, ctx, 0.3)
    G = Hq // Hkv
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(bf16_bits_to_f32(const[h // G]), (B, D)),
                                   rtol=1e-14, atol=1e-14)
    # (b) every valid K row equal -> uniform weights -> mean of valid V rows
    kc_c = kc.copy()
    for b in range(B):
        for t in range(ctx[b]):
            kc_c[bt[b, t // BS], t % BS] = const
    out = oracle_lib.paged_attention(q, kc_c, vc, bt, ctx, 0.3)
    for b in range(B):
        mean_v = bf16_bits_to_f32(Vc[b, : ctx[b]]).astype(np.float64).mean(axis=0)   # [Hkv, D]
        for h in range(Hq):
            np.testing.assert_allclose(out[b, h], mean_v[h // G], rtol=1e-12, atol=1e-12)
    # (c) ctx = 1 -> output is that token's V row
    np.testing.assert_allclose(out[1, 0], bf16_bits_to_f32(Vc[1, 0, 0]), rtol=0, atol=0)
    # (d) a dominant score picks one token's V
    q2 = np.zeros_like(q)
    kc_d = kc.copy()
    big = bf16(np.full(D, 4.0))
    q2[:] = big
    kc_d[bt[0, 3 // BS], 3 % BS, 0] = bf16(np.full(D, 8.0))
    out = oracle_lib.paged_attention(q2, kc_d, vc, bt, ctx, 1.0)
    np.testing.assert_allclose(out[0, 0], bf16_bits_to_f32(Vc[0, 3, 0]), atol=1e-12)


def test_dense_empty_context_is_zero(oracle_lib):
    rng = np.random.default_rng(4)
    Kc, Vc, kc, vc, bt, _ = contiguous_paged(rng, 2, 1, 8, 4, [5, 3])
    q = rand_bf16(rng, (2, 2, 8))
    out = oracle_lib.paged_attention(q, kc, vc, bt, np.array([0, 3], dtype=np.int32), 1.0)
    assert (out[0] == 0).all() and np.isfinite(out[1]).all()


def test_masked_poison_does_not_leak(oracle_lib):
    w = workloads.make("tiny", poison=True)
    w2 = workloads.make("tiny", poison=False)
    # identical valid data, different content past ctx and in unused blocks
    for a in (w, w2):
        oracle_lib.reshape_and_cache(a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping)
    o1 = oracle_lib.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens, w.scale)
    o2 = oracle_lib.paged_attention(w2.q, w2.key_cache, w2.value_cache, w2.block_tables, w2.context_lens, w2.scale)
    assert np.isfinite(o1).all()
    np.testing.assert_array_equal(o1, o2)


# ---------------------------------------------- online softmax and split-KV


@pytest.mark.parametrize("chunk", [1, 3, 16, 1000])
def test_online_softmax_equals_two_pass(oracle_lib, chunk):
    rng = np.random.default_rng(5)
    ctx = np.array([37, 100, 1], dtype=np.int32)
    _, _, kc, vc, bt, _ = contiguous_paged(rng, 3, 2, 32, 16, ctx, poison=True)
    q = rand_bf16(rng, (3, 8, 32), scale=3.0)   # large logits so the max moves
    a = oracle_lib.paged_attention(q, kc, vc, bt, ctx, 0.5)
    b = oracle_lib.paged_attention_online(q, kc, vc, bt, ctx, 0.5, chunk)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_split_combine_equals_two_pass(oracle_lib, splits):
    rng = np.random.default_rng(6)
    ctx = np.array([37, 100, 2], dtype=np.int32)
    _, _, kc, vc, bt, _ = contiguous_paged(rng, 3, 2, 32, 16, ctx, poison=True)
    q = rand_bf16(rng, (3, 8, 32), scale=3.0)
    a = oracle_lib.paged_attention(q, kc, vc, bt, ctx, 0.5)
    b = oracle_lib.paged_attention_split(q, kc, vc, bt, ctx, 0.5, splits)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


def test_sampled_rows_equal_full(oracle_lib):
    w = workloads.make("tiny")
    oracle_lib.reshape_and_cache(w.key, w.value, w.key_cache, w.value_cache, w.slot_mapping)
    full = oracle_lib.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens, w.scale)
    rows = [(1, 3), (0, 0), (1, 1)]
    part = oracle_lib.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens,
                                      w.scale, rows=rows)
    for i, (b, h) in enumerate(rows):
        np.testing.assert_array_equal(part[i], full[b, h])


# --------------------------------------------------------- sparse attention


def test_sparse_all_blocks_equals_dense(oracle_lib):
    w = workloads.make("tiny")
    oracle_lib.reshape_and_cache(w.key, w.value, w.key_cache, w.value_cache, w.slot_mapping)
    nb = w.num_blocks()
    K = int(nb.max()) + 2
    sel = np.full((w.B, w.Hkv, K), -1, dtype=np.int32)
    for b in range(w.B):
        sel[b, :, : nb[b]] = np.arange(nb[b])
    dense = oracle_lib.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens, w.scale)
    sparse = oracle_lib.sparse_attention(w.q, w.key_cache, w.value_cache, w.block_tables,
                                         w.context_lens, sel, w.scale)
    np.testing.assert_array_equal(sparse, dense)


def test_sparse_matches_sdpa_on_selected_tokens(oracle_lib):
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, BS = 2, 6, 2, 16, 4
    ctx = np.array([23, 9], dtype=np.int32)
    Kc, Vc, kc, vc, bt, MBS = contiguous_paged(rng, B, Hkv, D, BS, ctx, poison=True)
    q = rand_bf16(rng, (B, Hq, D))
    K = 3
    # per KV head selections, including the partial last block and padding
    sel = np.array([[[0, 2, 5], [1, 4, -1]], [[2, -1, -1], [0, 1, 2]]], dtype=np.int32)
    got = oracle_lib.sparse_attention(q, kc, vc, bt, ctx, sel, 0.4)
    G = Hq // Hkv
    for b in range(B):
        for kvh in range(Hkv):
            toks = [t for j in sel[b, kvh] if j >= 0 for t in range(j * BS, min((j + 1) * BS, ctx[b]))]
            qq = q[b:b + 1, kvh * G:(kvh + 1) * G]
            Ks = Kc[b:b + 1, toks][:, :, kvh:kvh + 1]
            Vs = Vc[b:b + 1, toks][:, :, kvh:kvh + 1]
            want = sdpa_reference(qq, Ks, Vs, np.array([len(toks)]), 0.4)
            np.testing.assert_allclose(got[b, kvh * G:(kvh + 1) * G], want[0], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ Quest metadata


def test_rebuild_meta_is_elementwise_min_max(oracle_lib):
    w = workloads.make("tiny")
    oracle_lib.reshape_and_cache(w.key, w.value, w.key_cache, w.value_cache, w.slot_mapping)
    kmin, kmax = oracle_lib.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    nb = w.num_blocks()
    for b in range(w.B):
        for j in range(nb[b]):
            p = w.block_tables[b, j]
            n = min(w.BS, int(w.context_lens[b]) - j * w.BS)
            vals = bf16_bits_to_f32(w.key_cache[p, :n])            # [n, Hkv, D]
            assert np.isfinite(vals).all()
            np.testing.assert_array_equal(bf16_bits_to_f32(kmin[p]), vals.min(axis=0))
            np.testing.assert_array_equal(bf16_bits_to_f32(kmax[p]), vals.max(axis=0))


def _meta_brute(kmin0, kmax0, key, slots, BS):
    kmin, kmax = bf16_bits_to_f32(kmin0).copy(), bf16_bits_to_f32(kmax0).copy()
    kf = bf16_bits_to_f32(key)
    blocks = {}
    for t, s in enumerate(slots):
        if s >= 0:
            blocks.setdefault(s // BS, []).append(t)
    for p, ts in blocks.items():
        vals = kf[ts]
        if any(slots[t] % BS == 0 for t in ts):
            kmin[p], kmax[p] = vals.min(axis=0), vals.max(axis=0)
        else:
            kmin[p] = np.minimum(kmin[p], vals.min(axis=0))
            kmax[p] = np.maximum(kmax[p], vals.max(axis=0))
    return kmin, kmax


def test_update_meta_brute_force_and_order_independent(oracle_lib):
    rng = np.random.default_rng(9)
    NB, BS, Hkv, D = 6, 4, 2, 8
    kmin0 = rand_bf16(rng, (NB, Hkv, D))
    kmax0 = rand_bf16(rng, (NB, Hkv, D))
    # tokens into blocks 1 (offsets 1,2: merge), 3 (offsets 0,3: reset), 5 (offset 2)
    slots = np.array([1 * BS + 1, 3 * BS + 3, -1, 1 * BS + 2, 3 * BS + 0, 5 * BS + 2], dtype=np.int64)
    key = rand_bf16(rng, (len(slots), Hkv, D))
    a_min, a_max = kmin0.copy(), kmax0.copy()
    oracle_lib.quest_update_meta(a_min, a_max, key, slots, BS)
    w_min, w_max = _meta_brute(kmin0, kmax0, key, slots, BS)
    np.testing.assert_array_equal(bf16_bits_to_f32(a_min), w_min)
    np.testing.assert_array_equal(bf16_bits_to_f32(a_max), w_max)
    # blocks not touched are unchanged
    for p in (0, 2, 4):
        np.testing.assert_array_equal(a_min[p], kmin0[p])
    perm = rng.permutation(len(slots))
    b_min, b_max = kmin0.copy(), kmax0.copy()
    oracle_lib.quest_update_meta(b_min, b_max, key[perm], slots[perm], BS)
    np.testing.assert_array_equal(a_min, b_min)
    np.testing.assert_array_equal(a_max, b_max)


def test_update_meta_signed_zero_is_order_independent(oracle_lib):
    NB, BS, Hkv, D = 2, 4, 1, 2
    key = np.array([[[0x8000, 0x0000]], [[0x0000, 0x8000]]], dtype=np.uint16)   # -0/+0 mixes
    slots = np.array([0, 1], dtype=np.int64)
    a_min = np.zeros((NB, Hkv, D), np.uint16)
    a_max = np.zeros((NB, Hkv, D), np.uint16)
    oracle_lib.quest_update_meta(a_min, a_max, key, slots, BS)
    b_min, b_max = np.zeros_like(a_min), np.zeros_like(a_max)
    oracle_lib.quest_update_meta(b_min, b_max, key[::-1].copy(), slots[::-1].copy(), BS)
    np.testing.assert_array_equal(a_min, b_min)
    assert (a_min[0] == 0x8000).all() and (a_max[0] == 0x0000).all()


def test_incremental_decode_meta_equals_rebuild(oracle_lib):
    """Appending one token per step, the running metadata equals the rebuild."""
    rng = np.random.default_rng(10)
    B, Hkv, D, BS, steps = 3, 2, 8, 4, 11
    ctx0 = np.array([1, 4, 6])
    MBS = (int(ctx0.max()) + steps + BS - 1) // BS
    NB = B * MBS
    bt = rng.permutation(NB).astype(np.int32).reshape(B, MBS)
    kc = np.full((NB, BS, Hkv, D), 0x7FC0, dtype=np.uint16)
    ctx = ctx0.copy()
    for b in range(B):
        for t in range(ctx[b]):
            kc[bt[b, t // BS], t % BS] = rand_bf16(rng, (Hkv, D))
    kmin, kmax = oracle_lib.quest_rebuild_meta(kc, bt, ctx.astype(np.int32))
    for _ in range(steps):
        key = rand_bf16(rng, (B, Hkv, D))
        slots = np.array([bt[b, ctx[b] // BS] * BS + ctx[b] % BS for b in range(B)], dtype=np.int64)
        oracle_lib.reshape_and_cache(key, key, kc, kc.copy(), slots)
        oracle_lib.quest_update_meta(kmin, kmax, key, slots, BS)
        ctx += 1
        r_min, r_max = oracle_lib.quest_rebuild_meta(kc, bt, ctx.astype(np.int32),
                                                     kmin.copy(), kmax.copy())
        np.testing.assert_array_equal(kmin, r_min)
        np.testing.assert_array_equal(kmax, r_max)


# ------------------------------------------------------------- Quest score
#
# Two oracle functions compute the block score: quest_scores (the method's
# sum written out term by term in fp64) and quest_scores_kernel_order (fp32 in
# the CUDA kernel's evaluation order, for bit-exact comparison). Each is
# pinned to closed forms and brute force; the kernel-order one is also held
# to the stated fp32 error bound around the plain one.


def _both(oracle_lib, q, kmin, kmax, bt, ctx, BS):
    return (oracle_lib.quest_scores(q, kmin, kmax, bt, ctx, BS),
            oracle_lib.quest_scores_kernel_order(q, kmin, kmax, bt, ctx, BS).astype(np.float64))


def test_quest_score_exact_on_integers(oracle_lib):
    """Small-integer inputs make every fp32 and fp64 step exact: both score
    functions must equal the integer value of sum_h sum_d max(q*min, q*max)."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, BS = 2, 6, 2, 64, 4
    NB = 8
    q = bf16(rng.integers(-4, 5, (B, Hq, D)).astype(np.float32))
    lo = rng.integers(-8, 8, (NB, Hkv, D))
    hi = lo + rng.integers(0, 5, (NB, Hkv, D))
    kmin, kmax = bf16(lo.astype(np.float32)), bf16(hi.astype(np.float32))
    bt = rng.permutation(NB).astype(np.int32).reshape(B, 4)
    ctx = np.array([13, 5], dtype=np.int32)
    qi = bf16_bits_to_f32(q).astype(np.int64)
    want = np.full((B, Hkv, 4), -np.inf)
    G = Hq // Hkv
    for b in range(B):
        for j in range((int(ctx[b]) + BS - 1) // BS):
            p = bt[b, j]
            for kvh in range(Hkv):
                qq = qi[b, kvh * G:(kvh + 1) * G]                  # [G, D]
                want[b, kvh, j] = np.maximum(qq * lo[p, kvh], qq * hi[p, kvh]).sum()
    for got in _both(oracle_lib, q, kmin, kmax, bt, ctx, BS):
        np.testing.assert_array_equal(got, want)
        assert np.isneginf(got[1, :, 2:]).all()          # blocks past ctx excluded


def test_quest_score_identical_tokens_is_group_dot_product(oracle_lib):
    """A block whose tokens all hold the same key k has min = max = k, and the
    bound collapses to the group-summed logit sum_h q_h . k: a library dot
    product (numpy, fp64)."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, D, BS, NB = 3, 28, 4, 128, 16, 9
    q = rand_bf16(rng, (B, Hq, D))
    k = rand_bf16(rng, (NB, Hkv, D))
    bt = rng.permutation(NB).astype(np.int32).reshape(B, 3)
    ctx = np.array([40, 33, 17], dtype=np.int32)
    plain, korder = _both(oracle_lib, q, k, k, bt, ctx, BS)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    kf = bf16_bits_to_f32(k).astype(np.float64)
    G = Hq // Hkv
    for b in range(B):
        for j in range((int(ctx[b]) + BS - 1) // BS):
            for kvh in range(Hkv):
                want = np.dot(qf[b, kvh * G:(kvh + 1) * G].sum(axis=0), kf[bt[b, j], kvh])
                assert abs(plain[b, kvh, j] - want) <= 1e-12 * (1 + abs(want))
                assert abs(korder[b, kvh, j] - want) <= 1e-4 * (1 + abs(want))


def test_quest_score_sign_closed_forms(oracle_lib):
    """With every query element >= 0 the bound takes the max side everywhere:
    score = (sum_h q_h) . max; with every element <= 0 it takes the min side:
    score = (sum_h q_h) . min (library dot products)."""
    rng = np.random.default_rng(22)
    B, Hq, Hkv, D, BS, NB = 2, 8, 2, 64, 16, 6
    lo = rng.standard_normal((NB, Hkv, D)).astype(np.float32)
    kmin = bf16(lo)
    kmax = bf16(lo + np.abs(rng.standard_normal((NB, Hkv, D))).astype(np.float32) + 0.25)
    bt = rng.permutation(NB).astype(np.int32).reshape(B, 3)
    ctx = np.array([48, 20], dtype=np.int32)
    mn = bf16_bits_to_f32(kmin).astype(np.float64)
    mx = bf16_bits_to_f32(kmax).astype(np.float64)
    G = Hq // Hkv
    for sign, side in ((1.0, mx), (-1.0, mn)):
        q = bf16(sign * np.abs(rng.standard_normal((B, Hq, D))).astype(np.float32))
        qf = bf16_bits_to_f32(q).astype(np.float64)
        plain, korder = _both(oracle_lib, q, kmin, kmax, bt, ctx, BS)
        for b in range(B):
            for j in range((int(ctx[b]) + BS - 1) // BS):
                for kvh in range(Hkv):
                    want = np.dot(qf[b, kvh * G:(kvh + 1) * G].sum(axis=0), side[bt[b, j], kvh])
                    assert abs(plain[b, kvh, j] - want) <= 1e-12 * (1 + abs(want))
                    assert abs(korder[b, kvh, j] - want) <= 1e-4 * (1 + abs(want))


def test_quest_score_group_mapping(oracle_lib):
    """Query head h belongs to KV head h // G: with one non-zero query head,
    only its KV head's score row is non-zero."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, D, BS, NB = 1, 12, 3, 64, 16, 4
    kmin = rand_bf16(rng, (NB, Hkv, D))
    kmax = bf16(bf16_bits_to_f32(kmin) + 1.0)
    bt = np.arange(NB, dtype=np.int32).reshape(1, NB)
    ctx = np.array([NB * BS], dtype=np.int32)
    G = Hq // Hkv
    for h0 in (0, 5, 11):
        q = np.zeros((B, Hq, D), dtype=np.uint16)
        q[0, h0] = rand_bf16(rng, (D,))
        for sc in _both(oracle_lib, q, kmin, kmax, bt, ctx, BS):
            nz = np.abs(sc[0]).sum(axis=1) > 0
            np.testing.assert_array_equal(nz, np.arange(Hkv) == h0 // G)


def test_quest_score_abs_sum(oracle_lib):
    """A = sum_h sum_d |q| max(|min|, |max|) bounds |score|, and equals the
    score when q and the metadata are all non-negative."""
    rng = np.random.default_rng(24)
    B, Hq, Hkv, D, BS, NB = 2, 8, 2, 64, 16, 6
    bt = rng.permutation(NB).astype(np.int32).reshape(B, 3)
    ctx = np.array([48, 20], dtype=np.int32)
    q = rand_bf16(rng, (B, Hq, D))
    lo = rng.standard_normal((NB, Hkv, D)).astype(np.float32)
    kmin, kmax = bf16(lo), bf16(lo + 0.5)
    s, a = oracle_lib.quest_scores(q, kmin, kmax, bt, ctx, BS, with_abs=True)
    fin = np.isfinite(s)
    assert (a[fin] >= np.abs(s[fin])).all() and (a[~fin] == 0).all()
    q = bf16(np.abs(bf16_bits_to_f32(q)))
    kmin = bf16(np.abs(lo))
    kmax = bf16(np.abs(lo) + 0.5)
    s, a = oracle_lib.quest_scores(q, kmin, kmax, bt, ctx, BS, with_abs=True)
    np.testing.assert_array_equal(a[fin], s[fin])


@pytest.mark.parametrize("name", ["tiny", "quest_8k"])
def test_quest_score_kernel_order_within_fp32_bound(oracle_lib, name):
    """The fp32 kernel-order score stays within the stated rounding bound
    E = (gamma_{G+D/32+5}(2^-24) + gamma_{G*D}(2^-53)) * A of the plain fp64
    score, on every block of the workload (the bound the selection check
    relies on)."""
    from tests.selection_check import score_error_bound
    kw = {} if name == "tiny" else dict(batch=4, ctx_scale=0.25, topk=16)
    w = workloads.make(name, poison=False, **kw)
    kmin, kmax = oracle_lib.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    plain, a = oracle_lib.quest_scores(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, with_abs=True)
    korder = oracle_lib.quest_scores_kernel_order(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS)
    fin = np.isfinite(plain)
    assert (np.isfinite(korder) == fin).all()
    E = score_error_bound(a, w.Hq // w.Hkv, w.D)
    err = np.abs(korder[fin].astype(np.float64) - plain[fin])
    assert (err <= E[fin]).all(), float((err / E[fin]).max())


def test_quest_bound_dominates_true_max(oracle_lib):
    """sum_d max(q*min, q*max) >= max over the block's valid tokens of q.k,
    per query head and for the group sum (brute force)."""
    w = workloads.make("tiny")
    oracle_lib.reshape_and_cache(w.key, w.value, w.key_cache, w.value_cache, w.slot_mapping)
    kmin, kmax = oracle_lib.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    qf = bf16_bits_to_f32(w.q).astype(np.float64)
    mn = bf16_bits_to_f32(kmin).astype(np.float64)
    mx = bf16_bits_to_f32(kmax).astype(np.float64)
    plain, korder = _both(oracle_lib, w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        for j in range(w.num_blocks()[b]):
            p = w.block_tables[b, j]
            n = min(w.BS, int(w.context_lens[b]) - j * w.BS)
            K = bf16_bits_to_f32(w.key_cache[p, :n]).astype(np.float64)   # [n, Hkv, D]
            for kvh in range(w.Hkv):
                group_logits = np.zeros(n)
                for g in range(G):
                    qq = qf[b, kvh * G + g]
                    bound_h = np.maximum(qq * mn[p, kvh], qq * mx[p, kvh]).sum()
                    logits = K[:, kvh] @ qq
                    assert bound_h >= logits.max() - 1e-9
                    group_logits += logits
                assert plain[b, kvh, j] >= group_logits.max() - 1e-9
                assert korder[b, kvh, j] >= group_logits.max() - 1e-3


# -------------------------------------------------------------- Quest top-K


def test_topk_brute_force_with_ties(oracle_lib):
    rng = np.random.default_rng(12)
    B, Hkv, MBS, BS, K = 3, 2, 40, 16, 7
    scores = rng.integers(0, 6, (B, Hkv, MBS)).astype(np.float32)   # many ties
    ctx = np.array([40 * 16, 5 * 16 - 3, 9 * 16], dtype=np.int32)
    sel = oracle_lib.quest_topk(scores, ctx, BS, K)
    for b in range(B):
        nb = (int(ctx[b]) + BS - 1) // BS
        for kvh in range(Hkv):
            s = scores[b, kvh, :nb]
            order = np.lexsort((np.arange(nb), -s))      # score desc, index asc
            want = np.sort(order[: min(K, nb)])
            row = sel[b, kvh]
            np.testing.assert_array_equal(row[: len(want)], want)
            assert (row[len(want):] == -1).all()


def test_topk_f64_brute_force_with_ties_and_signs(oracle_lib):
    """The top-K over fp64 scores (the plain score's type): negative and
    positive scores, -0 ranked below +0, planted ties, against a lexsort."""
    rng = np.random.default_rng(13)
    B, Hkv, MBS, BS, K = 3, 2, 50, 16, 9
    scores = rng.integers(-4, 4, (B, Hkv, MBS)).astype(np.float64) * 0.375
    scores[0, 0, :6] = [0.0, -0.0, 0.0, -0.0, 1e300, -1e300]
    ctx = np.array([50 * 16, 6 * 16 - 1, 20 * 16], dtype=np.int32)
    sel = oracle_lib.quest_topk(scores, ctx, BS, K)
    for b in range(B):
        nb = (int(ctx[b]) + BS - 1) // BS
        for kvh in range(Hkv):
            s = scores[b, kvh, :nb]
            signbit = np.signbit(s).astype(np.int8)            # -0 ranks below +0
            order = np.lexsort((np.arange(nb), signbit * (s == 0), -s))
            want = np.sort(order[: min(K, nb)])
            row = sel[b, kvh]
            np.testing.assert_array_equal(row[: len(want)], want)
            assert (row[len(want):] == -1).all()


def test_topk_fewer_blocks_than_k_selects_all(oracle_lib):
    scores = np.array([[[3.0, -1.0, 2.0, 9.0]]], dtype=np.float32)
    sel = oracle_lib.quest_topk(scores, np.array([40], dtype=np.int32), 16, 5)
    np.testing.assert_array_equal(sel[0, 0], [0, 1, 2, -1, -1])


def test_topk_tie_goes_to_lower_index(oracle_lib):
    scores = np.array([[[1.0, 5.0, 5.0, 5.0, 0.0]]], dtype=np.float32)
    sel = oracle_lib.quest_topk(scores, np.array([80], dtype=np.int32), 16, 2)
    np.testing.assert_array_equal(sel[0, 0], [1, 2])


def test_quest_topk_at_least_blocks_equals_dense(oracle_lib):
    """Quest with topk >= number of blocks attends to everything: equals dense."""
    w = workloads.make("tiny")
    oracle_lib.reshape_and_cache(w.key, w.value, w.key_cache, w.value_cache, w.slot_mapping)
    kmin, kmax = oracle_lib.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    sel = oracle_lib.quest_select(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, w.MBS)
    dense = oracle_lib.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens, w.scale)
    sparse = oracle_lib.sparse_attention(w.q, w.key_cache, w.value_cache, w.block_tables,
                                         w.context_lens, sel, w.scale)
    np.testing.assert_array_equal(sparse, dense)
    # the tiny workload's first sequence has exactly 3 blocks and topk 3
    sel3 = oracle_lib.quest_select(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, 3)
    np.testing.assert_array_equal(sel3[0, 0], [0, 1, 2])
    s3 = oracle_lib.sparse_attention(w.q, w.key_cache, w.value_cache, w.block_tables,
                                     w.context_lens, sel3, w.scale)
    np.testing.assert_array_equal(s3[0], dense[0])
