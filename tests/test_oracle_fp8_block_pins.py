"""Pins for the oracle's 8-bit cache with per-block power-of-two scales,
independent of the oracle's own code.

The scale rule is fixed by its statement: the stored scale of a (block, KV
head) is the smallest power of two 2^e (e >= -126) with every finite |x|
written since the block restarted at most 448 * 2^e. Against that: the
library's float8_e4m3fn cast (PyTorch) of x / 2^e for every code written in
the same call as the scale's last change, a hand-worked example, the
from-scratch encoding of a block's tokens with its final scale (exact in the
E4M3 normal range, one subnormal step otherwise), the pinned metadata
rebuild, and the pinned bf16 attention and score functions on caches whose
elements are the dequantised values (exact in bf16 for power-of-two scales).
"""

import math

import numpy as np

from tests.test_oracle_fp8_pins import V_ORDER, bf16, torch_decode, torch_encode_sat, v_token_major
from workloads import bf16_bits_to_f32


def fit_exponent(a: float) -> int:
    """Smallest e >= -126 with a <= 448 * 2^e, by its definition."""
    e = -126
    while a > 448.0 * 2.0 ** e:
        e += 1
    return e


def empty(NB, Hkv, D, BS=16):
    kc = np.zeros((NB, BS, Hkv, D), dtype=np.uint8)
    vc = np.zeros((NB, Hkv, D, BS), dtype=np.uint8)
    ks = np.zeros((NB, Hkv), dtype=np.float32)
    vs = np.zeros((NB, Hkv), dtype=np.float32)
    kmin = np.zeros((NB, Hkv, D), dtype=np.uint8)
    kmax = np.zeros((NB, Hkv, D), dtype=np.uint8)
    return kc, vc, ks, vs, kmin, kmax


def test_hand_worked_example(oracle_lib):
    """One KV head, D = 16. Token 0 (offset 0): largest |k| = 2, so the scale
    is 2^-7 (2 <= 448 * 2^-7 = 3.5, 2 > 448 * 2^-8 = 1.75) and k = 1, -2,
    0.5 are stored as 128, -256, 64. Token 1 (offset 1) holds 100: the scale
    grows to 2^-2 (100 <= 112, 100 > 56); token 0's codes are re-encoded
    with the factor 2^-5 (to 4, -8, 2, exact), and 100 / 2^-2 = 400 lies
    halfway between the grid points 384 and 416 of [256, 512): ties to the
    even mantissa give 384."""
    kc, vc, ks, vs, kmin, kmax = empty(2, 1, 16)
    k0 = np.zeros((1, 1, 16), dtype=np.float32)
    k0[0, 0, :3] = [1.0, -2.0, 0.5]
    oracle_lib.reshape_and_cache_fp8_block(bf16(k0), bf16(k0), kc, vc, np.array([16], dtype=np.int64),
                                           ks, vs, kmin, kmax)
    assert ks[1, 0] == 2.0 ** -7 and ks[0, 0] == 0.0
    np.testing.assert_array_equal(torch_decode(kc[1, 0, 0, :3]), [128.0, -256.0, 64.0])
    k1 = np.zeros((1, 1, 16), dtype=np.float32)
    k1[0, 0, 0] = 100.0
    oracle_lib.reshape_and_cache_fp8_block(bf16(k1), bf16(k1), kc, vc, np.array([17], dtype=np.int64),
                                           ks, vs, kmin, kmax)
    assert ks[1, 0] == 2.0 ** -2 and vs[1, 0] == 2.0 ** -2
    np.testing.assert_array_equal(torch_decode(kc[1, 0, 0, :3]), [4.0, -8.0, 2.0])
    assert torch_decode(kc[1, 1, 0, 0]) == 384.0
    # metadata: elementwise min / max of the two tokens' codes
    np.testing.assert_array_equal(torch_decode(kmax[1, 0, :3]), [384.0, 0.0, 2.0])
    np.testing.assert_array_equal(torch_decode(kmin[1, 0, :3]), [4.0, -8.0, 0.0])
    # V: the same values in the V layout (token o at byte V_ORDER.index(o))
    col0, col1 = list(V_ORDER).index(0), list(V_ORDER).index(1)
    np.testing.assert_array_equal(torch_decode(vc[1, 0, :3, col0]), [4.0, -8.0, 2.0])
    assert torch_decode(vc[1, 0, 0, col1]) == 384.0


def test_first_write_scale_and_codes(oracle_lib):
    """A call into empty blocks: each (block, head) scale is the smallest
    power of two that fits the call's tokens of that block, and every code
    is the library cast of x / scale (no value saturates). Negative slots
    and blocks no token lands in are left alone."""
    rng = np.random.default_rng(11)
    NB, Hkv, D, T = 6, 3, 32, 40
    kc, vc, ks, vs, kmin, kmax = empty(NB, Hkv, D)
    kc[:] = 0x11
    mag = np.array([0.01, 1.0, 300.0])[None, :, None]  # very different ranges per head
    key = bf16(rng.standard_normal((T, Hkv, D)) * mag)
    value = bf16(rng.standard_normal((T, Hkv, D)) * mag[:, ::-1])
    slots = rng.permutation(5 * 16)[:T].astype(np.int64)  # blocks 0..4, block 5 untouched
    slots[[3, 17]] = -1
    assert oracle_lib.reshape_and_cache_fp8_block(key, value, kc, vc, slots, ks, vs, kmin, kmax) == 0
    kf, vf = bf16_bits_to_f32(key).astype(np.float64), bf16_bits_to_f32(value).astype(np.float64)
    vnat = v_token_major(vc)
    for p in range(NB):
        members = [t for t in range(T) if slots[t] >= 0 and slots[t] // 16 == p]
        for h in range(Hkv):
            if not members:
                assert ks[p, h] == 0.0 and vs[p, h] == 0.0
                continue
            ek = fit_exponent(np.abs(kf[members, h]).max())
            ev = fit_exponent(np.abs(vf[members, h]).max())
            assert ks[p, h] == 2.0 ** ek and vs[p, h] == 2.0 ** ev
            for t in members:
                o = slots[t] % 16
                np.testing.assert_array_equal(kc[p, o, h], torch_encode_sat(kf[t, h] / 2.0 ** ek))
                np.testing.assert_array_equal(vnat[p, o, h], torch_encode_sat(vf[t, h] / 2.0 ** ev))
    assert (kc[5] == 0x11).all()


def _decode_steps(oracle_lib, rng, NB, Hkv, D, B, steps, growth):
    """Sequences appended one token per call, magnitudes growing with time
    so that the block scales keep rising. Returns the history of written
    tokens and the final state."""
    BS = 16
    MBS = (steps + BS - 1) // BS
    bt = rng.permutation(NB)[: B * MBS].astype(np.int32).reshape(B, MBS)
    kc, vc, ks, vs, kmin, kmax = empty(NB, Hkv, D)
    hist_k = np.zeros((NB, BS, Hkv, D)), np.zeros((NB, BS, Hkv, D))
    for step in range(steps):
        f = growth ** step
        key = bf16(rng.standard_normal((B, Hkv, D)) * f)
        value = bf16(rng.standard_normal((B, Hkv, D)) * f * 0.5)
        slots = np.array([bt[b, step // BS] * BS + step % BS for b in range(B)], dtype=np.int64)
        oracle_lib.reshape_and_cache_fp8_block(key, value, kc, vc, slots, ks, vs, kmin, kmax)
        for b in range(B):
            p, o = bt[b, step // BS], step % BS
            hist_k[0][p, o] = bf16_bits_to_f32(key[b])
            hist_k[1][p, o] = bf16_bits_to_f32(value[b])
        ctx = np.full(B, step + 1, dtype=np.int32)
        r_min, r_max = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx, kmin.copy(), kmax.copy())
        np.testing.assert_array_equal(kmin, r_min, err_msg=f"step {step}: metadata vs rebuild")
        np.testing.assert_array_equal(kmax, r_max, err_msg=f"step {step}: metadata vs rebuild")
    return bt, hist_k, (kc, vc, ks, vs, kmin, kmax)


def test_incremental_equals_from_scratch(oracle_lib):
    """Tokens appended one call at a time with growing magnitudes (the scale
    rises several times per block): the final scale is the smallest power of
    two fitting every token of the block, the codes equal the from-scratch
    cast of x / final scale wherever that value is an E4M3 normal (>= 2^-6),
    and differ by at most one subnormal step (2^-9) elsewhere; the running
    metadata equals the rebuild after every call."""
    rng = np.random.default_rng(12)
    NB, Hkv, D, B, steps = 12, 2, 16, 3, 40
    bt, (hk, hv), (kc, vc, ks, vs, kmin, kmax) = _decode_steps(oracle_lib, rng, NB, Hkv, D, B, steps,
                                                               growth=1.09)
    vnat = v_token_major(vc)
    grew = 0
    for b in range(B):
        for j in range(bt.shape[1]):
            p = bt[b, j]
            n = min(16, steps - 16 * j)
            for h in range(Hkv):
                for codes, hist, sc in ((kc[p, :n, h], hk[p, :n, h], ks[p, h]), (vnat[p, :n, h], hv[p, :n, h],
                                                                                   vs[p, h])):
                    e = fit_exponent(np.abs(hist).max())
                    assert sc == 2.0 ** e
                    grew += fit_exponent(np.abs(hist[0]).max()) < e
                    direct = torch_encode_sat(hist / 2.0 ** e)
                    normal = np.abs(torch_decode(direct)) >= 2.0 ** -6
                    np.testing.assert_array_equal(codes[normal], direct[normal])
                    diff = np.abs(torch_decode(codes) - torch_decode(direct))
                    assert diff.max() <= 2.0 ** -9
    assert grew > 0, "the case should make block scales grow"


def test_restart_resets_scale_and_keeps_other_rows(oracle_lib):
    """A token landing at offset 0 restarts the block: its scale fits that
    token alone (even when the old scale was larger) and the block's other
    rows keep their bytes."""
    rng = np.random.default_rng(13)
    NB, Hkv, D = 3, 2, 16
    kc, vc, ks, vs, kmin, kmax = empty(NB, Hkv, D)
    big = bf16(rng.standard_normal((5, Hkv, D)) * 1000)
    oracle_lib.reshape_and_cache_fp8_block(big, big, kc, vc, np.arange(16, 21, dtype=np.int64), ks, vs,
                                           kmin, kmax)
    assert (ks[1] >= 2.0).all()
    kc0, vn0 = kc.copy(), v_token_major(vc).copy()
    small = bf16(rng.standard_normal((1, Hkv, D)) * 0.1)
    oracle_lib.reshape_and_cache_fp8_block(small, small, kc, vc, np.array([16], dtype=np.int64), ks, vs,
                                           kmin, kmax)
    sf = bf16_bits_to_f32(small).astype(np.float64)
    for h in range(Hkv):
        assert ks[1, h] == 2.0 ** fit_exponent(np.abs(sf[0, h]).max())
        np.testing.assert_array_equal(kc[1, 0, h], torch_encode_sat(sf[0, h] / float(ks[1, h])))
        np.testing.assert_array_equal(kmin[1, h], np.minimum.reduce([kc[1, 0, h]]))
    np.testing.assert_array_equal(kc[1, 1:], kc0[1, 1:])
    np.testing.assert_array_equal(v_token_major(vc)[1, 1:], vn0[1, 1:])


def test_out_of_pool_and_zero_rows(oracle_lib):
    """Slots past the pool are counted and skipped; an all-zero token into an
    empty block takes the floor scale 2^-126 and zero codes."""
    kc, vc, ks, vs, kmin, kmax = empty(2, 1, 16)
    z = bf16(np.zeros((2, 1, 16)))
    assert oracle_lib.reshape_and_cache_fp8_block(z, z, kc, vc, np.array([5, 40], dtype=np.int64), ks, vs,
                                                  kmin, kmax) == 1
    assert ks[0, 0] == 2.0 ** -126 and vs[0, 0] == 2.0 ** -126 and ks[1, 0] == 0.0
    assert (kc == 0).all()


# ---------------------------------------------------- attention and scores


def _block_case(rng, B=3, Hq=6, Hkv=2, D=32, MBS=3):
    NB = B * MBS + 2
    ctx = np.array([MBS * 16, 21, 1][:B], dtype=np.int32)
    bt = rng.permutation(NB)[: B * MBS].astype(np.int32).reshape(B, MBS)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    kc = rng.choice(finite, size=(NB, 16, Hkv, D)).astype(np.uint8)
    vc = rng.choice(finite, size=(NB, Hkv, D, 16)).astype(np.uint8)
    q = bf16(rng.standard_normal((B, Hq, D)))
    ks = (2.0 ** rng.integers(-9, 3, (NB, Hkv))).astype(np.float32)
    vs = (2.0 ** rng.integers(-9, 3, (NB, Hkv))).astype(np.float32)
    return q, kc, vc, ks, vs, bt, ctx


def test_block_attention_equals_bf16_attention_on_exact_values(oracle_lib):
    """Per-block power-of-two scales: every dequantised element is a bf16
    value, so the attention (dense and sparse) equals the bf16 oracle's on
    a cache holding decode(code) * scale[p, h], bit for bit."""
    rng = np.random.default_rng(14)
    q, kc, vc, ks, vs, bt, ctx = _block_case(rng)
    kval = torch_decode(kc) * ks[:, None, :, None]
    vval = torch_decode(v_token_major(vc)) * vs[:, None, :, None]
    kb, vb = bf16(kval), bf16(vval)
    np.testing.assert_array_equal(bf16_bits_to_f32(kb), kval)
    np.testing.assert_array_equal(bf16_bits_to_f32(vb), vval)
    scale = 1 / math.sqrt(32)
    np.testing.assert_array_equal(oracle_lib.attention_fp8(q, kc, vc, ks, vs, bt, ctx, scale),
                                  oracle_lib.paged_attention(q, kb, vb, bt, ctx, scale))
    sel = np.array([[[2, 0], [1, -1]], [[0, 1], [1, 2]], [[0, -1], [-1, -1]]], dtype=np.int32)
    np.testing.assert_array_equal(oracle_lib.attention_fp8(q, kc, vc, ks, vs, bt, ctx, scale, selected=sel),
                                  oracle_lib.sparse_attention(q, kb, vb, bt, ctx, sel, scale))


def test_block_scores_equal_bf16_scores_on_scaled_meta(oracle_lib):
    """The block score with per-block scales equals the (pinned) bf16 score
    on metadata decode(code) * scale[p, h] (exact in bf16), in the plain fp64
    form and in the fp32 kernel order, bit for bit; both differ from the
    per-KV-head form (no scale) by exactly the block's factor."""
    rng = np.random.default_rng(15)
    q, kc, vc, ks, vs, bt, ctx = _block_case(rng)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx)
    bmin = bf16(torch_decode(kmin) * ks[:, :, None])
    bmax = bf16(torch_decode(kmax) * ks[:, :, None])
    BS = 16
    a = oracle_lib.quest_scores_fp8(q, kmin, kmax, bt, ctx, BS, k_bscale=ks)
    np.testing.assert_array_equal(a, oracle_lib.quest_scores(q, bmin, bmax, bt, ctx, BS))
    a32 = oracle_lib.quest_scores_kernel_order_fp8(q, kmin, kmax, bt, ctx, BS, k_bscale=ks)
    np.testing.assert_array_equal(a32, oracle_lib.quest_scores_kernel_order(q, bmin, bmax, bt, ctx, BS))
    plain = oracle_lib.quest_scores_kernel_order_fp8(q, kmin, kmax, bt, ctx, BS)
    B, Hkv, MBS = plain.shape
    fac = np.full_like(plain, np.nan)
    for b in range(B):
        for j in range(MBS):
            fac[b, :, j] = ks[bt[b, j]]
    live = np.isfinite(plain)
    np.testing.assert_array_equal(a32[live], plain[live] * fac[live])


def test_block_score_bounds_every_token(oracle_lib):
    """The block score is at least the group-summed logit q . k of every
    token of the block, with keys dequantised by their block's scale."""
    rng = np.random.default_rng(16)
    q, kc, vc, ks, vs, bt, ctx = _block_case(rng)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx)
    sc = oracle_lib.quest_scores_fp8(q, kmin, kmax, bt, ctx, 16, k_bscale=ks)
    B, Hq, D = q.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    kd = torch_decode(kc)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    for b in range(B):
        for kvh in range(Hkv):
            qs = qf[b, kvh * G:(kvh + 1) * G].sum(axis=0)
            for j in range((ctx[b] + 15) // 16):
                n = min(16, ctx[b] - j * 16)
                p = bt[b, j]
                logits = kd[p, :n, kvh] @ qs * float(ks[p, kvh])
                assert sc[b, kvh, j] >= logits.max() - 1e-9 * (abs(sc[b, kvh, j]) + 1.0)
