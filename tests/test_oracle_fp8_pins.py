"""Pins for the oracle's 8-bit (E4M3) KV-cache functions, independent of the
oracle's own code: the format's constants, PyTorch's float8_e4m3fn casts (a
library implementation of the same format), brute-force nearest-value search,
numpy min/max, and the already-pinned bf16 oracle functions on caches whose
elements are exactly the dequantised fp8 values."""

import math

import numpy as np
import pytest
import torch

from workloads import bf16_bits_to_f32, f32_to_bf16_bits


def bf16(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def torch_decode(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy().astype(np.float64)


def torch_encode(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def torch_encode_sat(x) -> np.ndarray:
    """Library cast after clamping to +-448 (the saturating reading; NaN kept)."""
    x = np.asarray(x, dtype=np.float32)
    return torch_encode(np.where(np.isnan(x), x, np.clip(x, -448.0, 448.0)))


ALL_CODES = np.arange(256, dtype=np.uint8)

# token order inside a 16-byte row of the 8-bit V layout (the format's definition)
V_ORDER = np.array([0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15])


def v_token_major(vc):
    """[NB, Hkv, D, 16] V codes (rows in V_ORDER) as [NB, 16, Hkv, D]."""
    nat = np.empty_like(vc)
    nat[..., V_ORDER] = vc
    return np.ascontiguousarray(nat.transpose(0, 3, 1, 2))
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


# ------------------------------------------------------------------ codec


def test_e4m3_format_constants(oracle_lib):
    """Values the format fixes: zero, signed zero, smallest subnormal, largest
    subnormal, smallest normal, one, largest finite, NaN."""
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    dec = oracle_lib.e4m3_decode(np.array(list(cases), dtype=np.uint8))
    np.testing.assert_array_equal(dec, np.array(list(cases.values())))
    z = oracle_lib.e4m3_decode(np.array([0x80], dtype=np.uint8))[0]
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert np.isnan(oracle_lib.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_matches_library_on_every_code(oracle_lib):
    ours = oracle_lib.e4m3_decode(ALL_CODES)
    ref = torch_decode(ALL_CODES)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])


def test_e4m3_encode_matches_library_in_range(oracle_lib):
    """Below the 448/480 midpoint the library cast and the oracle agree:
    random magnitudes over every binade, every exact midpoint between
    neighbouring codes (ties to the even mantissa) and their neighbours."""
    rng = np.random.default_rng(1)
    mags = np.exp2(rng.uniform(-13, math.log2(463.9), 20000)).astype(np.float32)
    x = mags * rng.choice([-1.0, 1.0], mags.size).astype(np.float32)
    vals = np.sort(np.unique(torch_decode(FINITE)))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)      # exact in fp32
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    x = np.concatenate([x, mids, -mids, near, -near, vals.astype(np.float32)])
    x = x[np.abs(x) < 464.0]
    np.testing.assert_array_equal(oracle_lib.e4m3_encode(x), torch_encode(x))


def test_e4m3_encode_saturates_and_keeps_nan(oracle_lib):
    x = np.array([448.0, 463.9, 464.0, 470.0, 1e30, np.inf, -470.0, -np.inf, np.nan], dtype=np.float32)
    np.testing.assert_array_equal(oracle_lib.e4m3_encode(x),
                                  np.array([0x7E] * 6 + [0xFE, 0xFE, 0x7F], dtype=np.uint8))


def test_e4m3_encode_is_brute_force_nearest_even(oracle_lib):
    """The code whose value is nearest, found by trying all 254 finite codes;
    a tie takes the even mantissa."""
    rng = np.random.default_rng(2)
    dec = torch_decode(FINITE)
    x = np.concatenate([rng.standard_normal(400) * 4, rng.uniform(-0.02, 0.02, 200),
                        ((dec[:-1] + dec[1:]) / 2)[::3]]).astype(np.float32)
    got = oracle_lib.e4m3_encode(x)
    for xi, g in zip(x, got):
        d = np.abs(dec - float(xi))
        best = FINITE[d == d.min()]
        if best.size > 1:  # tie (or +-0): even mantissa, and the sign of x for zero
            best = best[(best & 1) == 0]
            if best.size > 1:
                best = best[(best >> 7) == (1 if math.copysign(1.0, float(xi)) < 0 else 0)]
        assert g == best[0], (xi, g, best)


# ------------------------------------------------------------- write path


def test_fp8_write_quantises_each_element(oracle_lib):
    """Written rows are the library cast of fl32(x / scale[h]); negative
    slots are skipped and untouched rows keep their bytes."""
    rng = np.random.default_rng(3)
    NB, BS, Hkv, D, T = 5, 16, 3, 16, 9
    kc = rng.integers(0, 256, (NB, BS, Hkv, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (NB, Hkv, D, BS), dtype=np.uint8)
    kc0, vc0 = kc.copy(), vc.copy()
    key = bf16(rng.standard_normal((T, Hkv, D)) * 3)
    value = bf16(rng.standard_normal((T, Hkv, D)) * 3)
    ks = np.array([0.011, 0.0137, 0.02], dtype=np.float32)
    vs = np.array([0.009, 0.031, 0.0077], dtype=np.float32)
    slots = np.array([0, 21, -1, 79, 7, -3, 40, 53, 18], dtype=np.int64)
    assert oracle_lib.reshape_and_cache_fp8(key, value, kc, vc, slots, ks, vs) == 0
    written = np.zeros((NB * BS,), dtype=bool)
    vnat, vnat0 = v_token_major(vc).reshape(NB * BS, -1), v_token_major(vc0).reshape(NB * BS, -1)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        written[s] = True
        kq = torch_encode_sat(bf16_bits_to_f32(key[t]) / ks[:, None])
        vq = torch_encode_sat(bf16_bits_to_f32(value[t]) / vs[:, None])
        np.testing.assert_array_equal(kc.reshape(NB * BS, Hkv, D)[s], kq)
        np.testing.assert_array_equal(vnat[s].reshape(Hkv, D), vq)
    np.testing.assert_array_equal(kc.reshape(NB * BS, -1)[~written], kc0.reshape(NB * BS, -1)[~written])
    np.testing.assert_array_equal(vnat[~written], vnat0[~written])


# --------------------------------------------------------------- metadata


def _random_fp8_cache(rng, NB, BS, Hkv, D):
    return rng.choice(FINITE, size=(NB, BS, Hkv, D)).astype(np.uint8)


def test_fp8_rebuild_meta_is_numeric_min_max(oracle_lib):
    rng = np.random.default_rng(4)
    B, Hkv, D, BS = 3, 2, 16, 4
    ctx = np.array([5, 12, 1], dtype=np.int32)
    MBS = 3
    NB = B * MBS
    bt = rng.permutation(NB).astype(np.int32).reshape(B, MBS)
    kc = _random_fp8_cache(rng, NB, BS, Hkv, D)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx)
    dec = torch_decode(kc)
    for b in range(B):
        for j in range((ctx[b] + BS - 1) // BS):
            p = bt[b, j]
            n = min(BS, ctx[b] - j * BS)
            np.testing.assert_array_equal(torch_decode(kmin[p]), dec[p, :n].min(axis=0))
            np.testing.assert_array_equal(torch_decode(kmax[p]), dec[p, :n].max(axis=0))


def test_fp8_incremental_meta_equals_rebuild(oracle_lib):
    """One new token per sequence per step, quantised into the cache and
    folded into the metadata: the running metadata equals the rebuild."""
    rng = np.random.default_rng(5)
    B, Hkv, D, BS, steps = 3, 2, 16, 16, 11
    ctx = np.array([1, 13, 30])
    MBS = (int(ctx.max()) + steps + BS - 1) // BS
    NB = B * MBS
    bt = rng.permutation(NB).astype(np.int32).reshape(B, MBS)
    kc = _random_fp8_cache(rng, NB, BS, Hkv, D)
    vc = np.ascontiguousarray(kc.transpose(0, 2, 3, 1))
    ks = np.array([0.013, 0.021], dtype=np.float32)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx.astype(np.int32))
    for _ in range(steps):
        key = bf16(rng.standard_normal((B, Hkv, D)) * 2)
        slots = np.array([bt[b, ctx[b] // BS] * BS + ctx[b] % BS for b in range(B)], dtype=np.int64)
        oracle_lib.reshape_and_cache_fp8(key, key, kc, vc, slots, ks, ks)
        oracle_lib.quest_update_meta_fp8(kmin, kmax, key, slots, ks, BS)
        ctx += 1
        r_min, r_max = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx.astype(np.int32),
                                                         kmin.copy(), kmax.copy())
        np.testing.assert_array_equal(kmin, r_min)
        np.testing.assert_array_equal(kmax, r_max)


# -------------------------------------------------------------- attention


def _case(rng, B=3, Hq=6, Hkv=2, D=32, BS=16, MBS=3):
    NB = B * MBS + 2
    ctx = np.array([MBS * BS, 21, 1][:B], dtype=np.int32)
    bt = rng.permutation(NB)[: B * MBS].astype(np.int32).reshape(B, MBS)
    kc = _random_fp8_cache(rng, NB, BS, Hkv, D)
    vc = np.ascontiguousarray(_random_fp8_cache(rng, NB, BS, Hkv, D).transpose(0, 2, 3, 1))
    q = bf16(rng.standard_normal((B, Hq, D)))
    return q, kc, vc, bt, ctx


def test_fp8_attention_equals_bf16_attention_on_exact_values(oracle_lib):
    """With power-of-two scales every dequantised element is a bf16 value:
    the fp8 attention (dense and sparse) equals the bf16 oracle's on a cache
    holding those values, bit for bit."""
    rng = np.random.default_rng(6)
    q, kc, vc, bt, ctx = _case(rng)
    ks = np.array([2.0 ** -5, 2.0 ** -3], dtype=np.float32)
    vs = np.array([2.0 ** -4, 2.0 ** 1], dtype=np.float32)
    kb = bf16(torch_decode(kc) * ks[None, None, :, None])
    vb = bf16(torch_decode(v_token_major(vc)) * vs[None, None, :, None])
    np.testing.assert_array_equal(bf16_bits_to_f32(kb), torch_decode(kc) * ks[None, None, :, None])
    scale = 1 / math.sqrt(32)
    a = oracle_lib.attention_fp8(q, kc, vc, ks, vs, bt, ctx, scale)
    b = oracle_lib.paged_attention(q, kb, vb, bt, ctx, scale)
    np.testing.assert_array_equal(a, b)
    sel = np.array([[[2, 0], [1, -1]], [[0, 1], [1, 2]], [[0, -1], [-1, -1]]], dtype=np.int32)
    a = oracle_lib.attention_fp8(q, kc, vc, ks, vs, bt, ctx, scale, selected=sel)
    b = oracle_lib.sparse_attention(q, kb, vb, bt, ctx, sel, scale)
    np.testing.assert_array_equal(a, b)


def test_fp8_attention_brute_force_any_scale(oracle_lib):
    """Explicit softmax over the dequantised tokens (library decode times the
    head's scale) for arbitrary scales."""
    rng = np.random.default_rng(7)
    q, kc, vc, bt, ctx = _case(rng)
    ks = np.array([0.0173, 0.0091], dtype=np.float32)
    vs = np.array([0.033, 0.0121], dtype=np.float32)
    scale = 0.21
    got = oracle_lib.attention_fp8(q, kc, vc, ks, vs, bt, ctx, scale)
    B, Hq, D = q.shape
    BS, Hkv, G = kc.shape[1], kc.shape[2], Hq // kc.shape[2]
    kd, vd = torch_decode(kc), torch_decode(v_token_major(vc))
    for b in range(B):
        for h in range(Hq):
            kvh = h // G
            n = int(ctx[b])
            K = np.stack([kd[bt[b, t // BS], t % BS, kvh] for t in range(n)]) * float(ks[kvh])
            V = np.stack([vd[bt[b, t // BS], t % BS, kvh] for t in range(n)]) * float(vs[kvh])
            s = scale * (K @ bf16_bits_to_f32(q[b, h]).astype(np.float64))
            p = np.exp(s - s.max())
            np.testing.assert_allclose(got[b, h], p @ V / p.sum(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ Quest score


def test_fp8_scores_equal_bf16_scores_on_decoded_meta(oracle_lib):
    """Decoded E4M3 metadata is exactly representable in bf16, so the fp8
    score equals the (pinned) bf16 score on those values, bit for bit."""
    rng = np.random.default_rng(8)
    q, kc, vc, bt, ctx = _case(rng)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx)
    bmin, bmax = bf16(torch_decode(kmin)), bf16(torch_decode(kmax))
    a = oracle_lib.quest_scores_kernel_order_fp8(q, kmin, kmax, bt, ctx, kc.shape[1])
    b = oracle_lib.quest_scores_kernel_order(q, bmin, bmax, bt, ctx, kc.shape[1])
    np.testing.assert_array_equal(a, b)
    a = oracle_lib.quest_scores_fp8(q, kmin, kmax, bt, ctx, kc.shape[1])
    b = oracle_lib.quest_scores(q, bmin, bmax, bt, ctx, kc.shape[1])
    np.testing.assert_array_equal(a, b)


def test_fp8_score_bounds_every_token(oracle_lib):
    """score * scale[kvh] >= the group-summed logit q . k of every token of
    the block (dequantised keys), up to fp32 rounding of the score."""
    rng = np.random.default_rng(9)
    q, kc, vc, bt, ctx = _case(rng)
    ks = np.array([0.02, 0.007], dtype=np.float32)
    kmin, kmax = oracle_lib.quest_rebuild_meta_fp8(kc, bt, ctx)
    sc = oracle_lib.quest_scores_fp8(q, kmin, kmax, bt, ctx, kc.shape[1])
    sk = oracle_lib.quest_scores_kernel_order_fp8(q, kmin, kmax, bt, ctx, kc.shape[1])
    B, Hq, D = q.shape
    BS, Hkv = kc.shape[1], kc.shape[2]
    G = Hq // Hkv
    kd = torch_decode(kc)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    for b in range(B):
        for kvh in range(Hkv):
            qs = qf[b, kvh * G:(kvh + 1) * G].sum(axis=0)
            for j in range((ctx[b] + BS - 1) // BS):
                n = min(BS, ctx[b] - j * BS)
                logits = kd[bt[b, j], :n, kvh] @ qs * ks[kvh]
                bound = float(sc[b, kvh, j]) * float(ks[kvh])
                assert bound >= logits.max() - 1e-9 * (abs(bound) + 1.0)
                bound = float(sk[b, kvh, j]) * float(ks[kvh])
                assert bound >= logits.max() - 1e-5 * (abs(bound) + 1.0)
