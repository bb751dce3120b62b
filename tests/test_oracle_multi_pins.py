"""Pins for the oracle's multi-token query rows (right-aligned causal masks):
single-token rows reduce to the pinned dense decode; PyTorch's
scaled_dot_product_attention with a torch.tril causal mask on contiguous
K/V; rows past their sequence's context give zeros."""

import numpy as np
import torch

from tests.test_oracle_pins import bf16, contiguous_paged, rand_bf16
from workloads import bf16_bits_to_f32


def _cu(q_lens):
    return np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)


def test_single_token_rows_equal_dense(oracle_lib):
    rng = np.random.default_rng(31)
    B, Hq, Hkv, D, BS = 4, 6, 2, 32, 4
    ctx = np.array([9, 1, 16, 5], dtype=np.int32)
    _, _, kc, vc, bt, _ = contiguous_paged(rng, B, Hkv, D, BS, ctx)
    q = rand_bf16(rng, (B, Hq, D))
    a = oracle_lib.paged_attention_multi(q, kc, vc, bt, _cu(np.ones(B, int)), ctx, 0.3)
    b = oracle_lib.paged_attention(q, kc, vc, bt, ctx, 0.3)
    np.testing.assert_array_equal(a, b)


def test_multi_rows_match_sdpa_with_tril_mask(oracle_lib):
    """Row i of a sequence with q_len new tokens and context ctx sees keys
    0 .. ctx - q_len + i: the lower triangle of the [q_len, ctx] score
    matrix, right-aligned (torch.tril with diagonal ctx - q_len)."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, D, BS = 3, 8, 2, 16, 4
    ctx = np.array([11, 6, 20], dtype=np.int32)
    q_lens = np.array([3, 6, 1])
    Kc, Vc, kc, vc, bt, _ = contiguous_paged(rng, B, Hkv, D, BS, ctx)
    cu = _cu(q_lens)
    q = rand_bf16(rng, (int(cu[-1]), Hq, D))
    scale = 0.25
    got = oracle_lib.paged_attention_multi(q, kc, vc, bt, cu, ctx, scale)
    for b in range(B):
        n, ql = int(ctx[b]), int(q_lens[b])
        qq = torch.from_numpy(bf16_bits_to_f32(q[cu[b]:cu[b + 1]]).astype(np.float64)).permute(1, 0, 2)
        kk = torch.from_numpy(bf16_bits_to_f32(Kc[b, :n]).astype(np.float64)).permute(1, 0, 2)
        vv = torch.from_numpy(bf16_bits_to_f32(Vc[b, :n]).astype(np.float64)).permute(1, 0, 2)
        mask = torch.ones(ql, n, dtype=torch.bool).tril(diagonal=n - ql)
        o = torch.nn.functional.scaled_dot_product_attention(qq[None], kk[None], vv[None], attn_mask=mask,
                                                             scale=scale, enable_gqa=True)
        np.testing.assert_allclose(got[cu[b]:cu[b + 1]], o[0].permute(1, 0, 2).numpy(), rtol=1e-12,
                                   atol=1e-13)


def test_rows_before_the_context_are_zero_and_empty_sequences_skip(oracle_lib):
    """q_len > ctx: the first q_len - ctx rows have no key to see (zero
    output); a sequence with q_len 0 owns no row."""
    rng = np.random.default_rng(33)
    B, Hq, Hkv, D, BS = 3, 4, 1, 16, 4
    ctx = np.array([2, 7, 5], dtype=np.int32)
    q_lens = np.array([5, 0, 2])
    _, _, kc, vc, bt, _ = contiguous_paged(rng, B, Hkv, D, BS, ctx)
    cu = _cu(q_lens)
    q = rand_bf16(rng, (int(cu[-1]), Hq, D))
    got = oracle_lib.paged_attention_multi(q, kc, vc, bt, cu, ctx, 0.5)
    assert (got[:3] == 0).all()
    assert np.abs(got[3:5]).sum() > 0
    # the last row of sequence 0 sees exactly the whole context: it equals
    # single-token decode of that sequence
    one = oracle_lib.paged_attention(q[4:5], kc, vc, bt[:1], ctx[:1], 0.5)
    np.testing.assert_array_equal(got[4], one[0])
