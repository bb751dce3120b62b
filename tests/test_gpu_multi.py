"""Parity of multi-token query rows (pa_decode_multi, right-aligned causal
masks) against the CPU oracle, and its reduction to pa_decode."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import (DeviceStep, assert_close_attention, gather_rows, to_dev_bf16,
                            to_host_f64)
from workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def multi_case(w, max_qlen, seed, force_short=True):
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(0, max_qlen + 1, w.B)
    if force_short:
        # a sequence with more query rows than context (leading rows see nothing)
        b = int(np.argmin(w.context_lens))
        q_lens[b] = max(q_lens[b], int(min(w.context_lens[b], max_qlen)) + 2)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = f32_to_bf16_bits(rng.standard_normal((int(cu[-1]), w.Hq, w.D)).astype(np.float32))
    return q, cu


def run_multi(w, q, cu, rows=None):
    import paged_gqa_decode_reshape_gb300 as pg
    dev = DeviceStep(w)
    d = dev.dev
    qd = to_dev_bf16(q, d)
    out = torch.empty_like(qd)
    cud = torch.from_numpy(cu).to(d)
    ws = torch.zeros(pg.pa_decode_multi_workspace_size(max(q.shape[0], 1), w.Hq, w.Hkv, w.D), dtype=torch.uint8,
                     device=d)
    pg.pa_decode_multi(out, qd, dev.kc, dev.vc, dev.bt, cud, dev.ctx, w.scale, workspace=ws)
    want = oracle.paged_attention_multi(q, w.key_cache, w.value_cache, w.block_tables, cu, w.context_lens,
                                        w.scale, rows=rows)
    got = to_host_f64(out)
    assert pg.pa_workspace_status(ws) == 0
    return (got if rows is None else gather_rows(got, rows)), want, got


@pytest.mark.parametrize("name,kw,max_qlen", [
    ("quest_8k", dict(batch=4, ctx_scale=0.05), 8),
    ("mixed_b128", dict(batch=24, ctx_scale=0.02), 5),
    ("long_40k", dict(batch=2, ctx_scale=0.02), 16),
    ("tiny", {}, 3),
])
def test_multi_rows_small_elementwise(name, kw, max_qlen):
    w = workloads.make(name, poison=False, **kw)
    q, cu = multi_case(w, max_qlen, seed=7)
    got, want, full = run_multi(w, q, cu)
    assert_close_attention(got, want, f"{name} multi q_len<={max_qlen}")
    # rows that see no key are exactly zero
    for b in range(w.B):
        ql = int(cu[b + 1] - cu[b])
        dead = max(0, ql - int(w.context_lens[b]))
        assert (full[cu[b]:cu[b] + dead] == 0).all()


def test_multi_many_rows_sampled():
    """The maximum row count: 2048 query rows (256 sequences x 8), sampled rows."""
    w = workloads.make("mixed_b128", poison=False, batch=256, ctx_scale=0.25)
    rng = np.random.default_rng(8)
    q_lens = np.full(w.B, 8)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    assert cu[-1] == 2048
    q = f32_to_bf16_bits(rng.standard_normal((2048, w.Hq, w.D)).astype(np.float32))
    rows = np.stack([rng.integers(0, 2048, 64), rng.integers(0, w.Hq, 64)], axis=1).astype(np.int32)
    got, want, _ = run_multi(w, q, cu, rows=rows)
    assert_close_attention(got, want, "multi 2048 rows (sampled)")


def test_single_token_rows_match_dense_oracle():
    """One query row per sequence is plain decode: the multi-row kernel (one
    consumer warp streaming each sequence) matches the dense oracle."""
    w = workloads.make("quest_8k", poison=False, batch=8, ctx_scale=0.1)
    cu = np.arange(w.B + 1, dtype=np.int32)
    got, _, _ = run_multi(w, w.q, cu)
    want = oracle.paged_attention(w.q, w.key_cache, w.value_cache, w.block_tables, w.context_lens, w.scale)
    assert_close_attention(got, want, "multi, one row per sequence")
