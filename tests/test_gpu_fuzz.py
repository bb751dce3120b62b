"""Seeded random shapes through every decode path against the CPU oracle:
batch, group size, KV heads, head_dim, context lengths (empty sequences and
sequences shorter than a block included), topk (odd values included) and
CTA budgets drawn per case. Each case runs the whole step (bf16), the fused
Quest decode under its budgets, the dense decode under a budget, rows of
several query tokens, and, for head_dim 128, the 8-bit steps with per-head
and per-block scales."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64
from tests.test_gpu_fp8 import run_fp8_compare
from tests.test_gpu_fp8_block import run_block_compare
from tests.test_gpu_multi import multi_case, run_multi
from tests.test_gpu_parity import run_full_compare
from tests.test_gpu_quest_decode import run_compare

pytestmark = pytest.mark.gpu

N_CASES = 32


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def draw_case(i: int, poison: bool = True):
    """Case i: a seeded random shape (the same on every run)."""
    rng = np.random.default_rng(9000 + i)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 7, 8]))
    while Hkv * G > 32:
        G = max(1, G // 2)
    D = 128 if i % 3 else 64
    B = int(rng.integers(1, 13))
    ctx = rng.integers(1, int(rng.choice([600, 2600, 9000, 20000])), size=B)
    short = rng.random(B) < 0.2
    ctx[short] = rng.integers(1, 17, size=int(short.sum()))  # within one block
    empty = rng.random(B) < 0.15
    topk = int(rng.integers(1, 81))
    seed = np.random.SeedSequence(77 + i)
    w = workloads.build_workload(f"fuzz{i}", B=B, Hq=G * Hkv, Hkv=Hkv, D=D, BS=16, ctx=ctx,
                                 seed_seq=seed, topk=topk, scale=1.0 / math.sqrt(D),
                                 pool_blocks=int(((ctx + 15) // 16).sum()) + int(rng.integers(0, 9)),
                                 poison=poison)
    w.context_lens[empty] = 0
    w.slot_mapping[empty] = -1
    budgets = (0, int(rng.integers(1, 9)), int(rng.integers(9, 160)))
    return w, budgets


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shapes(i):
    import paged_gqa_decode_reshape_gb300 as pg
    w, budgets = draw_case(i)
    # the whole bf16 step: caches, metadata, scores and selection bit-exact,
    # attention within tolerance
    run_full_compare(w)
    # the fused Quest decode, under the drawn CTA budgets
    run_compare(w, budgets=budgets)
    # the dense decode under a CTA budget
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    out = torch.full_like(dev.out, float("nan"))
    pg.pa_decode_budget(out, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, w.scale, budgets[2], workspace=dev.ws)
    assert_close_attention(to_host_f64(out), ora.dense(), f"fuzz {i} dense budget {budgets[2]}")
    # rows of several query tokens (a pool without poisoned slots: no write)
    wm, _ = draw_case(i, poison=False)
    q, cu = multi_case(wm, max_qlen=1 + i % 6, seed=i)
    got, want, _ = run_multi(wm, q, cu)
    assert_close_attention(got, want, f"fuzz {i} multi")
    # the 8-bit steps (head_dim 128 only); per-block scales want a pool with
    # enough (block, KV head) pairs to carry several distinct scales
    if w.D == 128:
        c = run_fp8_compare(w)
        want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens,
                                    w.scale)
        out = torch.full_like(c.out, float("nan"))
        pg.pa_decode_fp8_budget(out, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, budgets[1],
                                workspace=c.ws)
        assert_close_attention(to_host_f64(out), want, f"fuzz {i} fp8 dense budget {budgets[1]}")
        # the fused 8-bit Quest decode under a budget: the selection of the
        # separate call and the bytes of the sparse call on the same grid
        qws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS), dtype=torch.uint8,
                          device=c.q.device)
        fsel = torch.full_like(c.sel, -7)
        pg.quest_decode_fp8(out, fsel, c.q, c.kmin, c.kmax, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.topk,
                            w.scale, max_ctas=budgets[2], workspace=qws)
        assert torch.equal(fsel, c.sel)
        ref = torch.full_like(c.out, float("nan"))
        pg.quest_sparse_decode_fp8_budget(ref, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, fsel, w.scale,
                                          budgets[2], workspace=c.ws)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert pg.pa_workspace_status(qws) == 0 and pg.pa_workspace_status(c.ws) == 0
        if w.NB * w.Hkv >= 64:
            b = run_block_compare(w)
            want = oracle.attention_fp8(w.q, b.okc, b.ovc, b.oks, b.ovs, w.block_tables, w.context_lens,
                                        w.scale)
            out = torch.full_like(b.out, float("nan"))
            pg.pa_decode_fp8_block_budget(out, b.q, b.kc, b.vc, b.ks, b.vs, b.bt, b.ctx, w.scale,
                                          budgets[2], workspace=b.ws)
            assert_close_attention(to_host_f64(out), want, f"fuzz {i} block fp8 dense budget {budgets[2]}")
