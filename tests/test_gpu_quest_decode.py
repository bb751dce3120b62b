"""quest_decode: the block scores, then one launch whose CTAs select the top-K
blocks of their own segments and attend over them.

Against the CPU oracle: the selection bit for bit (the kernel-order scores'
top-K) and against the top-K of the plain fp64 scores, the output within the
attention tolerances. Against the separate calls: the same selection as
quest_select_topk, and the same output bytes as quest_sparse_decode_budget on
that selection with the same CTA cap. Small variants of every workload, the
full sizes, an 8-bit cache, empty sequences, and rows too long for the
shared-memory key cache.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": ("tiny", {}),
    "dense_small": ("dense_b32", dict(batch=6, ctx_scale=0.05, topk=8)),
    "quest_small": ("quest_8k", dict(batch=4, ctx_scale=0.05, topk=6)),
    "long_small": ("long_40k", dict(batch=2, ctx_scale=0.02, topk=16)),
    "mixed_small": ("mixed_b128", dict(batch=16, ctx_scale=0.02, topk=8)),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def run_compare(w, budgets=(0,)):
    import paged_gqa_decode_reshape_gb300 as pg
    from paged_gqa_decode_reshape_gb300 import quest_rebuild_meta
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    quest_rebuild_meta(dev.kmin, dev.kmax, dev.kc, dev.bt, dev.ctx)
    kmin, kmax = ora.rebuild_meta()
    want_sel = ora.select(kmin, kmax)
    want_out = ora.sparse(want_sel)
    ws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS), dtype=torch.uint8,
                     device=dev.dev)
    for budget in budgets:
        sel = torch.full((w.B, w.Hkv, w.topk), -7, dtype=torch.int32, device=dev.dev)
        out = torch.full_like(dev.out, float("nan"))
        pg.quest_decode(out, sel, dev.q, dev.kmin, dev.kmax, dev.kc, dev.vc, dev.bt, dev.ctx, w.topk, w.scale,
                        max_ctas=budget, workspace=ws)
        got_sel = sel.cpu().numpy()
        np.testing.assert_array_equal(got_sel, want_sel)
        ora.check_plain(got_sel, kmin, kmax, what=f"{w.name} quest_decode selection vs plain scores")
        assert_close_attention(to_host_f64(out), want_out, f"{w.name} quest_decode (max_ctas {budget})")
        # the same bytes as the separate sparse call on that selection and grid
        ref = torch.full_like(dev.out, float("nan"))
        pg.quest_sparse_decode_budget(ref, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, sel, w.scale, budget,
                                      workspace=dev.ws)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"budget {budget}"
        assert pg.pa_workspace_status(ws) == 0
    return dev


@pytest.mark.parametrize("case", list(SMALL))
def test_small(case):
    name, kw = SMALL[case]
    run_compare(workloads.make(name, **kw), budgets=(0, 3, 64))


@pytest.mark.parametrize("name", ["dense_b32", "quest_8k", "long_40k", "mixed_b128"])
def test_full_size(name):
    w = workloads.make(name)
    run_compare(w, budgets=(0, 76))


def test_empty_and_short_sequences():
    """ctx = 0 (a -1 row, zero output), sequences with fewer blocks than topk
    (all their blocks, then -1), and all-tied scores (lowest indices)."""
    ctx = np.array([0, 40, 5000, 0, 16 * 33])
    w = workloads.build_workload("edges", B=len(ctx), Hq=8, Hkv=2, D=128, BS=16, ctx=np.maximum(ctx, 100),
                                 seed_seq=np.random.SeedSequence(31), topk=32, scale=1.0 / math.sqrt(128))
    w.context_lens[ctx == 0] = 0
    w.slot_mapping[ctx == 0] = -1
    dev = run_compare(w, budgets=(0, 2))
    import paged_gqa_decode_reshape_gb300 as pg
    # constant metadata: every score of a segment tied
    dev.kmin.fill_(0.5)
    dev.kmax.fill_(0.5)
    sel = torch.empty((w.B, w.Hkv, w.topk), dtype=torch.int32, device=dev.dev)
    out = torch.empty_like(dev.out)
    pg.quest_decode(out, sel, dev.q, dev.kmin, dev.kmax, dev.kc, dev.vc, dev.bt, dev.ctx, w.topk, w.scale)
    nb = w.num_blocks()
    got = sel.cpu().numpy()
    for b in range(w.B):
        want = np.r_[np.arange(min(nb[b], w.topk)), -np.ones(max(w.topk - nb[b], 0))].astype(np.int32)
        assert (got[b] == want).all()


def test_rows_longer_than_the_key_cache():
    """A sequence with more blocks than the CTA's shared-memory key cache
    holds (49,160 blocks): its keys are read from L2 on every pass."""
    ctx = np.array([49160 * 16 - 5, 3000])
    w = workloads.build_workload("long787k", B=2, Hq=2, Hkv=1, D=64, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(787), topk=48, scale=1.0 / math.sqrt(64),
                                 pool_blocks=int(((ctx + 15) // 16).sum()) + 3, poison=False)
    run_compare(w, budgets=(0,))


@pytest.mark.parametrize("topk,max_ctas", [(24, 0), (23, 0), (23, 5)])
def test_fp8_cache(topk, max_ctas):
    """The 8-bit cache (two blocks per ring item): an odd topk leaves a
    segment's last item one entry, and a small CTA budget puts several
    segments, and ranges that start mid-segment, in one CTA."""
    import paged_gqa_decode_reshape_gb300 as pg
    from tests.test_gpu_fp8 import Fp8Case
    w = workloads.make("quest_8k", batch=4, ctx_scale=0.25, topk=topk)
    c = Fp8Case(w)
    kmin, kmax = c.write_step()
    want_sel = oracle.quest_select_kernel_order_fp8(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS,
                                                    w.topk)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens, w.scale,
                                selected=want_sel)
    ws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS), dtype=torch.uint8,
                     device=c.q.device)
    sel = torch.empty((w.B, w.Hkv, w.topk), dtype=torch.int32, device=c.q.device)
    out = torch.empty_like(c.out)
    pg.quest_decode_fp8(out, sel, c.q, c.kmin, c.kmax, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.topk, w.scale,
                        max_ctas=max_ctas, workspace=ws)
    np.testing.assert_array_equal(sel.cpu().numpy(), want_sel)
    assert_close_attention(to_host_f64(out), want, "fp8 quest_decode")
    assert pg.pa_workspace_status(ws) == 0
