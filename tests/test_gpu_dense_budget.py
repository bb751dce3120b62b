"""pa_decode_budget: the dense decode on at most max_ctas CTAs. Parity
against the CPU oracle for budgets from one CTA to more than the GPU has,
the same bytes on a repeated call, and the same bytes as pa_decode when the
budget is at least one CTA per SM."""

import math

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


@pytest.fixture(scope="module")
def case():
    # 6 sequences, one of them empty, one shorter than a block
    ctx = np.array([2900, 0, 1700, 9, 4100, 1300])
    empty = ctx == 0
    ctx = np.where(empty, 300, ctx)
    w = workloads.build_workload("dense_budget", B=6, Hq=28, Hkv=4, D=128, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(2024), topk=16,
                                 scale=1.0 / math.sqrt(128), pool_blocks=int(((ctx + 15) // 16).sum()) + 5)
    w.context_lens[empty] = 0
    w.slot_mapping[empty] = -1
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    return w, dev, ora.dense()


@pytest.mark.parametrize("max_ctas", [1, 5, 37, 100, 0])
def test_dense_budget_matches_the_oracle(case, max_ctas):
    import paged_gqa_decode_reshape_gb300 as pg
    w, dev, want = case
    outs = []
    for _ in range(2):
        out = torch.full_like(dev.out, float("nan"))
        pg.pa_decode_budget(out, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, w.scale, max_ctas, workspace=dev.ws)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close_attention(to_host_f64(outs[0]), want, f"budget {max_ctas}")
    assert pg.pa_workspace_status(dev.ws) == 0


def test_a_budget_of_every_sm_is_pa_decode(case):
    import paged_gqa_decode_reshape_gb300 as pg
    w, dev, _ = case
    sms = torch.cuda.get_device_properties(dev.dev).multi_processor_count
    ref = torch.full_like(dev.out, float("nan"))
    pg.pa_decode(ref, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, w.scale, workspace=dev.ws)
    for budget in (sms, 4 * sms):
        out = torch.full_like(dev.out, float("nan"))
        pg.pa_decode_budget(out, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, w.scale, budget, workspace=dev.ws)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"budget {budget}"


@pytest.mark.parametrize("max_ctas", [1, 37, 0])
def test_fp8_dense_budget_matches_the_oracle(max_ctas):
    """pa_decode_fp8_budget and pa_decode_fp8_block_budget (two-block ring
    items) against the oracle, and equal to the calls without a budget when
    the budget is 0."""
    import paged_gqa_decode_reshape_gb300 as pg
    import oracle
    from tests.test_gpu_fp8 import Fp8Case
    from tests.test_gpu_fp8_block import BlockCase
    w = workloads.make("quest_8k", batch=4, ctx_scale=0.05, topk=6)
    c = Fp8Case(w)
    c.write_step()  # the step's tokens (their slots hold poison until written)
    out = torch.full_like(c.out, float("nan"))
    pg.pa_decode_fp8_budget(out, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, max_ctas, workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens, w.scale)
    assert_close_attention(to_host_f64(out), want, f"fp8 budget {max_ctas}")
    if max_ctas == 0:
        ref = torch.full_like(c.out, float("nan"))
        pg.pa_decode_fp8(ref, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, workspace=c.ws)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    b = BlockCase(w)
    b.write_step()
    outb = torch.full_like(b.out, float("nan"))
    pg.pa_decode_fp8_block_budget(outb, b.q, b.kc, b.vc, b.ks, b.vs, b.bt, b.ctx, w.scale, max_ctas,
                                  workspace=b.ws)
    wantb = oracle.attention_fp8(w.q, b.okc, b.ovc, b.oks, b.ovs, w.block_tables, w.context_lens, w.scale)
    assert_close_attention(to_host_f64(outb), wantb, f"fp8 block budget {max_ctas}")
    assert pg.pa_workspace_status(c.ws) == 0 and pg.pa_workspace_status(b.ws) == 0
