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
