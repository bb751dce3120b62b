"""Sparse decode of small selections: the grid follows the (sequence, KV
head) segments, each cut into equal pieces (one CTA each, their number set
by the CTA budget) that are merged with the split-KV combine. Parity against the CPU oracle (bf16
and 8-bit caches), with an empty sequence and a sequence shorter than the
selection (-1 padding, so some pieces hold invalid entries) in the batch."""

import math

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64
from tests.test_gpu_fp8 import run_fp8_compare
from tests.test_gpu_parity import run_full_compare

pytestmark = pytest.mark.gpu

# name: (B, Hq, Hkv, topk, context lengths); with the default CTA budget (half
# the SMs, as these segments fit in it) and at least 16 items per piece the
# segments split into 4, 4, 8 and 8 pieces (fewer under a smaller budget)
CASES = {
    "pieces2": (4, 28, 4, 64, [0, 700, 1500, 2200]),
    "pieces4": (4, 28, 4, 128, [2500, 0, 1000, 3000]),
    "pieces4_group8": (4, 16, 2, 128, [2100, 2600, 900, 0]),
    "pieces8": (2, 28, 4, 192, [3500, 1200]),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def make_case(name):
    B, Hq, Hkv, topk, ctx = CASES[name]
    ctx = np.array(ctx)
    empty = ctx == 0
    ctx = np.where(empty, 300, ctx)   # drawn with tokens, then emptied (no new token either)
    w = workloads.build_workload(name, B=B, Hq=Hq, Hkv=Hkv, D=128, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(len(name) * 7 + topk), topk=topk,
                                 scale=1.0 / math.sqrt(128), pool_blocks=int(((ctx + 15) // 16).sum()) + 7)
    assert w.slot_mapping.shape == (B,)   # one new token per sequence
    w.context_lens[empty] = 0
    w.slot_mapping[empty] = -1
    return w


@pytest.mark.parametrize("name", list(CASES))
def test_segment_pieces_whole_step(name):
    """The whole step (selection bit-exact, sparse attention on it)."""
    run_full_compare(make_case(name))


@pytest.mark.parametrize("name", list(CASES))
def test_segment_pieces_fixed_selection(name):
    """A seeded selection that is not the top-K, with entries past the
    sequence and an all-invalid segment mixed in."""
    w = make_case(name)
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    sel = workloads.random_selection(w, seed=3)
    nb = w.num_blocks()
    full = int(np.argmax(nb))
    sel[full, 0, 1] = 10_000          # past the sequence: ignored
    sel[full, w.Hkv - 1, :] = -1      # nothing selected: zero output for that group
    got = to_host_f64(dev.sparse(torch.from_numpy(sel).to(dev.dev)))
    assert_close_attention(got, ora.sparse(sel), f"{name} fixed selection")
    G = w.Hq // w.Hkv
    assert (got[full, (w.Hkv - 1) * G:] == 0).all()
    for b in np.flatnonzero(w.context_lens == 0):
        assert (got[b] == 0).all()
    ws = dev.ws.cpu().numpy()
    assert (ws[: 256 + w.B * w.Hkv * 4] == 0).all()


@pytest.mark.parametrize("name", ["pieces2", "pieces8"])
def test_segment_pieces_fp8(name):
    run_fp8_compare(make_case(name))


@pytest.mark.parametrize("max_ctas", [1, 3, 16, 64, 0])
@pytest.mark.parametrize("name", ["pieces4", "pieces8"])
def test_segment_pieces_under_a_cta_budget(name, max_ctas):
    """quest_sparse_decode_budget: one CTA for everything, a few CTAs holding
    several segments each, and segments cut into fewer pieces than the whole
    GPU allows; each result within tolerance of the oracle and the same on a
    second call."""
    import paged_gqa_decode_reshape_gb300 as pg
    w = make_case(name)
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    sel_h = workloads.random_selection(w, seed=4)
    sel = torch.from_numpy(sel_h).to(dev.dev)
    outs = []
    for _ in range(2):
        out = torch.full_like(dev.out, float("nan"))
        pg.quest_sparse_decode_budget(out, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, sel, w.scale, max_ctas,
                                      workspace=dev.ws)
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close_attention(to_host_f64(outs[0]), ora.sparse(sel_h), f"{name} budget {max_ctas}")
    assert pg.pa_workspace_status(dev.ws) == 0
