"""A whole decode step -- the fused write path, dense decode, Quest selection
and Quest sparse decode -- captured in one CUDA graph. Replaying the graph
must give the same bytes as calling the entry points one by one: caches,
metadata, both attention outputs and the selection. The step launches with
programmatic dependent launch, so the capture also records those edges. The
replayed results are also checked against the CPU oracle."""

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64, to_host_u16

pytestmark = pytest.mark.gpu

CASES = {
    "quest_small": ("quest_8k", dict(batch=4, ctx_scale=0.05, topk=6)),
    "mixed_small": ("mixed_b128", dict(batch=16, ctx_scale=0.02, topk=8)),
    "quest_8k": ("quest_8k", {}),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def _calls(dev: DeviceStep):
    import paged_gqa_decode_reshape_gb300 as pg
    w = dev.w
    return [
        lambda: pg.quest_reshape_and_cache(dev.key, dev.value, dev.kc, dev.vc, dev.kmin, dev.kmax,
                                           dev.slots),
        lambda: pg.pa_decode(dev.out, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, w.scale, workspace=dev.ws),
        lambda: pg.quest_select_topk(dev.sel, dev.q, dev.kmin, dev.kmax, dev.bt, dev.ctx, w.BS,
                                     workspace=dev.sel_ws),
        lambda: pg.quest_sparse_decode(dev.out_sparse, dev.q, dev.kc, dev.vc, dev.bt, dev.ctx, dev.sel,
                                       w.scale, workspace=dev.ws),
    ]


def _state(dev):
    return [dev.kc, dev.vc, dev.kmin, dev.kmax]


def _outputs(dev):
    return _state(dev) + [dev.out, dev.out_sparse, dev.sel]


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _reset(dev, s0):
    """Put the cache and metadata back to the pre-step state and fill the
    outputs with garbage, so every byte compared was written by the step."""
    for t, s in zip(_state(dev), s0):
        t.copy_(s)
    dev.out.view(torch.int16).fill_(0x7FC1)
    dev.out_sparse.view(torch.int16).fill_(0x7FC1)
    dev.sel.fill_(-7)


def _check_against_oracle(dev, w):
    """The replayed step's results against the CPU oracle run on the same
    pre-step state: caches and metadata byte for byte, the selection bit for
    bit (and against the plain score's top-K), both attention outputs within
    the tolerances."""
    import oracle
    ora = OracleStep(w)
    pre_ctx = (w.context_lens - 1).clip(0).astype(np.int32)
    kmin, kmax = oracle.quest_rebuild_meta(ora.kc, w.block_tables, pre_ctx)
    ora.reshape()
    oracle.quest_update_meta(kmin, kmax, w.key, w.slot_mapping, w.BS)
    np.testing.assert_array_equal(to_host_u16(dev.kc), ora.kc)
    np.testing.assert_array_equal(to_host_u16(dev.vc), ora.vc)
    np.testing.assert_array_equal(to_host_u16(dev.kmin), kmin)
    np.testing.assert_array_equal(to_host_u16(dev.kmax), kmax)
    sel = dev.sel.cpu().numpy()
    np.testing.assert_array_equal(sel, ora.select(kmin, kmax))
    ora.check_plain(sel, kmin, kmax, what=f"{w.name} replayed selection vs plain scores")
    assert_close_attention(to_host_f64(dev.out), ora.dense(), f"{w.name} replayed dense")
    assert_close_attention(to_host_f64(dev.out_sparse), ora.sparse(sel), f"{w.name} replayed sparse")


@pytest.mark.parametrize("case", list(CASES))
def test_graph_replay_is_bit_identical_to_eager(case):
    from paged_gqa_decode_reshape_gb300 import pa_workspace_status, quest_rebuild_meta
    name, kw = CASES[case]
    w = workloads.make(name, **kw)
    dev = DeviceStep(w)
    # metadata of the cache as it stood before this step's new tokens
    pre_ctx = torch.from_numpy((w.context_lens - 1).clip(0).astype(np.int32)).to(dev.dev)
    quest_rebuild_meta(dev.kmin, dev.kmax, dev.kc, dev.bt, pre_ctx)
    torch.cuda.synchronize()
    s0 = [t.clone() for t in _state(dev)]
    calls = _calls(dev)

    _reset(dev, s0)
    for c in calls:
        c()
    torch.cuda.synchronize()
    eager = [_bits(t).clone() for t in _outputs(dev)]

    _reset(dev, s0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    torch.cuda.synchronize()
    names = ["key_cache", "value_cache", "kmin", "kmax", "out", "out_sparse", "selected"]
    for rep in range(3):
        _reset(dev, s0)
        g.replay()
        torch.cuda.synchronize()
        for n, t, e in zip(names, _outputs(dev), eager):
            assert torch.equal(_bits(t), e), f"replay {rep}: {n} differs from the eager step"
    assert pa_workspace_status(dev.ws) == 0
    _check_against_oracle(dev, w)
    # the workspaces are left as the next call expects them: eager after replay
    _reset(dev, s0)
    for c in calls:
        c()
    torch.cuda.synchronize()
    for n, t, e in zip(names, _outputs(dev), eager):
        assert torch.equal(_bits(t), e), f"eager after replay: {n} differs"
