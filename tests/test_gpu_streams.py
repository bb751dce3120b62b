"""The step's calls on two streams give results bit-identical to the same
calls on one stream. On two streams the Quest path (quest_decode) runs
beside the dense decode, and each decode call has its own workspace.
Every kernel's output is a deterministic function of its inputs (the split-KV
combine merges the pieces in a fixed order), so running calls at the same
time may change timing but never a bit of the results. The results are
also checked against the CPU oracle (bf16 cache)."""

import numpy as np
import pytest
import torch

import bench
import workloads
from tests.gpu_util import OracleStep, assert_close_attention, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def _check_against_oracle(st, w):
    """The step's results (the last, two-stream run) against the CPU oracle:
    the selection bit for bit and against the plain score's top-K, both
    attention outputs within the tolerances."""
    ora = OracleStep(w)
    ora.reshape()
    kmin, kmax = ora.rebuild_meta()
    sel = st.sel.cpu().numpy()
    np.testing.assert_array_equal(sel, ora.select(kmin, kmax))
    ora.check_plain(sel, kmin, kmax, what=f"{w.name} two-stream selection vs plain scores")
    assert_close_attention(to_host_f64(st.out), ora.dense(), f"{w.name} two-stream dense")
    assert_close_attention(to_host_f64(st.out_sparse), ora.sparse(sel), f"{w.name} two-stream sparse")


@pytest.mark.parametrize("name,kw,kv", [
    ("quest_8k", dict(batch=8, ctx_scale=0.25, topk=32), "bf16"),
    ("long_40k", dict(batch=2, ctx_scale=0.1, topk=64), "bf16"),
    ("quest_8k", dict(batch=8, ctx_scale=0.25, topk=32), "fp8"),
])
def test_two_stream_step_matches_one_stream(name, kw, kv):
    w = workloads.make(name, poison=False, **kw)
    st = bench.Step(w, torch.device("cuda:0"), kv)
    results = []
    for serial in (True, False, True, False):
        # the same grids in both orders
        run = bench.step_runner(torch, st, serial, quest=st.quest_beside(), dense=st.dense_beside())
        for _ in range(2):  # the write path is idempotent: the same tokens into the same slots
            st.out_buf.zero_()
            run()
        torch.cuda.synchronize()
        results.append(st.out_buf.clone())
    for r in results[1:]:
        assert torch.equal(r, results[0])
    if kv == "bf16":
        _check_against_oracle(st, w)
    # the workspaces are left clean after both orders
    assert int(st.ws[:4].view(torch.int32)[0]) == 0
    assert int(st.ws_sparse[:4].view(torch.int32)[0]) == 0
