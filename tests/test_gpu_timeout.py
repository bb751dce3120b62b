"""The decode kernel's bounded waits run out and it returns an error status.

Every wait inside the decode kernel (a consumer waiting for a staged tile, the
producer waiting for a free stage, the merge waiting for its slot, the drain
before exit) gives up after a limit, records PA_ERR_DEVICE in the workspace
status word and lets the kernel finish. The library fixes that limit at 0.5 s;
the failure-test build of the library (libpaged_decode_faulttest.so, the same
kernels with api.cu built with -DPA_FAULT_TEST) lets this test shorten it and
stop the producer part-way through its range, so the consumers wait for
stages that are never armed. Nothing faults: the copies already issued land
before each CTA exits, and the context stays usable, which the test shows by
running the same call again, correctly, after zeroing the workspace.
"""

import ctypes
import time

import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64

pytestmark = pytest.mark.gpu

PA_OK, PA_ERR_DEVICE = 0, -5
WAIT_NS = 200_000  # 0.2 ms per bounded wait in the failure runs


@pytest.fixture(scope="module")
def flib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as pgb
    pgb.build()
    L = ctypes.CDLL(pgb.FAULT_LIB)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.pa_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, f32, vp, sz, vp]
    L.pa_decode.restype = i32
    L.quest_sparse_decode.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i64,
                                      f32, vp, sz, vp]
    L.quest_sparse_decode.restype = i32
    L.pa_workspace_status.argtypes = [vp, vp]
    L.pa_workspace_status.restype = i32
    L.pa_fault_test_configure.argtypes = [i32, ctypes.c_uint64]
    L.pa_fault_test_configure.restype = None
    yield L
    L.pa_fault_test_configure(-1, 0)


def _run(L, dev, w, sel=None):
    stream = torch.cuda.current_stream(dev.dev).cuda_stream
    out = dev.out_sparse if sel is not None else dev.out
    common = (dev.q.data_ptr(), dev.kc.data_ptr(), dev.vc.data_ptr(), dev.bt.data_ptr(), w.MBS, dev.ctx.data_ptr())
    if sel is None:
        rc = L.pa_decode(out.data_ptr(), *common, w.B, w.Hq, w.Hkv, w.D, w.BS, w.NB, w.scale,
                         dev.ws.data_ptr(), dev.ws.numel(), stream)
    else:
        rc = L.quest_sparse_decode(out.data_ptr(), *common, sel.data_ptr(), sel.shape[2], w.B, w.Hq, w.Hkv,
                                   w.D, w.BS, w.NB, w.scale, dev.ws.data_ptr(), dev.ws.numel(), stream)
    assert rc == PA_OK
    return L.pa_workspace_status(dev.ws.data_ptr(), stream)


@pytest.mark.parametrize("sparse", [False, True], ids=["dense", "sparse"])
@pytest.mark.parametrize("stop_item", [0, 8])
def test_wait_runs_out_then_status_and_recovery(flib, sparse, stop_item):
    # about 27 dense items per CTA (4 sequences of ~4K tokens over 152 SMs) and
    # 12 items per sparse CTA: the producer issues 8 items per step, so with
    # stop_item 8 the first step's copies land and every later stage is never
    # armed; with 0 nothing is issued at all
    w = workloads.make("quest_8k", batch=4, ctx_scale=0.5, topk=12)
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    sel_h = workloads.random_selection(w, seed=3) if sparse else None
    sel = torch.from_numpy(sel_h).to(dev.dev) if sparse else None
    torch.cuda.synchronize()

    # the producer of every CTA stops at item stop_item of its range: the
    # consumers' waits for the later stages run out
    flib.pa_fault_test_configure(stop_item, WAIT_NS)
    t0 = time.perf_counter()
    st = _run(flib, dev, w, sel)
    elapsed = time.perf_counter() - t0
    flib.pa_fault_test_configure(-1, 0)
    assert st == PA_ERR_DEVICE, f"status {st}: the timeout was not recorded"
    assert elapsed < 5.0, f"the failed call took {elapsed:.2f} s"

    # the caller clears the workspace (as after any failed call) and the
    # context is still usable: the same call now gives the oracle's result
    dev.ws.zero_()
    assert _run(flib, dev, w, sel) == PA_OK
    want = ora.sparse(sel_h) if sparse else ora.dense()
    got = to_host_f64(dev.out_sparse if sparse else dev.out)
    assert_close_attention(got, want, f"after recovery ({'sparse' if sparse else 'dense'})")
