"""pa_decode_no_alloc: the decode entry point for callers that may not
allocate device memory (its scratch is a fixed buffer inside the library).

Called through the C ABI, twice in a row, it must give the same result as
pa_decode with a caller-provided workspace, within the attention tolerance
the other tests use. This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes on its
own in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import MAX_ABS_TOL, MEAN_ABS_TOL, DeviceStep

pytestmark = pytest.mark.gpu


def _no_alloc_fn():
    import paged_gqa_decode_reshape_gb300 as pg
    import paged_gqa_decode_reshape_gb300.build as pgb
    pgb.build()
    lib = pg.load_library()
    f = lib.pa_decode_no_alloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, ctypes.c_float, vp]
    f.restype = i32
    return f


@pytest.mark.parametrize("name,kw", [("quest_8k", dict(batch=6, ctx_scale=0.1, topk=8)),
                                     ("mixed_b128", dict(batch=24, ctx_scale=0.05, topk=8))])
def test_no_alloc_matches_workspace_decode_twice(name, kw):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    f = _no_alloc_fn()
    w = workloads.make(name, **kw)
    dev = DeviceStep(w)
    dev.reshape()
    want = dev.decode().float().cpu().numpy()
    stream = torch.cuda.current_stream(dev.dev).cuda_stream
    for _ in range(2):
        out = torch.full_like(dev.out, float("nan"))
        rc = f(out.data_ptr(), dev.q.data_ptr(), dev.kc.data_ptr(), dev.vc.data_ptr(), dev.bt.data_ptr(),
               w.MBS, dev.ctx.data_ptr(), w.B, w.Hq, w.Hkv, w.D, w.BS, w.NB, w.scale, stream)
        assert rc == 0
        got = out.float().cpu().numpy()
        err = np.abs(got.astype(np.float64) - want)
        assert np.isfinite(got).all()
        assert err.max() <= MAX_ABS_TOL and err.mean() <= MEAN_ABS_TOL
