"""pa_decode_no_alloc: the decode entry point for callers that may not
allocate device memory (its scratch is a fixed buffer inside the library).

Called through the C ABI, twice in a row, it must give exactly the bytes
pa_decode gives with a caller-provided workspace (the same kernel, the same
fixed-order combine), and both must be within the attention tolerance of the
CPU oracle. Its status query reads PA_OK after the calls. A shape too large
for the buffer and an invalid head shape are refused on the host. This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep, assert_close_attention, to_host_f64

pytestmark = pytest.mark.gpu

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_WORKSPACE = 0, -1, -3


def _lib():
    import paged_gqa_decode_reshape_gb300 as pg
    import paged_gqa_decode_reshape_gb300.build as pgb
    pgb.build()
    lib = pg.load_library()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.pa_decode_no_alloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64,
                                       ctypes.c_float, vp]
    lib.pa_decode_no_alloc.restype = i32
    lib.pa_decode_no_alloc_status.argtypes = [vp]
    lib.pa_decode_no_alloc_status.restype = i32
    return lib


def _call(lib, out, dev, w, B=None, Hq=None, Hkv=None):
    stream = torch.cuda.current_stream(dev.dev).cuda_stream
    return lib.pa_decode_no_alloc(out.data_ptr(), dev.q.data_ptr(), dev.kc.data_ptr(), dev.vc.data_ptr(),
                                  dev.bt.data_ptr(), w.MBS, dev.ctx.data_ptr(), B or w.B, Hq or w.Hq,
                                  Hkv or w.Hkv, w.D, w.BS, w.NB, w.scale, stream)


@pytest.mark.parametrize("name,kw", [("quest_8k", dict(batch=6, ctx_scale=0.1, topk=8)),
                                     ("mixed_b128", dict(batch=24, ctx_scale=0.05, topk=8))])
def test_no_alloc_matches_workspace_decode_twice(name, kw):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = _lib()
    w = workloads.make(name, **kw)
    dev = DeviceStep(w)
    dev.reshape()
    want = dev.decode().clone()
    ora = OracleStep(w)
    ora.reshape()
    ref = ora.dense()
    assert_close_attention(to_host_f64(want), ref, f"{name} pa_decode")
    stream = torch.cuda.current_stream(dev.dev).cuda_stream
    for i in range(2):
        out = torch.full_like(dev.out, float("nan"))
        assert _call(lib, out, dev, w) == PA_OK
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want.view(torch.int16)), f"call {i}: differs from pa_decode"
        assert_close_attention(to_host_f64(out), ref, f"{name} pa_decode_no_alloc call {i}")
    assert lib.pa_decode_no_alloc_status(stream) == PA_OK


def test_no_alloc_refuses_what_it_cannot_run():
    """A batch whose split-KV partials need more than the fixed buffer is
    refused with PA_ERR_WORKSPACE, and Hq not a multiple of Hkv with
    PA_ERR_INVALID_ARG; both on the host, before any launch, with the output
    untouched."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = _lib()
    w = workloads.make("quest_8k", batch=2, ctx_scale=0.05, topk=4)
    dev = DeviceStep(w)
    out = torch.full_like(dev.out, 3.0)
    torch.cuda.synchronize()
    # 1024 sequences x 4 KV heads: about 17 MB of partials, over the 8 MiB buffer
    assert _call(lib, out, dev, w, B=1024, Hq=32, Hkv=4) == PA_ERR_WORKSPACE
    assert _call(lib, out, dev, w, Hq=30, Hkv=4) == PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (out.float() == 3.0).all()
