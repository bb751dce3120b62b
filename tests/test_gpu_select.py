"""Quest selection (scores + top-K) on the GPU against the CPU oracle: a
sequence whose keys do not fit the top-K kernel's shared-memory cache
(8199 blocks; the cache holds 3072 keys), and every score of a segment
tied (the lower block index wins). Scores and selections must be
bit-exact."""

import math

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import DeviceStep, OracleStep
from tests.test_gpu_parity import run_full_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def test_select_long_sequence_keys_from_global_memory():
    ctx = np.array([8192 * 16 + 100, 3000])   # 8199 and 188 blocks
    w = workloads.build_workload("long131k", B=2, Hq=4, Hkv=1, D=64, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(131), topk=64, scale=1.0 / math.sqrt(64),
                                 pool_blocks=int(((ctx + 15) // 16).sum()) + 3)
    run_full_compare(w, sample=8, seed=4)


def test_select_ties_across_parts():
    """Constant metadata: every block of a segment has the same score, so the
    selection is the topk lowest block indices."""
    ctx = np.array([5000, 4100, 700])          # 313, 257, 44 blocks
    w = workloads.build_workload("ties", B=3, Hq=8, Hkv=2, D=128, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(77), topk=40, scale=1.0 / math.sqrt(128))
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.kmin.fill_(0.5)
    dev.kmax.fill_(0.5)
    half = np.uint16(0x3F00)                   # bf16 0.5
    kmin = np.full((w.NB, w.Hkv, w.D), half, dtype=np.uint16)
    kmax = kmin.copy()
    dsel = dev.select().cpu().numpy()
    osel = ora.select(kmin, kmax)
    np.testing.assert_array_equal(dsel, osel)
    assert ora.check_plain(dsel, kmin, kmax, what="all-tied selection vs plain scores") == 0
    nb = w.num_blocks()
    for b in range(w.B):
        want = np.arange(w.topk) if nb[b] > w.topk else np.r_[np.arange(nb[b]), -np.ones(w.topk - nb[b])]
        assert (osel[b] == want.astype(np.int32)).all()
