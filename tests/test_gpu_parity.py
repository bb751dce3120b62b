"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Small variants of every workload are compared element by element; the full
sizes are compared in the same launch configuration the benchmark times, on
every cache byte, every metadata byte, every block score and selection, and
on a seeded sample of attention rows. Caches, metadata, scores and
selections must be bit-exact; attention outputs within max-abs 1e-2 and
mean-abs 1e-3 of the fp64 oracle.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import (DeviceStep, OracleStep, assert_close_attention, gather_rows,
                            sample_rows, to_host_f64, to_host_u16)

pytestmark = pytest.mark.gpu

SMALL = {
    # name: (workload, make() overrides) -- several KV blocks per sequence,
    # ragged last blocks, many split-KV pieces per sequence
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


def run_full_compare(w, sample=None, seed=0):
    """Whole step on both sides; compare everything (sampled attention rows if
    `sample` is an int)."""
    dev = DeviceStep(w)
    ora = OracleStep(w)
    # a1 ReshapeAndCache: caches bit-exact
    dev.reshape()
    ora.reshape()
    np.testing.assert_array_equal(to_host_u16(dev.kc), ora.kc)
    np.testing.assert_array_equal(to_host_u16(dev.vc), ora.vc)
    # metadata (rebuild from the cache) bit-exact on every block a sequence uses
    from paged_gqa_decode_reshape_gb300 import quest_rebuild_meta
    quest_rebuild_meta(dev.kmin, dev.kmax, dev.kc, dev.bt, dev.ctx)
    kmin, kmax = ora.rebuild_meta()
    used = np.unique(w.block_tables[w.block_tables >= 0])
    np.testing.assert_array_equal(to_host_u16(dev.kmin)[used], kmin[used])
    np.testing.assert_array_equal(to_host_u16(dev.kmax)[used], kmax[used])
    # a3 + a4 dense decode
    rows = None if sample is None else sample_rows(w, sample, seed)
    got = to_host_f64(dev.decode())
    want = ora.dense(rows)
    assert_close_attention(got if rows is None else gather_rows(got, rows), want, f"{w.name} dense")
    # a5 + a6 selection: scores and sets bit-exact
    dsel = dev.select()
    ds = dev.scores()
    os_ = ora.scores(kmin, kmax)
    nb = w.num_blocks()
    for b in range(w.B):
        np.testing.assert_array_equal(ds[b, :, : nb[b]], os_[b, :, : nb[b]])
    osel = ora.select(kmin, kmax)
    np.testing.assert_array_equal(dsel.cpu().numpy(), osel)
    # and against the method's definition: top-K of the plain fp64 scores
    ora.check_plain(dsel.cpu().numpy(), kmin, kmax, what=f"{w.name} selection vs plain scores")
    # a7 sparse decode on the oracle's selection
    got = to_host_f64(dev.sparse(torch.from_numpy(osel).to(dev.dev)))
    want = ora.sparse(osel, rows)
    assert_close_attention(got if rows is None else gather_rows(got, rows), want, f"{w.name} sparse")
    # the workspace is left clean (status and arrival counters zero)
    ws = dev.ws.cpu().numpy()
    assert (ws[: 256 + w.B * w.Hkv * 4] == 0).all()
    return dev, ora


@pytest.mark.parametrize("case", list(SMALL))
def test_small_elementwise(case):
    name, kw = SMALL[case]
    w = workloads.make(name, **kw)
    run_full_compare(w)


@pytest.mark.parametrize("case", list(SMALL))
def test_sparse_on_fixed_selection(case):
    """Sparse attention on a seeded selection that does not come from the
    scoring kernels: kernel error separated from selection error."""
    name, kw = SMALL[case]
    w = workloads.make(name, **kw)
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    sel = workloads.random_selection(w, seed=5)
    got = to_host_f64(dev.sparse(torch.from_numpy(sel).to(dev.dev)))
    assert_close_attention(got, ora.sparse(sel), f"{case} sparse fixed selection")


@pytest.mark.parametrize("name", ["dense_b32", "quest_8k", "long_40k", "mixed_b128"])
def test_full_size(name):
    """Full sizes, in the benchmark's launch configuration: every cache and
    metadata byte, every score and selection, every attention row."""
    w = workloads.make(name)
    run_full_compare(w)


def test_update_meta_incremental_bit_exact():
    """quest_update_meta after the step's writes equals the oracle's update
    (and the rebuild) on every block."""
    from paged_gqa_decode_reshape_gb300 import quest_rebuild_meta, quest_update_meta
    import oracle
    w = workloads.make("mixed_b128", batch=24, ctx_scale=0.03, topk=8)
    dev, ora = DeviceStep(w), OracleStep(w)
    # metadata of the cache before the step (positions < ctx - 1 hold data)
    pre_ctx = w.context_lens - 1
    pre_ctx_d = torch.from_numpy(pre_ctx.astype(np.int32)).to(dev.dev)
    quest_rebuild_meta(dev.kmin, dev.kmax, dev.kc, dev.bt, pre_ctx_d)
    kmin, kmax = oracle.quest_rebuild_meta(ora.kc, w.block_tables, pre_ctx.astype(np.int32))
    used = np.unique(w.block_tables[w.block_tables >= 0])
    np.testing.assert_array_equal(to_host_u16(dev.kmin)[used], kmin[used])
    dev.reshape()
    ora.reshape()
    quest_update_meta(dev.kmin, dev.kmax, dev.key, dev.slots, w.BS)
    oracle.quest_update_meta(kmin, kmax, w.key, w.slot_mapping, w.BS)
    np.testing.assert_array_equal(to_host_u16(dev.kmin)[used], kmin[used])
    np.testing.assert_array_equal(to_host_u16(dev.kmax)[used], kmax[used])
    # and equals the metadata rebuilt from the updated cache, for sequences
    # whose new token was written
    rmin, rmax = oracle.quest_rebuild_meta(ora.kc, w.block_tables, w.context_lens)
    written = w.slot_mapping >= 0
    for b in np.nonzero(written)[0]:
        p = w.block_tables[b, (w.context_lens[b] - 1) // w.BS]
        np.testing.assert_array_equal(kmin[p], rmin[p])
        np.testing.assert_array_equal(kmax[p], rmax[p])


def test_update_meta_many_tokens_per_block():
    """A prefill-like call: many tokens land in the same blocks, some at offset 0."""
    from paged_gqa_decode_reshape_gb300 import quest_update_meta
    import oracle
    rng = np.random.default_rng(3)
    NB, BS, Hkv, D = 12, 16, 4, 128
    kmin0 = workloads.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, D)).astype(np.float32))
    kmax0 = workloads.f32_to_bf16_bits(rng.standard_normal((NB, Hkv, D)).astype(np.float32))
    slots = np.concatenate([np.arange(2 * BS, 3 * BS + 5), np.arange(7 * BS + 3, 7 * BS + 9),
                            [-1, -3], rng.permutation(np.arange(9 * BS, 10 * BS))[:7]])
    slots = rng.permutation(slots).astype(np.int64)
    key = workloads.f32_to_bf16_bits(rng.standard_normal((len(slots), Hkv, D)).astype(np.float32))
    d = torch.device("cuda:0")
    from tests.gpu_util import to_dev_bf16
    dmin, dmax = to_dev_bf16(kmin0, d), to_dev_bf16(kmax0, d)
    quest_update_meta(dmin, dmax, to_dev_bf16(key, d), torch.from_numpy(slots).to(d), BS)
    omin, omax = kmin0.copy(), kmax0.copy()
    oracle.quest_update_meta(omin, omax, key, slots, BS)
    np.testing.assert_array_equal(to_host_u16(dmin), omin)
    np.testing.assert_array_equal(to_host_u16(dmax), omax)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 1, 128), (4, 4, 64), (16, 2, 128), (3, 3, 128), (8, 8, 64)])
def test_group_sizes_and_head_dims(Hq, Hkv, D):
    rng = np.random.default_rng(Hq * 100 + Hkv * 10 + D)
    ctx = np.array([1, 15, 16, 17, 33, 250, 64, 2])
    w = workloads.build_workload("groups", B=len(ctx), Hq=Hq, Hkv=Hkv, D=D, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(int(rng.integers(1 << 30))),
                                 topk=4, scale=1.0 / math.sqrt(D), pool_blocks=int(((ctx + 15) // 16).sum()) + 5)
    run_full_compare(w)


def test_zero_length_sequences_and_invalid_selection_entries():
    w = workloads.make("dense_b32", batch=5, ctx_scale=0.04, topk=6)
    w.context_lens[1] = 0
    w.context_lens[3] = 0
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    got = to_host_f64(dev.decode())
    assert (got[1] == 0).all() and (got[3] == 0).all()
    assert_close_attention(got, ora.dense(), "zero-length dense")
    sel = workloads.random_selection(w, seed=2)
    sel[0, 0, 1] = 10_000         # past the sequence's blocks: ignored
    sel[2, 1, :] = -1             # nothing selected: zero output for that group
    got = to_host_f64(dev.sparse(torch.from_numpy(sel).to(dev.dev)))
    want = ora.sparse(sel)
    assert_close_attention(got, want, "invalid-entry sparse")
    G = w.Hq // w.Hkv
    assert (got[2, G:2 * G] == 0).all()


def test_many_short_sequences_direct_write_path():
    """4096 short sequences: many segments fit inside one warp's range, so
    the kernel writes final outputs directly (no partials)."""
    rng = np.random.default_rng(9)
    ctx = rng.integers(1, 48, 4096)
    w = workloads.build_workload("short4096", B=4096, Hq=28, Hkv=4, D=128, BS=16, ctx=ctx,
                                 seed_seq=np.random.SeedSequence(9), topk=2, scale=1 / math.sqrt(128))
    dev, ora = DeviceStep(w), OracleStep(w)
    dev.reshape()
    ora.reshape()
    rows = sample_rows(w, 400, 1)
    got = to_host_f64(dev.decode())
    assert_close_attention(gather_rows(got, rows), ora.dense(rows), "short4096 dense")


def test_out_of_range_metadata_never_faults():
    """Bad slots and block-table entries are skipped, not followed; the
    checker counts them."""
    import paged_gqa_decode_reshape_gb300 as pg
    # no poison: the token whose slot is invalid stays unwritten inside ctx
    w = workloads.make("tiny", poison=False)
    w.slot_mapping[0] = w.NB * w.BS + 3            # past the pool
    w.block_tables[1, 2] = w.NB + 100               # past the pool
    w.block_tables[1, 4] = -5
    dev = DeviceStep(w)
    kc0 = to_host_u16(dev.kc)
    dev.reshape()
    np.testing.assert_array_equal(to_host_u16(dev.kc), kc0)   # nothing written
    out = to_host_f64(dev.decode())
    assert np.isfinite(out).all()
    counts = pg.pa_check_metadata(dev.slots, dev.bt, dev.ctx, w.BS, w.NB)
    assert counts == [1, 0, 2, 0]
    assert pg.pa_workspace_status(dev.ws) == 0


def test_repeated_calls_reuse_workspace():
    """The workspace is reusable across calls and stays zeroed; results are
    identical call after call."""
    w = workloads.make("quest_8k", batch=3, ctx_scale=0.1, topk=8)
    dev = DeviceStep(w)
    dev.reshape()
    a = dev.decode().clone()
    for _ in range(3):
        b = dev.decode()
        assert torch.equal(a, b)
    sel = workloads.random_selection(w, seed=1)
    s1 = dev.sparse(torch.from_numpy(sel).to(dev.dev)).clone()
    s2 = dev.sparse(torch.from_numpy(sel).to(dev.dev))
    assert torch.equal(s1, s2)


@pytest.mark.parametrize("name,kw", [("mixed_b128", dict(batch=24, ctx_scale=0.03, topk=8)),
                                     ("tiny", {})])
def test_fused_write_path_equals_separate_calls(name, kw):
    """quest_reshape_and_cache = pa_reshape_and_cache + quest_update_meta,
    bit for bit, and equal to the oracle's two steps."""
    import oracle
    from paged_gqa_decode_reshape_gb300 import quest_rebuild_meta, quest_reshape_and_cache
    w = workloads.make(name, **kw)
    dev, ora = DeviceStep(w), OracleStep(w)
    # metadata of the cache as it stood before the step's tokens, on both sides
    # from the same cache (the oracle's own rebuild seeds the oracle's update)
    pre_ctx_h = (w.context_lens - 1).clip(0).astype(np.int32)
    quest_rebuild_meta(dev.kmin, dev.kmax, dev.kc, dev.bt, torch.from_numpy(pre_ctx_h).to(dev.dev))
    kmin, kmax = oracle.quest_rebuild_meta(ora.kc, w.block_tables, pre_ctx_h)
    # (blocks outside every sequence's context stay zero on both sides)
    np.testing.assert_array_equal(to_host_u16(dev.kmin), kmin)
    np.testing.assert_array_equal(to_host_u16(dev.kmax), kmax)
    quest_reshape_and_cache(dev.key, dev.value, dev.kc, dev.vc, dev.kmin, dev.kmax, dev.slots)
    ora.reshape()
    oracle.quest_update_meta(kmin, kmax, w.key, w.slot_mapping, w.BS)
    np.testing.assert_array_equal(to_host_u16(dev.kc), ora.kc)
    np.testing.assert_array_equal(to_host_u16(dev.vc), ora.vc)
    np.testing.assert_array_equal(to_host_u16(dev.kmin), kmin)
    np.testing.assert_array_equal(to_host_u16(dev.kmax), kmax)
