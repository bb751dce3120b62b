"""Parity of the 8-bit (E4M3) KV-cache path (through the C ABI) against the
CPU oracle: the quantised caches and metadata, the block scores and the
selection bit for bit; dense and sparse attention within max-abs 1e-2 and
mean-abs 1e-3 of the oracle's fp64 attention on the dequantised cache.

Both sides build their 8-bit pool from the same bf16 pool, each with its own
write path (every slot of the pool written once), then run the step."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import assert_close_attention, gather_rows, sample_rows, to_host_f64
from tests.selection_check import check_selection

pytestmark = pytest.mark.gpu

SMALL = {
    "quest_small": ("quest_8k", dict(batch=4, ctx_scale=0.05, topk=6)),
    "mixed_small": ("mixed_b128", dict(batch=16, ctx_scale=0.02, topk=8)),
    "long_small": ("long_40k", dict(batch=2, ctx_scale=0.02, topk=16)),
    "dense_small": ("dense_b32", dict(batch=6, ctx_scale=0.05, topk=8)),
    # odd topk: a segment's last two-block item of the 8-bit decode holds one entry
    "odd_topk": ("quest_8k", dict(batch=4, ctx_scale=0.05, topk=7)),
    "odd_topk_long": ("long_40k", dict(batch=2, ctx_scale=0.02, topk=15)),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


class Fp8Case:
    """One workload on both sides with an 8-bit cache."""

    def __init__(self, w):
        import paged_gqa_decode_reshape_gb300 as pg
        self.pg, self.w = pg, w
        d = torch.device("cuda:0")
        NB, BS, Hkv, D = w.key_cache.shape
        ks, vs = workloads.fp8_scales(Hkv)
        self.ks_h, self.vs_h = ks, vs
        self.ks, self.vs = torch.from_numpy(ks).to(d), torch.from_numpy(vs).to(d)

        def d16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(d).view(torch.bfloat16)

        self.q = d16(w.q)
        self.key, self.value = d16(w.key), d16(w.value)
        self.slots = torch.from_numpy(w.slot_mapping).to(d)
        self.bt = torch.from_numpy(w.block_tables).to(d)
        self.ctx = torch.from_numpy(w.context_lens).to(d)
        # the pool: every slot written once through each side's write path
        pool_slots = np.arange(NB * BS, dtype=np.int64)
        self.kc = torch.empty((NB, BS, Hkv, D), dtype=torch.uint8, device=d)
        self.vc = torch.empty((NB, Hkv, D, BS), dtype=torch.uint8, device=d)
        pg.pa_reshape_and_cache_fp8(d16(w.key_cache.reshape(NB * BS, Hkv, D)),
                                    d16(w.value_cache.reshape(NB * BS, Hkv, D)), self.kc, self.vc,
                                    torch.from_numpy(pool_slots).to(d), self.ks, self.vs)
        self.okc = np.zeros((NB, BS, Hkv, D), dtype=np.uint8)
        self.ovc = np.zeros((NB, Hkv, D, BS), dtype=np.uint8)
        oracle.reshape_and_cache_fp8(w.key_cache.reshape(NB * BS, Hkv, D),
                                     w.value_cache.reshape(NB * BS, Hkv, D), self.okc, self.ovc,
                                     pool_slots, ks, vs)
        self.kmin = torch.zeros((NB, Hkv, D), dtype=torch.uint8, device=d)
        self.kmax = torch.zeros_like(self.kmin)
        self.out = torch.empty((w.B, w.Hq, D), dtype=torch.bfloat16, device=d)
        self.out_sparse = torch.empty_like(self.out)
        self.sel = torch.empty((w.B, Hkv, w.topk), dtype=torch.int32, device=d)
        self.ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, Hkv, D), dtype=torch.uint8, device=d)
        self.sel_ws = torch.zeros(pg.quest_select_workspace_size(w.B, Hkv, w.MBS), dtype=torch.uint8,
                                  device=d)
        self.used = np.unique(w.block_tables[w.block_tables >= 0])

    def write_step(self):
        """Metadata of the cache before the step's tokens, then the fused
        write path; returns the oracle's metadata after the step."""
        w, pg = self.w, self.pg
        pre = (w.context_lens - 1).clip(0).astype(np.int32)
        pg.quest_rebuild_meta_fp8(self.kmin, self.kmax, self.kc, self.bt,
                                  torch.from_numpy(pre).to(self.bt.device))
        kmin, kmax = oracle.quest_rebuild_meta_fp8(self.okc, w.block_tables, pre)
        np.testing.assert_array_equal(u8(self.kmin)[self.used], kmin[self.used])
        np.testing.assert_array_equal(u8(self.kmax)[self.used], kmax[self.used])
        pg.quest_reshape_and_cache_fp8(self.key, self.value, self.kc, self.vc, self.kmin, self.kmax,
                                       self.slots, self.ks, self.vs)
        oracle.reshape_and_cache_fp8(w.key, w.value, self.okc, self.ovc, w.slot_mapping, self.ks_h,
                                     self.vs_h)
        oracle.quest_update_meta_fp8(kmin, kmax, w.key, w.slot_mapping, self.ks_h, w.BS)
        return kmin, kmax


def run_fp8_compare(w, sample=None, seed=0):
    c = Fp8Case(w)
    pg = c.pg
    # the 8-bit pool, byte for byte
    np.testing.assert_array_equal(u8(c.kc), c.okc)
    np.testing.assert_array_equal(u8(c.vc), c.ovc)
    # the step's write path: caches and metadata byte for byte
    kmin, kmax = c.write_step()
    np.testing.assert_array_equal(u8(c.kc), c.okc)
    np.testing.assert_array_equal(u8(c.vc), c.ovc)
    np.testing.assert_array_equal(u8(c.kmin)[c.used], kmin[c.used])
    np.testing.assert_array_equal(u8(c.kmax)[c.used], kmax[c.used])
    # Quest scores and selection, bit for bit
    pg.quest_select_topk_fp8(c.sel, c.q, c.kmin, c.kmax, c.bt, c.ctx, w.BS, workspace=c.sel_ws)
    n = w.B * w.Hkv * w.MBS
    got_scores = c.sel_ws[: n * 4].view(torch.float32).cpu().numpy().reshape(w.B, w.Hkv, w.MBS)
    want_scores = oracle.quest_scores_kernel_order_fp8(w.q, kmin, kmax, w.block_tables, w.context_lens,
                                                       w.BS)
    nb = (np.minimum(w.context_lens, w.MBS * w.BS) + w.BS - 1) // w.BS
    for b in range(w.B):
        np.testing.assert_array_equal(got_scores[b, :, : nb[b]].view(np.uint32),
                                      want_scores[b, :, : nb[b]].view(np.uint32))
    sel = oracle.quest_topk(want_scores, w.context_lens, w.BS, w.topk)
    np.testing.assert_array_equal(c.sel.cpu().numpy(), sel)
    # and against the method's definition: top-K of the plain fp64 scores
    plain, absum = oracle.quest_scores_fp8(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS,
                                           with_abs=True)
    check_selection(c.sel.cpu().numpy(), plain, absum, w.context_lens, w.BS, w.topk, w.Hq // w.Hkv, w.D,
                    f"{w.name} fp8 selection vs plain scores")
    # attention
    rows = None if sample is None else sample_rows(w, sample, seed)
    pg.pa_decode_fp8(c.out, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens,
                                w.scale, rows=rows)
    got = to_host_f64(c.out)
    assert_close_attention(got if rows is None else gather_rows(got, rows), want, f"{w.name} fp8 dense")
    pg.quest_sparse_decode_fp8(c.out_sparse, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, c.sel, w.scale,
                               workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens,
                                w.scale, selected=sel, rows=rows)
    got = to_host_f64(c.out_sparse)
    assert_close_attention(got if rows is None else gather_rows(got, rows), want, f"{w.name} fp8 sparse")
    assert pg.pa_workspace_status(c.ws) == 0
    return c


@pytest.mark.parametrize("case", list(SMALL))
def test_fp8_small_elementwise(case):
    name, kw = SMALL[case]
    run_fp8_compare(workloads.make(name, **kw))


@pytest.mark.parametrize("name", ["dense_b32", "quest_8k", "long_40k"])
def test_fp8_full_size(name):
    run_fp8_compare(workloads.make(name), sample=48, seed=13)


def test_fp8_sparse_on_fixed_selection():
    """Sparse attention on a seeded selection that is not the top-K (kernel
    error kept apart from selection error), with invalid entries mixed in."""
    w = workloads.make("mixed_b128", batch=16, ctx_scale=0.02, topk=8)
    c = Fp8Case(w)
    c.write_step()  # the step's new tokens fill the last valid position of each sequence
    rng = np.random.default_rng(21)
    nb = (np.minimum(w.context_lens, w.MBS * w.BS) + w.BS - 1) // w.BS
    sel = np.full((w.B, w.Hkv, w.topk), -1, dtype=np.int32)
    for b in range(w.B):
        for g in range(w.Hkv):
            k = min(w.topk, int(nb[b]))
            sel[b, g, :k] = np.sort(rng.choice(int(nb[b]), k, replace=False))
    sel[0, 0, -1] = 10 ** 6            # past the sequence: ignored
    c.pg.quest_sparse_decode_fp8(c.out_sparse, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx,
                                 torch.from_numpy(sel).to(c.bt.device), w.scale, workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens,
                                w.scale, selected=sel)
    assert_close_attention(to_host_f64(c.out_sparse), want, "fp8 sparse, fixed selection")


def test_fp8_zero_length_sequences():
    """Sequences with no tokens get zero output; the others are unaffected."""
    w = workloads.make("quest_8k", batch=4, ctx_scale=0.05, topk=6)
    w.context_lens[1] = 0
    w.context_lens[3] = 0
    w.slot_mapping[1] = -1
    w.slot_mapping[3] = -1
    c = Fp8Case(w)
    c.write_step()
    c.pg.pa_decode_fp8(c.out, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.ks_h, c.vs_h, w.block_tables, w.context_lens,
                                w.scale)
    got = to_host_f64(c.out)
    assert (got[1] == 0).all() and (got[3] == 0).all()
    assert_close_attention(got, want, "fp8 dense with empty sequences")


@pytest.mark.parametrize("with_meta", [True, False])
def test_fp8_write_shuffled_tokens_sharing_blocks(with_meta):
    """One call whose tokens land in the same blocks in shuffled order, with
    padding slots, blocks that start fresh and blocks merged with their old
    metadata, over more than one 32-token chunk of the call. Caches and
    metadata byte for byte against the oracle (so the bytes of untouched
    slots are unchanged)."""
    import paged_gqa_decode_reshape_gb300 as pg
    rng = np.random.default_rng(21)
    NB, BS, Hkv, D, T = 12, 16, 2, 128, 70
    d = torch.device("cuda:0")
    slots = rng.choice(NB * BS, size=T, replace=False).astype(np.int64)
    slots[rng.choice(T, size=6, replace=False)] = -1
    key = workloads.f32_to_bf16_bits((rng.standard_normal((T, Hkv, D)) * 2).astype(np.float32))
    value = workloads.f32_to_bf16_bits((rng.standard_normal((T, Hkv, D)) * 2).astype(np.float32))
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    kc0 = rng.choice(finite, size=(NB, BS, Hkv, D)).astype(np.uint8)
    vc0 = rng.choice(finite, size=(NB, Hkv, D, BS)).astype(np.uint8)
    kmin0 = rng.choice(finite, size=(NB, Hkv, D)).astype(np.uint8)
    kmax0 = rng.choice(finite, size=(NB, Hkv, D)).astype(np.uint8)
    ks, vs = workloads.fp8_scales(Hkv)

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(d).view(torch.bfloat16)

    kc, vc = torch.from_numpy(kc0.copy()).to(d), torch.from_numpy(vc0.copy()).to(d)
    kmin, kmax = torch.from_numpy(kmin0.copy()).to(d), torch.from_numpy(kmax0.copy()).to(d)
    ksd, vsd = torch.from_numpy(ks).to(d), torch.from_numpy(vs).to(d)
    slots_d = torch.from_numpy(slots).to(d)
    if with_meta:
        pg.quest_reshape_and_cache_fp8(d16(key), d16(value), kc, vc, kmin, kmax, slots_d, ksd, vsd)
    else:
        pg.pa_reshape_and_cache_fp8(d16(key), d16(value), kc, vc, slots_d, ksd, vsd)
    okc, ovc = kc0.copy(), vc0.copy()
    oracle.reshape_and_cache_fp8(key, value, okc, ovc, slots, ks, vs)
    np.testing.assert_array_equal(u8(kc), okc)
    np.testing.assert_array_equal(u8(vc), ovc)
    okmin, okmax = kmin0.copy(), kmax0.copy()
    if with_meta:
        oracle.quest_update_meta_fp8(okmin, okmax, key, slots, ks, BS)
    np.testing.assert_array_equal(u8(kmin), okmin)
    np.testing.assert_array_equal(u8(kmax), okmax)
