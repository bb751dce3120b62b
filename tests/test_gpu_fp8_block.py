"""Parity of the 8-bit cache with per-block scales (through the C ABI)
against the CPU oracle: codes, per-block scales and metadata byte for byte
after every write (scales that restart, hold and grow, with the block's
other codes re-encoded); block scores and selections bit for bit (and
against the plain fp64 scores); dense, sparse and fused Quest attention
within max-abs 1e-2 and mean-abs 1e-3 of the oracle's fp64 attention.

The pools get power-of-two factors per (block, KV head) -- K from 2^-3 to
2, V from 2^-3 to 1 -- so that neighbouring blocks carry different scales,
and are written in two calls (offsets 0-7 of every block, which restart it,
then 8-15, which merge), each side with its own write path. (Larger factors
make the softmax so peaked that the f16 rounding of a few dominant weights,
which the per-KV-head path has too, exceeds the absolute max-abs bar; the
exact-agreement test below separates the per-block machinery from that.)"""

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


def d16(a, d):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(d).view(torch.bfloat16)


def spread_pool(w, seed=5):
    """The workload's bf16 pool with power-of-two factors per (block, KV
    head): exact in bf16 (the values stay in its normal range)."""
    rng = np.random.default_rng(seed)
    NB, BS, Hkv, D = w.key_cache.shape
    fk = 2.0 ** rng.integers(-3, 2, (NB, 1, Hkv, 1))
    fv = 2.0 ** rng.integers(-3, 1, (NB, 1, Hkv, 1))
    k = workloads.f32_to_bf16_bits((workloads.bf16_bits_to_f32(w.key_cache) * fk).astype(np.float32))
    v = workloads.f32_to_bf16_bits((workloads.bf16_bits_to_f32(w.value_cache) * fv).astype(np.float32))
    return k, v


class BlockCase:
    """One workload on both sides with a per-block-scaled 8-bit cache."""

    def __init__(self, w):
        import paged_gqa_decode_reshape_gb300 as pg
        self.pg, self.w = pg, w
        d = self.d = torch.device("cuda:0")
        NB, BS, Hkv, D = w.key_cache.shape
        kpool, vpool = spread_pool(w)
        self.q = d16(w.q, d)
        self.key, self.value = d16(w.key, d), d16(w.value, d)
        self.slots = torch.from_numpy(w.slot_mapping).to(d)
        self.bt = torch.from_numpy(w.block_tables).to(d)
        self.ctx = torch.from_numpy(w.context_lens).to(d)
        self.kc = torch.zeros((NB, BS, Hkv, D), dtype=torch.uint8, device=d)
        self.vc = torch.zeros((NB, Hkv, D, BS), dtype=torch.uint8, device=d)
        self.ks = torch.zeros((NB, Hkv), dtype=torch.float32, device=d)
        self.vs = torch.zeros_like(self.ks)
        self.okc = np.zeros((NB, BS, Hkv, D), dtype=np.uint8)
        self.ovc = np.zeros((NB, Hkv, D, BS), dtype=np.uint8)
        self.oks = np.zeros((NB, Hkv), dtype=np.float32)
        self.ovs = np.zeros_like(self.oks)
        kp, vp = kpool.reshape(NB * BS, Hkv, D), vpool.reshape(NB * BS, Hkv, D)
        for lo in (0, 8):  # two calls: offsets 0-7 (restart), then 8-15 (merge)
            slots = (np.arange(NB)[:, None] * BS + np.arange(lo, lo + 8)[None, :]).reshape(-1).astype(np.int64)
            pg.pa_reshape_and_cache_fp8_block(d16(kp[slots], d), d16(vp[slots], d), self.kc, self.vc,
                                              torch.from_numpy(slots).to(d), self.ks, self.vs)
            oracle.reshape_and_cache_fp8_block(kp[slots], vp[slots], self.okc, self.ovc, slots, self.oks,
                                               self.ovs)
        self.kmin = torch.zeros((NB, Hkv, D), dtype=torch.uint8, device=d)
        self.kmax = torch.zeros_like(self.kmin)
        self.out = torch.empty((w.B, w.Hq, D), dtype=torch.bfloat16, device=d)
        self.out_sparse = torch.empty_like(self.out)
        self.sel = torch.empty((w.B, Hkv, w.topk), dtype=torch.int32, device=d)
        self.ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, Hkv, D), dtype=torch.uint8, device=d)
        self.sel_ws = torch.zeros(pg.quest_select_workspace_size(w.B, Hkv, w.MBS), dtype=torch.uint8, device=d)
        self.used = np.unique(w.block_tables[w.block_tables >= 0])

    def check_pool(self, what):
        np.testing.assert_array_equal(u8(self.kc), self.okc, err_msg=f"{what}: K codes")
        np.testing.assert_array_equal(u8(self.vc), self.ovc, err_msg=f"{what}: V codes")
        np.testing.assert_array_equal(self.ks.cpu().numpy().view(np.uint32), self.oks.view(np.uint32),
                                      err_msg=f"{what}: K scales")
        np.testing.assert_array_equal(self.vs.cpu().numpy().view(np.uint32), self.ovs.view(np.uint32),
                                      err_msg=f"{what}: V scales")

    def write_step(self):
        """Metadata of the cache before the step's tokens, then the write path
        with the metadata update; returns the oracle's metadata after it."""
        w, pg = self.w, self.pg
        pre = (w.context_lens - 1).clip(0).astype(np.int32)
        pg.quest_rebuild_meta_fp8(self.kmin, self.kmax, self.kc, self.bt, torch.from_numpy(pre).to(self.d))
        kmin, kmax = oracle.quest_rebuild_meta_fp8(self.okc, w.block_tables, pre)
        pg.quest_reshape_and_cache_fp8_block(self.key, self.value, self.kc, self.vc, self.kmin, self.kmax,
                                             self.slots, self.ks, self.vs)
        oracle.reshape_and_cache_fp8_block(w.key, w.value, self.okc, self.ovc, w.slot_mapping, self.oks,
                                           self.ovs, kmin, kmax)
        return kmin, kmax


def run_block_compare(w, sample=None, seed=0):
    c = BlockCase(w)
    pg = c.pg
    c.check_pool("pool")
    assert len(np.unique(c.oks)) > 4, "the pool should carry several different block scales"
    kmin, kmax = c.write_step()
    c.check_pool("after the step's write")
    np.testing.assert_array_equal(u8(c.kmin)[c.used], kmin[c.used])
    np.testing.assert_array_equal(u8(c.kmax)[c.used], kmax[c.used])
    # block scores (times the blocks' K scales) and the selection, bit for bit
    pg.quest_select_topk_fp8_block(c.sel, c.q, c.kmin, c.kmax, c.ks, c.bt, c.ctx, w.BS, workspace=c.sel_ws)
    n = w.B * w.Hkv * w.MBS
    got_scores = c.sel_ws[: n * 4].view(torch.float32).cpu().numpy().reshape(w.B, w.Hkv, w.MBS)
    want_scores = oracle.quest_scores_kernel_order_fp8(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS,
                                                       k_bscale=c.oks)
    nb = (np.minimum(w.context_lens, w.MBS * w.BS) + w.BS - 1) // w.BS
    for b in range(w.B):
        np.testing.assert_array_equal(got_scores[b, :, : nb[b]].view(np.uint32),
                                      want_scores[b, :, : nb[b]].view(np.uint32))
    sel = oracle.quest_topk(want_scores, w.context_lens, w.BS, w.topk)
    np.testing.assert_array_equal(c.sel.cpu().numpy(), sel)
    plain, absum = oracle.quest_scores_fp8(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS,
                                           with_abs=True, k_bscale=c.oks)
    check_selection(c.sel.cpu().numpy(), plain, absum, w.context_lens, w.BS, w.topk, w.Hq // w.Hkv, w.D,
                    f"{w.name} per-block fp8 selection vs plain scores")
    # attention
    rows = None if sample is None else sample_rows(w, sample, seed)

    def pick(t):
        got = to_host_f64(t)
        return got if rows is None else gather_rows(got, rows)

    pg.pa_decode_fp8_block(c.out, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.scale, workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.oks, c.ovs, w.block_tables, w.context_lens, w.scale,
                                rows=rows)
    assert_close_attention(pick(c.out), want, f"{w.name} per-block fp8 dense")
    pg.quest_sparse_decode_fp8_block(c.out_sparse, c.q, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, c.sel, w.scale,
                                     workspace=c.ws)
    want = oracle.attention_fp8(w.q, c.okc, c.ovc, c.oks, c.ovs, w.block_tables, w.context_lens, w.scale,
                                selected=sel, rows=rows)
    assert_close_attention(pick(c.out_sparse), want, f"{w.name} per-block fp8 sparse")
    # the fused Quest decode: the same selection, the same bytes as the separate sparse call
    qws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS), dtype=torch.uint8,
                      device=c.d)
    fsel = torch.full_like(c.sel, -7)
    fout = torch.full_like(c.out, float("nan"))
    pg.quest_decode_fp8_block(fout, fsel, c.q, c.kmin, c.kmax, c.kc, c.vc, c.ks, c.vs, c.bt, c.ctx, w.topk,
                              w.scale, workspace=qws)
    np.testing.assert_array_equal(fsel.cpu().numpy(), sel)
    assert torch.equal(fout.view(torch.int16), c.out_sparse.view(torch.int16))
    assert pg.pa_workspace_status(c.ws) == 0 and pg.pa_workspace_status(qws) == 0
    return c


@pytest.mark.parametrize("case", list(SMALL))
def test_block_small_elementwise(case):
    name, kw = SMALL[case]
    run_block_compare(workloads.make(name, **kw))


@pytest.mark.parametrize("name", ["quest_8k", "long_40k"])
def test_block_full_size(name):
    run_block_compare(workloads.make(name), sample=48, seed=17)


@pytest.mark.parametrize("with_meta", [True, False])
def test_block_write_growing_scales(with_meta):
    """Tokens appended one call at a time with magnitudes that grow (so the
    scales grow and the blocks' other codes are re-encoded, K and V apart),
    a restart in the middle, then one multi-token call with tokens of the
    same blocks in shuffled order and padding slots: codes, scales and
    metadata byte for byte after every call."""
    import paged_gqa_decode_reshape_gb300 as pg
    rng = np.random.default_rng(23)
    NB, BS, Hkv, D, B = 10, 16, 3, 128, 4
    d = torch.device("cuda:0")
    kc = torch.zeros((NB, BS, Hkv, D), dtype=torch.uint8, device=d)
    vc = torch.zeros((NB, Hkv, D, BS), dtype=torch.uint8, device=d)
    ks = torch.zeros((NB, Hkv), dtype=torch.float32, device=d)
    vs = torch.zeros_like(ks)
    kmin = torch.zeros((NB, Hkv, D), dtype=torch.uint8, device=d)
    kmax = torch.zeros_like(kmin)
    okc, ovc = np.zeros((NB, BS, Hkv, D), np.uint8), np.zeros((NB, Hkv, D, BS), np.uint8)
    oks, ovs = np.zeros((NB, Hkv), np.float32), np.zeros((NB, Hkv), np.float32)
    okmin, okmax = np.zeros((NB, Hkv, D), np.uint8), np.zeros((NB, Hkv, D), np.uint8)
    blocks = rng.permutation(NB)[:B]

    def call(slots, key, value):
        sd = torch.from_numpy(slots).to(d)
        if with_meta:
            pg.quest_reshape_and_cache_fp8_block(d16(key, d), d16(value, d), kc, vc, kmin, kmax, sd, ks, vs)
            oracle.reshape_and_cache_fp8_block(key, value, okc, ovc, slots, oks, ovs, okmin, okmax)
        else:
            pg.pa_reshape_and_cache_fp8_block(d16(key, d), d16(value, d), kc, vc, sd, ks, vs)
            oracle.reshape_and_cache_fp8_block(key, value, okc, ovc, slots, oks, ovs)
        np.testing.assert_array_equal(u8(kc), okc)
        np.testing.assert_array_equal(u8(vc), ovc)
        np.testing.assert_array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
        np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))
        if with_meta:
            np.testing.assert_array_equal(u8(kmin), okmin)
            np.testing.assert_array_equal(u8(kmax), okmax)

    grew = 0
    for step in range(BS + 4):
        o = step % BS  # step 16 restarts each block at offset 0
        slots = (blocks * BS + o).astype(np.int64)
        f = 1.3 ** step * np.array([1.0, 0.25, 4.0])[None, :, None]
        key = workloads.f32_to_bf16_bits((rng.standard_normal((B, Hkv, D)) * f).astype(np.float32))
        value = workloads.f32_to_bf16_bits((rng.standard_normal((B, Hkv, D)) * f[:, ::-1]).astype(np.float32))
        before = oks.copy()
        call(slots, key, value)
        grew += int((oks > before).sum()) if o else 0
    assert grew > 0
    # one call, many tokens per block, shuffled, with padding slots
    T = 40
    slots = rng.choice(NB * BS, size=T, replace=False).astype(np.int64)
    slots[rng.choice(T, size=5, replace=False)] = -1
    key = workloads.f32_to_bf16_bits((rng.standard_normal((T, Hkv, D)) * 30).astype(np.float32))
    value = workloads.f32_to_bf16_bits((rng.standard_normal((T, Hkv, D)) * 0.01).astype(np.float32))
    call(slots, key, value)


def test_block_path_equals_head_path_when_scales_agree():
    """A pool whose blocks all get the same scale per KV head (every (block,
    head) holds one element of the same largest magnitude): the per-block
    cache then has the codes of the per-KV-head cache with those power-of-two
    scales, and dense, sparse and fused decode must give the same bytes on
    both paths (the per-block scale handling reduces to the per-head one)."""
    import paged_gqa_decode_reshape_gb300 as pg
    w = workloads.make("quest_8k", batch=4, ctx_scale=0.1, topk=12, poison=False)
    d = torch.device("cuda:0")
    NB, BS, Hkv, D = w.key_cache.shape
    k = workloads.bf16_bits_to_f32(w.key_cache).copy()
    v = workloads.bf16_bits_to_f32(w.value_cache).copy()
    k = np.clip(k, -7.0, 7.0)
    v = np.clip(v, -6.0, 6.0)
    k[:, 0, :, 0] = 7.0   # every (block, head): largest |k| = 7 -> scale 2^-6 (7 <= 448 / 64)
    v[:, 0, :, 0] = -6.0  # largest |v| = 6 -> 2^-6
    kb, vb = workloads.f32_to_bf16_bits(k), workloads.f32_to_bf16_bits(v)
    slots = torch.arange(NB * BS, dtype=torch.int64, device=d)
    kc_b = torch.zeros((NB, BS, Hkv, D), dtype=torch.uint8, device=d)
    vc_b = torch.zeros((NB, Hkv, D, BS), dtype=torch.uint8, device=d)
    ksb = torch.zeros((NB, Hkv), dtype=torch.float32, device=d)
    vsb = torch.zeros_like(ksb)
    pg.pa_reshape_and_cache_fp8_block(d16(kb.reshape(-1, Hkv, D), d), d16(vb.reshape(-1, Hkv, D), d), kc_b, vc_b,
                                      slots, ksb, vsb)
    assert (ksb == 2.0 ** -6).all() and (vsb == 2.0 ** -6).all()
    ksh = torch.full((Hkv,), 2.0 ** -6, dtype=torch.float32, device=d)
    vsh = ksh.clone()
    kc_h, vc_h = torch.zeros_like(kc_b), torch.zeros_like(vc_b)
    pg.pa_reshape_and_cache_fp8(d16(kb.reshape(-1, Hkv, D), d), d16(vb.reshape(-1, Hkv, D), d), kc_h, vc_h, slots,
                                ksh, vsh)
    assert torch.equal(kc_b, kc_h) and torch.equal(vc_b, vc_h)
    q = d16(w.q, d)
    bt = torch.from_numpy(w.block_tables).to(d)
    ctx = torch.from_numpy(w.context_lens).to(d)
    ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, Hkv, D), dtype=torch.uint8, device=d)
    out_h = torch.empty((w.B, w.Hq, D), dtype=torch.bfloat16, device=d)
    out_b = torch.empty_like(out_h)
    pg.pa_decode_fp8(out_h, q, kc_h, vc_h, ksh, vsh, bt, ctx, w.scale, workspace=ws)
    pg.pa_decode_fp8_block(out_b, q, kc_b, vc_b, ksb, vsb, bt, ctx, w.scale, workspace=ws)
    assert torch.equal(out_h.view(torch.int16), out_b.view(torch.int16))
    kmin = torch.zeros((NB, Hkv, D), dtype=torch.uint8, device=d)
    kmax = torch.zeros_like(kmin)
    pg.quest_rebuild_meta_fp8(kmin, kmax, kc_b, bt, ctx)
    sel_h = torch.empty((w.B, Hkv, w.topk), dtype=torch.int32, device=d)
    sel_b = torch.empty_like(sel_h)
    pg.quest_select_topk_fp8(sel_h, q, kmin, kmax, bt, ctx, BS)
    pg.quest_select_topk_fp8_block(sel_b, q, kmin, kmax, ksb, bt, ctx, BS)
    assert torch.equal(sel_h, sel_b)  # the per-block scores are the per-head ones times 2^-6
    pg.quest_sparse_decode_fp8(out_h, q, kc_h, vc_h, ksh, vsh, bt, ctx, sel_h, w.scale, workspace=ws)
    pg.quest_sparse_decode_fp8_block(out_b, q, kc_b, vc_b, ksb, vsb, bt, ctx, sel_b, w.scale, workspace=ws)
    assert torch.equal(out_h.view(torch.int16), out_b.view(torch.int16))
    qws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, Hkv, D, w.MBS), dtype=torch.uint8, device=d)
    pg.quest_decode_fp8(out_h, sel_h, q, kmin, kmax, kc_h, vc_h, ksh, vsh, bt, ctx, w.topk, w.scale, workspace=qws)
    pg.quest_decode_fp8_block(out_b, sel_b, q, kmin, kmax, kc_b, vc_b, ksb, vsb, bt, ctx, w.topk, w.scale,
                              workspace=qws)
    assert torch.equal(sel_h, sel_b) and torch.equal(out_h.view(torch.int16), out_b.view(torch.int16))
