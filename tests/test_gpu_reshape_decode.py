"""pa_reshape_and_decode and quest_reshape_and_decode: the step's write
folded into the step's first launch.

Each call starts from the cache and metadata as they were before the step
(metadata rebuilt over the positions before each sequence's new token) and
is compared with the separate calls on a copy of that state:
quest_reshape_and_cache with the same slots, then pa_decode / quest_decode.
Caches, metadata, selection and outputs must be equal byte for byte; the
outputs are also held to the oracle (its write with the slots the fused
call writes, then its attention) within the attention tolerances.

The fused calls write token b only at the slot of position ctx_b - 1 of
sequence b. The cases include padding slots (-1) and, in one case, slots
that point elsewhere in the pool, which the fused calls must leave alone."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import assert_close_attention, gather_rows, sample_rows, to_dev_bf16, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_gqa_decode_reshape_gb300.build as b
    b.build()


def position_slots(w):
    """The slot of position ctx_b - 1 of every sequence (-1 where there is none)."""
    out = np.full(w.B, -1, dtype=np.int64)
    for b in range(w.B):
        c = min(max(int(w.context_lens[b]), 0), w.MBS * w.BS)
        if c == 0:
            continue
        p = int(w.block_tables[b, (c - 1) // w.BS])
        if 0 <= p < w.NB:
            out[b] = p * w.BS + (c - 1) % w.BS
    return out


def written_slots(w, slots):
    """What the fused calls write: slot b where it is position ctx_b - 1's slot, else nothing."""
    pos = position_slots(w)
    return np.where((slots >= 0) & (slots == pos), slots, -1).astype(np.int64)


class State:
    """The cache, pre-step metadata and buffers of one workload on the GPU."""

    def __init__(self, w, slots):
        import paged_gqa_decode_reshape_gb300 as pg
        d = torch.device("cuda:0")
        self.w, self.pg, self.d = w, pg, d
        self.kc = to_dev_bf16(w.key_cache, d)
        self.vc = to_dev_bf16(w.value_cache, d)
        self.q = to_dev_bf16(w.q, d)
        self.key = to_dev_bf16(w.key, d)
        self.value = to_dev_bf16(w.value, d)
        self.slots = torch.from_numpy(slots).to(d)
        self.bt = torch.from_numpy(w.block_tables).to(d)
        self.ctx = torch.from_numpy(w.context_lens).to(d)
        pre = torch.from_numpy((w.context_lens - 1).clip(0).astype(np.int32)).to(d)
        self.kmin = torch.zeros((w.NB, w.Hkv, w.D), dtype=torch.bfloat16, device=d)
        self.kmax = torch.zeros_like(self.kmin)
        pg.quest_rebuild_meta(self.kmin, self.kmax, self.kc, self.bt, pre)
        self.out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=d)
        self.sel = torch.full((w.B, w.Hkv, w.topk), -7, dtype=torch.int32, device=d)
        self.ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D), dtype=torch.uint8, device=d)
        self.qws = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS), dtype=torch.uint8,
                               device=d)

    def clone(self):
        c = State.__new__(State)
        c.__dict__.update(self.__dict__)
        for k in ("kc", "vc", "kmin", "kmax", "out", "sel", "ws", "qws"):
            setattr(c, k, getattr(self, k).clone())
        return c


def same(a: torch.Tensor, b: torch.Tensor, what: str):
    assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b), what


def check(w, slots=None, max_ctas=0, sample=None):
    slots = w.slot_mapping if slots is None else slots
    rows = None if sample is None else sample_rows(w, sample, 29)

    def pick(t):
        got = to_host_f64(t)
        return got if rows is None else gather_rows(got, rows)

    wr = written_slots(w, slots)
    fused, sep = State(w, slots), State(w, wr)
    pg = fused.pg
    # the oracle: its write with the slots the fused call writes, then attention
    okc, ovc = w.key_cache.copy(), w.value_cache.copy()
    oracle.reshape_and_cache(w.key, w.value, okc, ovc, wr)

    # dense, with the metadata update
    f, s = fused.clone(), sep.clone()
    pg.pa_reshape_and_decode(f.out, f.q, f.key, f.value, f.slots, f.kc, f.vc, f.bt, f.ctx, w.scale,
                             kmin=f.kmin, kmax=f.kmax, workspace=f.ws)
    pg.quest_reshape_and_cache(s.key, s.value, s.kc, s.vc, s.kmin, s.kmax, s.slots)
    pg.pa_decode(s.out, s.q, s.kc, s.vc, s.bt, s.ctx, w.scale, workspace=s.ws)
    for name in ("kc", "vc", "kmin", "kmax", "out"):
        same(getattr(f, name), getattr(s, name), f"{w.name} pa_reshape_and_decode: {name}")
    np.testing.assert_array_equal(f.kc.view(torch.int16).cpu().numpy().view(np.uint16), okc)
    want = oracle.paged_attention(w.q, okc, ovc, w.block_tables, w.context_lens, w.scale, rows=rows)
    assert_close_attention(pick(f.out), want, f"{w.name} pa_reshape_and_decode vs oracle")
    assert pg.pa_workspace_status(f.ws) == 0

    # dense without metadata
    f = fused.clone()
    pg.pa_reshape_and_decode(f.out, f.q, f.key, f.value, f.slots, f.kc, f.vc, f.bt, f.ctx, w.scale, workspace=f.ws)
    same(f.kc, s.kc, "kc (no metadata)")
    same(f.out, s.out, "out (no metadata)")
    same(f.kmin, fused.kmin, "metadata left alone")

    # Quest
    f, s = fused.clone(), sep.clone()
    pg.quest_reshape_and_decode(f.out, f.sel, f.q, f.key, f.value, f.slots, f.kmin, f.kmax, f.kc, f.vc, f.bt,
                                f.ctx, w.topk, w.scale, max_ctas=max_ctas, workspace=f.qws)
    pg.quest_reshape_and_cache(s.key, s.value, s.kc, s.vc, s.kmin, s.kmax, s.slots)
    pg.quest_decode(s.out, s.sel, s.q, s.kmin, s.kmax, s.kc, s.vc, s.bt, s.ctx, w.topk, w.scale,
                    max_ctas=max_ctas, workspace=s.qws)
    for name in ("kc", "vc", "kmin", "kmax", "sel", "out"):
        same(getattr(f, name), getattr(s, name), f"{w.name} quest_reshape_and_decode: {name}")
    kmin, kmax = oracle.quest_rebuild_meta(okc, w.block_tables, w.context_lens)
    sel = oracle.quest_select_kernel_order(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, w.topk)
    np.testing.assert_array_equal(f.sel.cpu().numpy(), sel)
    want = oracle.sparse_attention(w.q, okc, ovc, w.block_tables, w.context_lens, sel, w.scale, rows=rows)
    assert_close_attention(pick(f.out), want, f"{w.name} quest_reshape_and_decode vs oracle")
    assert pg.pa_workspace_status(f.qws) == 0


SMALL = {
    "tiny": ("tiny", {}),
    "quest_small": ("quest_8k", dict(batch=4, ctx_scale=0.05, topk=6)),
    "mixed_small": ("mixed_b128", dict(batch=16, ctx_scale=0.02, topk=8)),
    "long_small": ("long_40k", dict(batch=2, ctx_scale=0.02, topk=16)),
    "dense_small": ("dense_b32", dict(batch=6, ctx_scale=0.05, topk=8)),
}


@pytest.mark.parametrize("case", list(SMALL))
def test_small(case):
    name, kw = SMALL[case]
    check(workloads.make(name, **kw), max_ctas=0)


@pytest.mark.parametrize("name", ["quest_8k", "long_40k", "mixed_b128"])
def test_full_size(name):
    check(workloads.make(name), max_ctas=76, sample=48)


def test_slots_elsewhere_are_not_written():
    """Slots that are not position ctx_b - 1's slot (another block of the
    pool, another offset, -1) are not written by the fused calls."""
    w = workloads.make("quest_8k", batch=6, ctx_scale=0.05, topk=6)
    slots = position_slots(w)
    # the positions these tokens would fill hold finite values before the step
    # (the workload poisons them with NaN, expecting the step's write)
    for b in (1, 2, 3):
        p, o = divmod(int(slots[b]), w.BS)
        w.key_cache[p, o] = w.key[0]
        w.value_cache[p, o] = w.value[0]
    slots[1] = -1
    slots[2] = slots[2] + 1 if (slots[2] + 1) % w.BS else slots[2] - 1  # another offset of the block
    used = set(np.unique(w.block_tables[w.block_tables >= 0]).tolist())
    spare = [p for p in range(w.NB) if p not in used]
    if spare:
        slots[3] = spare[0] * w.BS
    check(w, slots=slots)
