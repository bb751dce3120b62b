"""The Quest selection against the method's definition, on the CPU.

The fp32 kernel-order selection (the set the CUDA kernels must reproduce bit
for bit) is compared with the top-K of the plain fp64 scores on the full-size
workloads, bf16 and 8-bit metadata; every difference must lie within the fp32
score error bound (tests/selection_check.py), and the number of such exempt
rows is printed. The checker itself is shown to reject planted mistakes.
"""

import numpy as np
import pytest

import oracle
import workloads
from tests.selection_check import check_selection, score_error_bound

CASES = {
    "tiny": ("tiny", {}),
    "dense_b32": ("dense_b32", dict(topk=64)),
    "quest_8k": ("quest_8k", {}),
    "long_40k": ("long_40k", {}),
    # every context length drawn from the full distribution, a smaller batch
    "mixed_b128_b16": ("mixed_b128", dict(batch=16)),
}


def _meta(w, fp8=False):
    if not fp8:
        return oracle.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    ks, vs = workloads.fp8_scales(w.Hkv)
    NB, BS = w.NB, w.BS
    kc = np.zeros((NB, BS, w.Hkv, w.D), dtype=np.uint8)
    vc = np.zeros((NB, w.Hkv, w.D, BS), dtype=np.uint8)
    oracle.reshape_and_cache_fp8(w.key_cache.reshape(NB * BS, w.Hkv, w.D),
                                 w.value_cache.reshape(NB * BS, w.Hkv, w.D), kc, vc,
                                 np.arange(NB * BS, dtype=np.int64), ks, vs)
    return oracle.quest_rebuild_meta_fp8(kc, w.block_tables, w.context_lens)


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("case", list(CASES))
def test_kernel_order_selection_within_bound_of_plain(case, fp8):
    name, kw = CASES[case]
    w = workloads.make(name, poison=False, **kw)
    kmin, kmax = _meta(w, fp8)
    args = (w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS)
    if fp8:
        plain, absum = oracle.quest_scores_fp8(*args, with_abs=True)
        korder = oracle.quest_scores_kernel_order_fp8(*args)
    else:
        plain, absum = oracle.quest_scores(*args, with_abs=True)
        korder = oracle.quest_scores_kernel_order(*args)
    sel = oracle.quest_topk(korder, w.context_lens, w.BS, w.topk)
    n = check_selection(sel, plain, absum, w.context_lens, w.BS, w.topk, w.Hq // w.Hkv, w.D,
                        f"{case} {'fp8' if fp8 else 'bf16'} kernel-order selection")
    assert n <= w.B * w.Hkv


def _small():
    w = workloads.make("quest_8k", poison=False, batch=3, ctx_scale=0.1, topk=8)
    kmin, kmax = oracle.quest_rebuild_meta(w.key_cache, w.block_tables, w.context_lens)
    plain, absum = oracle.quest_scores(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, with_abs=True)
    sel = oracle.quest_topk(plain, w.context_lens, w.BS, w.topk)
    return w, plain, absum, sel


def _check(w, sel, plain, absum):
    return check_selection(sel, plain, absum, w.context_lens, w.BS, w.topk, w.Hq // w.Hkv, w.D, "planted")


def test_checker_accepts_exact_top_k():
    w, plain, absum, sel = _small()
    assert _check(w, sel, plain, absum) == 0


@pytest.mark.parametrize("slip", ["lowest_block", "descending", "duplicate", "padding", "out_of_range"])
def test_checker_rejects_planted_mistakes(slip):
    w, plain, absum, sel = _small()
    bad = sel.copy()
    row = bad[1, 2]
    nb = w.num_blocks()[1]
    if slip == "lowest_block":      # the lowest-scoring block in place of a selected one
        s = plain[1, 2, :nb]
        low = int(np.argmin(s))
        assert low not in row
        row[0] = low
        row.sort()
    elif slip == "descending":
        row[:] = row[::-1]
    elif slip == "duplicate":
        row[1] = row[0]
    elif slip == "padding":
        row[-1] = -1
    elif slip == "out_of_range":
        row[-1] = nb
    with pytest.raises(AssertionError):
        _check(w, bad, plain, absum)


def test_checker_exempts_a_near_tie_within_the_bound():
    """Move the best unselected block to within E of the K-th selected one:
    a set that swaps the two is then explained by fp32 rounding (exempt), and
    one block further out is not."""
    w, plain, absum, sel = _small()
    p = plain.copy()
    b, h = 1, 2
    nb = w.num_blocks()[b]
    s = p[b, h, :nb]
    E = score_error_bound(absum, w.Hq // w.Hkv, w.D)[b, h, :nb]
    row = sel[b, h]
    kth = row[np.argmin(s[row])]                     # the weakest selected block
    out = [j for j in np.argsort(-s) if j not in row]
    c = out[0]
    s[c] = s[kth] - 0.5 * (E[kth] + E[c])            # a near tie below the K-th place
    swapped = sel.copy()
    r = swapped[b, h]
    r[r == kth] = c
    r.sort()
    assert _check(w, swapped, p, absum) == 1
    s[c] = s[kth] - 2.0 * (E[kth] + E[c])            # beyond the bound: rejected
    with pytest.raises(AssertionError):
        _check(w, swapped, p, absum)
