"""Check a Quest selection against the method's own definition of the score.

The score of a logical block ("Ascend Kernel-to-Serving Pipeline", section
"Quest Sparse Attention"; the bound itself comes from the statement of the
method) is

    s_j = sum_{h in group} sum_d max(q[h,d] * min_j[d], q[h,d] * max_j[d]),

and the selection is the top-K blocks, ties to the lower index. The oracle
computes s_j term by term in fp64 (``oracle.quest_scores``), together with
A_j = sum_h sum_d |q[h,d]| * max(|min_j[d]|, |max_j[d]|).

The CUDA kernel evaluates the same sum in fp32. Every quantity it forms is a
sum or a product of the exact terms, so its rounding error obeys the standard
forward bound for an expression evaluated with rounding depth n (at most n
roundings on the path from any input to the result):

    |fl32(s_j) - s_j| <= gamma_n * A_j,   gamma_n = n*u / (1 - n*u), u = 2^-24.

The kernel's evaluation (group sums P_d, N_d of the positive and negative
query parts over G heads; the products with max_d and min_d and their sum;
D/32 dims summed per lane; five butterfly levels) has depth
n = (G - 1) + 2 + (D/32 - 1) + 5 = G + D/32 + 5. The oracle's own fp64 sum
adds at most gamma_{G*D} (u = 2^-53) times A_j. E_j is the sum of both.

A selected set S of a row is accepted when it is a valid selection (ascending
distinct block indices below the row's block count, min(K, nblk) of them,
padded with -1) and some choice of fp32 scores within E_j of the exact ones
ranks S first:

    min_{a in S} (s_a + E_a) >= max_{c not in S} (s_c - E_c).

A row whose set differs from the exact top-K but passes this test is an
"exempt" row: the difference is explained by a score gap at the K-th place
within the fp32 error bound. Any other difference fails.
"""

from __future__ import annotations

import numpy as np


def gamma(n: int, u: float) -> float:
    return n * u / (1.0 - n * u)


def score_error_bound(abs_sum: np.ndarray, G: int, D: int) -> np.ndarray:
    """E_j: bound on |fp32 kernel-order score - fp64 plain score| per block."""
    n32 = G + D // 32 + 5
    return (gamma(n32, 2.0 ** -24) + gamma(G * D, 2.0 ** -53)) * abs_sum


def check_selection(sel: np.ndarray, plain: np.ndarray, abs_sum: np.ndarray, context_lens: np.ndarray,
                    BS: int, topk: int, G: int, D: int, what: str = "selection") -> int:
    """Assert that every row of ``sel`` [B, Hkv, topk] is the top-K of the
    plain scores ``plain`` [B, Hkv, MBS] up to the fp32 error bound; return
    the number of exempt rows (sets that differ from the exact top-K)."""
    B, Hkv, K = sel.shape
    assert K == topk
    E = score_error_bound(abs_sum, G, D)
    exempt = []
    for b in range(B):
        nblk = min((max(int(context_lens[b]), 0) + BS - 1) // BS, plain.shape[2])
        k = min(topk, nblk)
        for h in range(Hkv):
            row = sel[b, h]
            where = f"{what}: row (b={b}, kvh={h})"
            assert (row[k:] == -1).all(), f"{where}: padding {row[k:]} (expected {topk - k} x -1)"
            s_set = row[:k]
            assert ((s_set >= 0) & (s_set < nblk)).all(), f"{where}: index out of range {s_set}"
            assert (np.diff(s_set) > 0).all(), f"{where}: not ascending and distinct {s_set}"
            s, e = plain[b, h, :nblk], E[b, h, :nblk]
            order = np.lexsort((np.arange(nblk), -s))           # score desc, index asc
            exact = np.sort(order[:k])
            if np.array_equal(exact, s_set):
                continue
            inside = np.zeros(nblk, dtype=bool)
            inside[s_set] = True
            lo_in = float(np.min(s[inside] + e[inside]))
            hi_out = float(np.max(s[~inside] - e[~inside]))
            assert lo_in >= hi_out, (
                f"{where}: set differs from the exact top-{k} beyond the fp32 error bound "
                f"(min over set of s+E = {lo_in!r} < max outside of s-E = {hi_out!r}); "
                f"got {sorted(set(s_set) - set(exact))} in place of {sorted(set(exact) - set(s_set))}")
            exempt.append((b, h))
    print(f"{what}: {B * Hkv} rows, {len(exempt)} exempt (set differs from the exact fp64 top-K "
          f"within the fp32 score error bound){': ' + str(exempt) if exempt else ''}")
    return len(exempt)
