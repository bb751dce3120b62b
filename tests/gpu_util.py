"""Helpers shared by the GPU tests: move a workload to the device, run the
CUDA path through the C ABI binding, run the oracle on the same inputs, and
compare with the tolerances of the method's statement (attention outputs
within max-abs 1e-2 and mean-abs 1e-3 of the oracle; caches, metadata and
selections bit-exact). The output is bf16, so the mean-abs bound counts on
top of the error that rounding the exact result to bf16 already carries:
about 1e-5 on the benchmark workloads, about 1e-3 on a batch whose rows each
attend to one token (each output row is then one V row, of magnitude ~1)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_gqa_decode_reshape_gb300 as pg
from tests.selection_check import check_selection
from workloads import bf16_bits_to_f32, f32_to_bf16_bits

MAX_ABS_TOL = 1e-2
MEAN_ABS_TOL = 1e-3


def to_dev_bf16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def to_host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DeviceStep:
    """A workload's tensors on the GPU, plus outputs and workspaces."""

    def __init__(self, w, dev="cuda:0"):
        self.w = w
        self.dev = torch.device(dev)
        d = self.dev
        self.q = to_dev_bf16(w.q, d)
        self.kc = to_dev_bf16(w.key_cache, d)
        self.vc = to_dev_bf16(w.value_cache, d)
        self.key = to_dev_bf16(w.key, d)
        self.value = to_dev_bf16(w.value, d)
        self.slots = torch.from_numpy(w.slot_mapping).to(d)
        self.bt = torch.from_numpy(w.block_tables).to(d)
        self.ctx = torch.from_numpy(w.context_lens).to(d)
        self.out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=d)
        self.out_sparse = torch.empty_like(self.out)
        self.kmin = torch.zeros((w.NB, w.Hkv, w.D), dtype=torch.bfloat16, device=d)
        self.kmax = torch.zeros_like(self.kmin)
        self.sel = torch.empty((w.B, w.Hkv, w.topk), dtype=torch.int32, device=d)
        self.ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D), dtype=torch.uint8,
                              device=d)
        self.sel_ws = torch.zeros(pg.quest_select_workspace_size(w.B, w.Hkv, w.MBS), dtype=torch.uint8,
                                  device=d)

    def reshape(self):
        pg.pa_reshape_and_cache(self.key, self.value, self.kc, self.vc, self.slots)

    def decode(self):
        w = self.w
        pg.pa_decode(self.out, self.q, self.kc, self.vc, self.bt, self.ctx, w.scale, workspace=self.ws)
        return self.out

    def select(self):
        pg.quest_select_topk(self.sel, self.q, self.kmin, self.kmax, self.bt, self.ctx, self.w.BS,
                             workspace=self.sel_ws)
        return self.sel

    def sparse(self, sel: torch.Tensor):
        w = self.w
        pg.quest_sparse_decode(self.out_sparse, self.q, self.kc, self.vc, self.bt, self.ctx, sel,
                               w.scale, workspace=self.ws)
        return self.out_sparse

    def scores(self) -> np.ndarray:
        w = self.w
        n = w.B * w.Hkv * w.MBS
        return self.sel_ws[: n * 4].view(torch.float32).cpu().numpy().reshape(w.B, w.Hkv, w.MBS)


class OracleStep:
    """The same step through the CPU oracle (host copies of the caches)."""

    def __init__(self, w):
        self.w = w
        self.kc = w.key_cache.copy()
        self.vc = w.value_cache.copy()

    def reshape(self):
        oracle.reshape_and_cache(self.w.key, self.w.value, self.kc, self.vc, self.w.slot_mapping)

    def rebuild_meta(self):
        w = self.w
        self.kmin, self.kmax = oracle.quest_rebuild_meta(self.kc, w.block_tables, w.context_lens)
        return self.kmin, self.kmax

    def dense(self, rows=None):
        w = self.w
        return oracle.paged_attention(w.q, self.kc, self.vc, w.block_tables, w.context_lens, w.scale,
                                      rows=rows)

    def scores(self, kmin, kmax):
        """fp32 scores in the kernel's evaluation order (bit-exact reproduction)."""
        w = self.w
        return oracle.quest_scores_kernel_order(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS)

    def select(self, kmin, kmax):
        """Top-K of the kernel-order scores: the CUDA path's exact set."""
        w = self.w
        return oracle.quest_topk(self.scores(kmin, kmax), w.context_lens, w.BS, w.topk)

    def check_plain(self, sel, kmin, kmax, fp8: bool = False, what: str = "selection") -> int:
        """The selected sets against the top-K of the plain fp64 scores (the
        method's definition), exact up to the fp32 score error bound; returns
        the number of exempt rows."""
        w = self.w
        fn = oracle.quest_scores_fp8 if fp8 else oracle.quest_scores
        plain, absum = fn(w.q, kmin, kmax, w.block_tables, w.context_lens, w.BS, with_abs=True)
        return check_selection(np.asarray(sel), plain, absum, w.context_lens, w.BS, w.topk,
                               w.Hq // w.Hkv, w.D, what)

    def sparse(self, sel, rows=None):
        w = self.w
        return oracle.sparse_attention(w.q, self.kc, self.vc, w.block_tables, w.context_lens, sel,
                                       w.scale, rows=rows)


def assert_close_attention(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite outputs"
    err = np.abs(got - want)
    max_abs, mean_abs = float(err.max()), float(err.mean())
    # the mean-abs error of the exact result rounded to the bf16 output
    floor = float(np.abs(bf16_bits_to_f32(f32_to_bf16_bits(want.astype(np.float32))) - want).mean())
    mean_tol = MEAN_ABS_TOL + floor
    print(f"{what}: max_abs={max_abs:.3e} mean_abs={mean_abs:.3e} (bf16 rounding floor {floor:.1e}) "
          f"{'PASS' if max_abs <= MAX_ABS_TOL and mean_abs <= mean_tol else 'FAIL'}")
    assert max_abs <= MAX_ABS_TOL, f"{what}: max-abs error {max_abs:.3e} > {MAX_ABS_TOL}"
    assert mean_abs <= mean_tol, f"{what}: mean-abs error {mean_abs:.3e} > {MEAN_ABS_TOL} + {floor:.1e}"


def sample_rows(w, n: int, seed: int):
    """A seeded sample of (b, h) pairs that always includes each sequence's
    first and last query head and the longest and shortest sequences."""
    rng = np.random.default_rng(seed)
    rows = {(int(b), int(h)) for b, h in zip(rng.integers(0, w.B, n), rng.integers(0, w.Hq, n))}
    for b in (int(np.argmax(w.context_lens)), int(np.argmin(w.context_lens))):
        rows.add((b, 0))
        rows.add((b, w.Hq - 1))
    return np.array(sorted(rows), dtype=np.int32)


def gather_rows(t: np.ndarray, rows: np.ndarray) -> np.ndarray:
    return t[rows[:, 0], rows[:, 1]]
