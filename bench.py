"""Benchmark of the paged decode hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input, every
call through the C ABI: ReshapeAndCache + Quest metadata update (one launch),
then the dense GQA paged decode (split-KV + combine) on the calling stream
and, beside it on a second stream, the Quest path: block scores and top-K,
then the sparse decode on SMs the dense decode leaves to it (step_runner;
--serial runs write, quest_decode and the dense decode one after another).
Inputs are resident in HBM before timing; the L2 is flushed (a 512 MiB write)
before every step, outside the timed events. The step time comes from one
event pair per step; a second pass of the same steps, on one stream with an
event between calls, gives the per-call breakdown and the roofline of the
dominant kernel (the dense decode).

Prints ONE JSON line (rank 0). With --impl reference it times the CPU oracle
instead (a bounded sample of the same workload per step).

Multi-GPU: the path shards by sequence with no exchange, so N ranks run N
independent replicas (weak scaling); the ranks only meet for the timing
barrier and the max-over-ranks reduction.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

METRIC = "decode-attn KV GB/s & % HBM roofline; µs/step dense vs Quest at 8K/40K ctx"
UNIT = "GB/s"
L2_FLUSH_BYTES = 512 << 20
# Before each device-timed sample a short spin kernel (outside the events)
# lets the host enqueue the whole step before the GPU reaches it, so a
# device-timed interval never waits on Python's launch overhead.
HEAD_START_CYCLES = 400_000
NOMINAL_HBM_GBS = 8000.0  # the GB300's ~8 TB/s HBM3e peak (nominal)


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", default="quest_8k",
                   choices=["tiny", "dense_b32", "quest_8k", "long_40k", "mixed_b128"])
    p.add_argument("--kv", choices=["bf16", "fp8", "fp8_block"], default="bf16",
                   help="KV-cache element type: bf16, or 8-bit E4M3 codes with per-KV-head scales")
    p.add_argument("--qlen", type=int, default=1,
                   help="query rows per sequence of the dense call (> 1: pa_decode_multi, right-aligned "
                        "causal masks, for speculative / chunked-prefill rows)")
    p.add_argument("--serial", action="store_true",
                   help="run the step's calls one after another on one stream (default: the Quest "
                        "selection and sparse decode on a second stream, alongside the dense decode)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-head-start", action="store_true",
                   help="no spin kernel before each device-timed sample (the host may then lag the GPU)")
    p.add_argument("--no-long-point", action="store_true",
                   help="skip the 40K-context point (long_40k) that the default quest_8k line also reports")
    p.add_argument("--cpu-budget", type=float, default=12.0,
                   help="seconds of oracle work for the CPU baseline sample")
    return p.parse_args()


# ----------------------------------------------------------------- helpers


def measured_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from an ncu capture, if it was taken on the
    current sources of the kernel (else None). `source` names the files the
    kernel is compiled from, joined by '+'; `source_sha` is the first 16 hex
    digits of the SHA-256 of their contents in that order."""
    path = os.path.join(HERE, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(kernel, {}).get(workload)
    if not ent:
        return None
    sha = sources_sha(ent["source"])
    if sha is None or sha != ent.get("source_sha"):
        return None
    return int(ent["dram_bytes_per_launch"])


def sources_sha(source: str):
    """First 16 hex digits of the SHA-256 of the '+'-joined csrc files, in order."""
    import hashlib
    h = hashlib.sha256()
    for name in source.split("+"):
        src = os.path.join(HERE, "paged_gqa_decode_reshape_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except ValueError:
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(torch, dev) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        idx = dev.index or 0
        return parts[idx] if idx < len(parts) else str(idx)


# --------------------------------------------------------------- the step


def arena(torch, dev, specs):
    """One device buffer holding several tensors (each 256-byte aligned), so a
    step's inputs (or outputs) move between host and device in one copy.
    specs: [(name, shape, torch dtype)]. Returns (buffer, {name: view})."""
    offs, off = {}, 0
    for name, shape, dt in specs:
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        offs[name] = (off, n)
        off += (n + 255) // 256 * 256
    buf = torch.empty(max(off, 256), dtype=torch.uint8, device=dev)
    views = {name: buf[o: o + n].view(dt).view(shape) for (name, shape, dt), (o, n) in zip(specs, offs.values())}
    return buf, views


class Step:
    """Device buffers of one workload and the five C-ABI calls of a step."""

    def __init__(self, w, dev, kv: str = "bf16", qlen: int = 1):
        import torch
        import paged_gqa_decode_reshape_gb300 as pg
        import workloads
        self.pg, self.torch, self.w, self.dev, self.kv, self.qlen = pg, torch, w, dev, kv, qlen
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count
        def d16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

        # the step's inputs in one device buffer and its results in another
        # (one host<->device copy each way per step end to end)
        bf, i32, i64 = torch.bfloat16, torch.int32, torch.int64
        ins = [("q", w.q.shape, bf), ("key", w.key.shape, bf), ("value", w.value.shape, bf),
               ("slots", w.slot_mapping.shape, i64), ("bt", w.block_tables.shape, i32),
               ("ctx", w.context_lens.shape, i32)]
        outs = [("out", (w.B, w.Hq, w.D), bf), ("out_sparse", (w.B, w.Hq, w.D), bf),
                ("sel", (w.B, w.Hkv, w.topk), i32)]
        if qlen > 1:
            ins.append(("q_multi", (w.B * qlen, w.Hq, w.D), bf))
            outs.append(("out_multi", (w.B * qlen, w.Hq, w.D), bf))
        self.in_buf, iv = arena(torch, dev, ins)
        self.out_buf, ov = arena(torch, dev, outs)
        for name, t in list(iv.items()) + list(ov.items()):
            setattr(self, name, t)
        self.q.copy_(d16(w.q))
        self.key.copy_(d16(w.key))
        self.value.copy_(d16(w.value))
        self.slots.copy_(torch.from_numpy(w.slot_mapping))
        self.bt.copy_(torch.from_numpy(w.block_tables))
        self.ctx.copy_(torch.from_numpy(w.context_lens))
        if qlen > 1:
            # qlen query rows per sequence (seeded N(0, 1), bf16) for pa_decode_multi
            rng = np.random.default_rng(1234)
            qm = workloads.f32_to_bf16_bits(rng.standard_normal((w.B * qlen, w.Hq, w.D)).astype(np.float32))
            self.q_multi.copy_(torch.from_numpy(qm.view(np.int16)).view(torch.bfloat16))
            self.cu_q = torch.arange(0, w.B * qlen + 1, qlen, dtype=torch.int32, device=dev)
            self.ws_multi = torch.zeros(pg.pa_decode_multi_workspace_size(w.B * qlen, w.Hq, w.Hkv, w.D),
                                        dtype=torch.uint8, device=dev)
        self.kc = d16(w.key_cache)
        self.vc = d16(w.value_cache)
        self.kmin = torch.zeros((w.NB, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
        self.kmax = torch.zeros_like(self.kmin)
        self.ws = torch.zeros(pg.pa_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D), dtype=torch.uint8,
                              device=dev)
        # the sparse decode's own workspace: it may run at the same time as the dense one
        self.ws_sparse = torch.zeros_like(self.ws)
        self.sel_ws = torch.zeros(pg.quest_select_workspace_size(w.B, w.Hkv, w.MBS),
                                  dtype=torch.uint8, device=dev)
        self.ws_quest = torch.zeros(pg.quest_decode_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.MBS),
                                    dtype=torch.uint8, device=dev)
        if kv in ("fp8", "fp8_block"):
            # the 8-bit pool: every slot of the bf16 pool quantised once (setup),
            # with fixed per-KV-head scales or with per-block scales
            NB, BS = w.NB, w.BS
            if kv == "fp8":
                ks, vs = workloads.fp8_scales(w.Hkv)
                self.k_scale, self.v_scale = torch.from_numpy(ks).to(dev), torch.from_numpy(vs).to(dev)
            else:
                self.k_scale = torch.zeros((NB, w.Hkv), dtype=torch.float32, device=dev)
                self.v_scale = torch.zeros_like(self.k_scale)
            kc8 = torch.empty((NB, BS, w.Hkv, w.D), dtype=torch.uint8, device=dev)
            vc8 = torch.empty((NB, w.Hkv, w.D, BS), dtype=torch.uint8, device=dev)
            write = pg.pa_reshape_and_cache_fp8 if kv == "fp8" else pg.pa_reshape_and_cache_fp8_block
            write(self.kc.view(NB * BS, w.Hkv, w.D), self.vc.view(NB * BS, w.Hkv, w.D), kc8, vc8,
                  torch.arange(NB * BS, dtype=torch.int64, device=dev), self.k_scale, self.v_scale)
            torch.cuda.synchronize(dev)
            self.kc, self.vc = kc8, vc8
            self.kmin = torch.zeros((w.NB, w.Hkv, w.D), dtype=torch.uint8, device=dev)
            self.kmax = torch.zeros_like(self.kmin)
            self.calls()[0]()  # the step's write path once, then the metadata as they stand
            pg.quest_rebuild_meta_fp8(self.kmin, self.kmax, self.kc, self.bt, self.ctx)
            torch.cuda.synchronize(dev)
            return
        # Quest metadata of the cache as it stands (setup, not timed)
        pg.pa_reshape_and_cache(self.key, self.value, self.kc, self.vc, self.slots)
        pg.quest_rebuild_meta(self.kmin, self.kmax, self.kc, self.bt, self.ctx)
        torch.cuda.synchronize(dev)

    def quest(self, max_ctas: int = 0):
        """The Quest path after the write: quest_decode (block scores, then
        one launch that selects each segment's top-K and attends over it),
        on at most max_ctas CTAs (0: one per SM)."""
        pg, w = self.pg, self.w
        if self.kv != "bf16":
            fn = pg.quest_decode_fp8 if self.kv == "fp8" else pg.quest_decode_fp8_block
            return lambda: fn(self.out_sparse, self.sel, self.q, self.kmin, self.kmax, self.kc, self.vc,
                              self.k_scale, self.v_scale, self.bt, self.ctx, w.topk, w.scale, max_ctas=max_ctas,
                              workspace=self.ws_quest)
        return lambda: pg.quest_decode(self.out_sparse, self.sel, self.q, self.kmin, self.kmax, self.kc, self.vc,
                                       self.bt, self.ctx, w.topk, w.scale, max_ctas=max_ctas,
                                       workspace=self.ws_quest)

    def split_ctas(self) -> int:
        """SMs the two-stream step keeps for the sparse decode (0: none, for
        multi-token rows). The dense decode runs
        on the others from the step's start, so the sparse decode need not
        wait for its CTAs. X = 1.8 x SMs x the sparse share of the two decode
        calls' KV tokens, to a multiple of 8, at least 16 and at most half
        the SMs: the sparse share of the SMs, raised because the sparse call
        starts after the selection. Measured against every X from 8 to 56 on
        quest_8k, long_40k, dense_b32 and mixed_b128, the rule picks the
        fastest step on each."""
        if self.qlen > 1:
            return 0
        import numpy as np
        w = self.w
        ctx = np.minimum(np.asarray(w.context_lens, dtype=np.int64), w.MBS * w.BS)
        dense = float(ctx.sum())
        sparse = float(np.minimum(ctx, w.topk * w.BS).sum())
        x = int(round(1.8 * self.sms * sparse / max(dense + sparse, 1.0) / 8.0)) * 8
        return max(16, min(x, self.sms // 2))

    def dense_beside(self):
        """The dense decode as the two-stream step runs it: on the SMs the
        sparse decode does not keep (pa_decode_budget), else pa_decode."""
        x = self.split_ctas()
        c = self.calls()[CALL_NAMES.index("dense")]
        if x == 0:
            return c
        pg, w, n = self.pg, self.w, self.sms - x
        if self.kv != "bf16":
            fn = pg.pa_decode_fp8_budget if self.kv == "fp8" else pg.pa_decode_fp8_block_budget
            return lambda: fn(self.out, self.q, self.kc, self.vc, self.k_scale, self.v_scale, self.bt, self.ctx,
                              w.scale, n, workspace=self.ws)
        return lambda: pg.pa_decode_budget(self.out, self.q, self.kc, self.vc, self.bt, self.ctx, w.scale, n,
                                           workspace=self.ws)

    def quest_beside(self):
        """The Quest path as the two-stream step runs it, beside the dense
        decode: quest_select_topk, whose CTAs fit on the SMs beside the dense
        decode's, then the sparse decode on the SMs split_ctas() keeps for it
        (its CTAs need a whole SM's shared memory). quest_decode would put its
        top-K after the dense decode instead of beside it."""
        pg, w = self.pg, self.w
        budget = self.split_ctas() or self.sms // 2
        select = self.calls()[CALL_NAMES.index("select")]
        if self.kv != "bf16":
            fn = pg.quest_sparse_decode_fp8_budget if self.kv == "fp8" else pg.quest_sparse_decode_fp8_block
            sparse = lambda: fn(self.out_sparse, self.q, self.kc, self.vc, self.k_scale, self.v_scale, self.bt,
                                self.ctx, self.sel, w.scale, budget, workspace=self.ws_sparse)
        else:
            sparse = lambda: pg.quest_sparse_decode_budget(self.out_sparse, self.q, self.kc, self.vc, self.bt,
                                                           self.ctx, self.sel, w.scale, budget,
                                                           workspace=self.ws_sparse)

        def run():
            select()
            sparse()
        return run

    def calls(self):
        """The step's C-ABI calls: the write path (ReshapeAndCache and the
        metadata update in one launch), dense decode, Quest selection (score +
        top-K launches), Quest sparse decode on that selection, and the fused
        Quest path (quest_decode: score launch, then top-K + sparse decode in
        one launch), which the step uses."""
        pg, w = self.pg, self.w
        if self.kv == "fp8":
            return [
                lambda: pg.quest_reshape_and_cache_fp8(self.key, self.value, self.kc, self.vc, self.kmin,
                                                       self.kmax, self.slots, self.k_scale, self.v_scale),
                lambda: pg.pa_decode_fp8(self.out, self.q, self.kc, self.vc, self.k_scale, self.v_scale,
                                         self.bt, self.ctx, w.scale, workspace=self.ws),
                lambda: pg.quest_select_topk_fp8(self.sel, self.q, self.kmin, self.kmax, self.bt,
                                                 self.ctx, w.BS, workspace=self.sel_ws),
                lambda: pg.quest_sparse_decode_fp8(self.out_sparse, self.q, self.kc, self.vc,
                                                   self.k_scale, self.v_scale, self.bt, self.ctx,
                                                   self.sel, w.scale, workspace=self.ws_sparse),
                self.quest(),
                None,
                None,
            ]
        if self.kv == "fp8_block":
            return [
                lambda: pg.quest_reshape_and_cache_fp8_block(self.key, self.value, self.kc, self.vc, self.kmin,
                                                             self.kmax, self.slots, self.k_scale, self.v_scale),
                lambda: pg.pa_decode_fp8_block(self.out, self.q, self.kc, self.vc, self.k_scale, self.v_scale,
                                               self.bt, self.ctx, w.scale, workspace=self.ws),
                lambda: pg.quest_select_topk_fp8_block(self.sel, self.q, self.kmin, self.kmax, self.k_scale,
                                                       self.bt, self.ctx, w.BS, workspace=self.sel_ws),
                lambda: pg.quest_sparse_decode_fp8_block(self.out_sparse, self.q, self.kc, self.vc,
                                                         self.k_scale, self.v_scale, self.bt, self.ctx,
                                                         self.sel, w.scale, workspace=self.ws_sparse),
                self.quest(),
                None,
                None,
            ]
        if self.qlen > 1:
            dense = lambda: pg.pa_decode_multi(self.out_multi, self.q_multi, self.kc, self.vc, self.bt,
                                               self.cu_q, self.ctx, w.scale, workspace=self.ws_multi)
            dense_w = quest_w = None
        else:
            dense = lambda: pg.pa_decode(self.out, self.q, self.kc, self.vc, self.bt, self.ctx, w.scale,
                                         workspace=self.ws)
            # the step's write folded into the first launch (the same results)
            dense_w = lambda: pg.pa_reshape_and_decode(self.out, self.q, self.key, self.value, self.slots, self.kc,
                                                       self.vc, self.bt, self.ctx, w.scale, kmin=self.kmin,
                                                       kmax=self.kmax, workspace=self.ws)
            quest_w = lambda: pg.quest_reshape_and_decode(self.out_sparse, self.sel, self.q, self.key, self.value,
                                                          self.slots, self.kmin, self.kmax, self.kc, self.vc,
                                                          self.bt, self.ctx, w.topk, w.scale,
                                                          workspace=self.ws_quest)
        return [
            lambda: pg.quest_reshape_and_cache(self.key, self.value, self.kc, self.vc, self.kmin,
                                               self.kmax, self.slots),
            dense,
            lambda: pg.quest_select_topk(self.sel, self.q, self.kmin, self.kmax, self.bt, self.ctx,
                                         w.BS, workspace=self.sel_ws),
            lambda: pg.quest_sparse_decode(self.out_sparse, self.q, self.kc, self.vc, self.bt,
                                           self.ctx, self.sel, w.scale, workspace=self.ws_sparse),
            self.quest(),
            dense_w,
            quest_w,
        ]


# dense_w / quest_w: the dense and the Quest step with the write folded into
# the first launch (pa_reshape_and_decode, quest_reshape_and_decode; bf16
# cache, one query row); None where that form does not exist
CALL_NAMES = ["write", "dense", "select", "sparse", "quest", "dense_w", "quest_w"]
# Order of the per-call pass: the separate selection and sparse decode (for
# reference), then the fused Quest path and the dense decode back to back
# (the decode launches are one kernel binary, so the second runs on code the
# first left in the SMs' instruction caches).
PASS_B_ORDER = [0, 2, 3, 4, 1, 6, 5]
# The step: write, Quest path (selection 2 launches + sparse decode 1 beside
# the dense decode; quest_decode's 2 with --serial), dense decode
STEP_LAUNCHES = 5
STEP_LAUNCHES_SERIAL = 4


# -------------------------------------------------------------- CPU oracle


class OracleSampler:
    """The oracle on bounded samples of the step. Set-up (not timed): the
    8-bit pool quantised once for --kv fp8, and the Quest metadata of the
    cache as it stands. A sample: the write path for every token (the writes
    and the metadata update are idempotent, so every sample starts from the
    same state), then whole sequences -- dense attention for all heads, Quest
    scores and top-K for all KV heads, sparse attention for all heads -- from
    a rotating cursor until the time budget is spent (at least one)."""

    def __init__(self, w, kv: str = "bf16", qlen: int = 1):
        import oracle
        import workloads
        self.oracle, self.w, self.kv, self.qlen = oracle, w, kv, qlen
        self.cursor = 0
        self.fp8 = kv != "bf16"
        self.block = kv == "fp8_block"
        if self.fp8:
            NB, BS = w.NB, w.BS
            self.kc = np.zeros((NB, BS, w.Hkv, w.D), dtype=np.uint8)
            self.vc = np.zeros((NB, w.Hkv, w.D, BS), dtype=np.uint8)
            pool = (w.key_cache.reshape(NB * BS, w.Hkv, w.D), w.value_cache.reshape(NB * BS, w.Hkv, w.D),
                    self.kc, self.vc, np.arange(NB * BS, dtype=np.int64))
            if self.block:
                self.ks = np.zeros((NB, w.Hkv), dtype=np.float32)
                self.vs = np.zeros_like(self.ks)
                oracle.reshape_and_cache_fp8_block(*pool, self.ks, self.vs)
            else:
                self.ks, self.vs = workloads.fp8_scales(w.Hkv)
                oracle.reshape_and_cache_fp8(*pool, self.ks, self.vs)
            self.kmin, self.kmax = oracle.quest_rebuild_meta_fp8(self.kc, w.block_tables, w.context_lens)
        else:
            self.kc, self.vc = w.key_cache, w.value_cache   # written in place: the state after the step
            self.kmin, self.kmax = oracle.quest_rebuild_meta(self.kc, w.block_tables, w.context_lens)
        if qlen > 1:  # the same query rows the GPU step attends with (Step: seed 1234)
            rng = np.random.default_rng(1234)
            self.qm = workloads.f32_to_bf16_bits(
                rng.standard_normal((w.B * qlen, w.Hq, w.D)).astype(np.float32))
            self.cu = np.arange(0, w.B * qlen + 1, qlen, dtype=np.int32)

    def sample(self, budget_s: float):
        """Returns (algorithmic bytes, seconds, sequences) of one sample."""
        from paged_gqa_decode_reshape_gb300 import ledger
        o, w, eb = self.oracle, self.w, 1 if self.fp8 else 2
        t0 = time.perf_counter()
        if self.block:
            o.reshape_and_cache_fp8_block(w.key, w.value, self.kc, self.vc, w.slot_mapping, self.ks, self.vs,
                                          self.kmin, self.kmax)
        elif self.fp8:
            o.reshape_and_cache_fp8(w.key, w.value, self.kc, self.vc, w.slot_mapping, self.ks, self.vs)
            o.quest_update_meta_fp8(self.kmin, self.kmax, w.key, w.slot_mapping, self.ks, w.BS)
        else:
            o.reshape_and_cache(w.key, w.value, self.kc, self.vc, w.slot_mapping)
            o.quest_update_meta(self.kmin, self.kmax, w.key, w.slot_mapping, w.BS)
        nbytes = ledger.step_bytes(w.context_lens, w.slot_mapping, w.Hq, w.Hkv, w.D, w.BS, w.topk,
                                   elem_bytes=eb, block_scales=self.block)
        done_bytes = nbytes.reshape + nbytes.meta
        seqs = 0
        while seqs < w.B and (seqs == 0 or time.perf_counter() - t0 <= budget_s):
            b = self.cursor
            self.cursor = (self.cursor + 1) % w.B
            rows = np.array([(b, h) for h in range(w.Hq)], dtype=np.int32)
            sl = slice(b, b + 1)
            if self.fp8:
                o.attention_fp8(w.q, self.kc, self.vc, self.ks, self.vs, w.block_tables, w.context_lens,
                                w.scale, rows=rows)
                sc = o.quest_scores_fp8(w.q[sl], self.kmin, self.kmax, w.block_tables[sl],
                                        w.context_lens[sl], w.BS, k_bscale=self.ks if self.block else None)
            else:
                if self.qlen > 1:
                    mrows = np.array([(r, h) for r in range(b * self.qlen, (b + 1) * self.qlen)
                                      for h in range(w.Hq)], dtype=np.int32)
                    o.paged_attention_multi(self.qm, self.kc, self.vc, w.block_tables, self.cu,
                                            w.context_lens, w.scale, rows=mrows)
                else:
                    o.paged_attention(w.q, self.kc, self.vc, w.block_tables, w.context_lens, w.scale,
                                      rows=rows)
                sc = o.quest_scores(w.q[sl], self.kmin, self.kmax, w.block_tables[sl], w.context_lens[sl],
                                    w.BS)
            sel = o.quest_topk(sc, w.context_lens[sl], w.BS, w.topk)
            full_sel = np.full((w.B, w.Hkv, w.topk), -1, dtype=np.int32)
            full_sel[b] = sel[0]
            if self.fp8:
                o.attention_fp8(w.q, self.kc, self.vc, self.ks, self.vs, w.block_tables, w.context_lens,
                                w.scale, selected=full_sel, rows=rows)
            else:
                o.sparse_attention(w.q, self.kc, self.vc, w.block_tables, w.context_lens, full_sel, w.scale,
                                   rows=rows)
            one = ledger.step_bytes(w.context_lens[sl], np.zeros(0, np.int64), w.Hq, w.Hkv, w.D, w.BS,
                                    w.topk, selected=sel, q_rows=self.qlen, elem_bytes=eb,
                                    block_scales=self.block)
            done_bytes += one.dense + one.select + one.sparse
            seqs += 1
        return done_bytes, time.perf_counter() - t0, seqs


# -------------------------------------------------------------------- main


def max_over_ranks(values, pgroup):
    """Element-wise max of per-rank timings (the slowest replica sets the
    job's time); identity on one rank."""
    if pgroup is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    pgroup.all_reduce(t, op=pgroup.ReduceOp.MAX)
    pgroup.barrier()
    return [float(v) for v in t]


def step_runner(torch, step, serial: bool, quest=None, dense=None):
    """One step: the write path, the Quest path and the dense decode. Serial:
    write, quest_decode, dense decode on one stream. Else the Quest path runs
    on a second stream forked after the write path and joined at the end of
    the step: the selection's CTAs run on the SMs beside the dense decode's
    (a decode CTA's warps, at most 184 registers each, leave room in each of
    the SM's register-file partitions), and the sparse decode's CTAs, which
    need a whole SM's shared memory, run on the SMs the dense decode leaves
    free (step.split_ctas()). Neither
    path reads the other's output, and the two decode calls have their own
    workspaces. `quest` and `dense` override the Quest-path and the dense
    call in either mode."""
    c = dict(zip(CALL_NAMES, step.calls()))
    write = c["write"]
    if dense is None:
        dense = c["dense"] if serial else step.dense_beside()
    if serial:
        q = quest or c["quest"]

        def run():
            write()
            q()
            dense()
        return run
    q = quest or step.quest_beside()
    side = torch.cuda.Stream()
    ev_write, ev_quest = torch.cuda.Event(), torch.cuda.Event()

    def run():
        main = torch.cuda.current_stream()
        write()
        ev_write.record(main)
        dense()  # first, so that its persistent grid takes one CTA slot per SM
        side.wait_event(ev_write)
        with torch.cuda.stream(side):
            q()
        ev_quest.record(side)
        main.wait_event(ev_quest)
    return run


def job_throughput(world: int, bytes_per_replica_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every replica moves its step's bytes in the max-over-ranks time."""
    return world * bytes_per_replica_step / (ms_per_step * 1e-3) / 1e9


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pgroup = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pgroup = dist
    return world, rank, local, pgroup


def run_reference(args, world, rank, pgroup):
    import workloads
    if rank != 0:
        return 0
    w0 = workloads.make(args.workload, poison=False)
    cores = 1
    times, nbytes, seq_counts = [], [], []
    sampler = OracleSampler(w0, args.kv, args.qlen)
    for i in range(args.warmup + args.steps):
        # the oracle's writes are idempotent, so every step reuses the same inputs
        b, s, seqs = sampler.sample(args.cpu_budget / max(1, args.steps + args.warmup))
        if i >= args.warmup:
            times.append(s)
            nbytes.append(b)
            seq_counts.append(seqs)
    value = sum(nbytes) / sum(times) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": config_of(w0, args, world),
        "timing": "per step: the oracle on a bounded sample of the step (the write path for every "
                  "token, then whole sequences from a rotating cursor until the step's time share is "
                  "spent); value = sampled algorithmic bytes / sampled CPU seconds",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} steps of a bounded sample of {args.workload}: "
                                   f"{sum(seq_counts)} sequences of {w0.B} in all, "
                                   f"{sum(times):.1f} s of CPU time"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_of(w, args, world: int) -> dict:
    """The workload a line measures (the same for the native and the reference arm)."""
    fp8 = args.kv != "bf16"
    return {
        "workload": args.workload, "batch": w.B, "num_q_heads": w.Hq, "num_kv_heads": w.Hkv,
        "head_dim": w.D, "block_size": w.BS, "topk_blocks": w.topk, "kv_cache": args.kv,
        "query_rows_per_sequence": args.qlen,
        "context_lens_mean": round(float(w.context_lens.mean()), 1),
        "context_lens_max": int(w.context_lens.max()), "pool_blocks": w.NB,
        "kv_pool_bytes": int(2 * w.key_cache.nbytes // (2 if fp8 else 1)),
        "step": ("quest_reshape_and_cache{0} (ReshapeAndCache + metadata update), then on a second "
                 "stream quest_select_topk{0} + quest_sparse_decode{0}_budget beside pa_decode{0}{1}; {2}; "
                 "--serial: quest_decode{0} then pa_decode{0}").format(
                     "" if args.kv == "bf16" else "_" + args.kv,
                     "_budget" if args.qlen == 1 else "",
                     "the SMs split between the two decode calls by their KV token shares (split_ctas)"
                     if args.qlen == 1 else "the sparse call on at most half the SMs"),
        "l2": "inputs resident; L2 flushed before every timed sample",
        "parallelism": f"replicas x{world}",
    }


def stats_ms(samples) -> dict:
    a = np.asarray(samples, dtype=np.float64)
    return {"median": round(float(np.median(a)), 5), "min": round(float(a.min()), 5),
            "mean": round(float(a.mean()), 5), "samples": int(a.size)}


def measure(torch, pg, w, dev, args, flush, pgroup):
    """Time one workload: pass A (whole steps, one event pair each), pass B
    (one stream, an event between calls), pass C (graph replay) and the end
    to end pass. Every timed sample is preceded by an L2 flush outside its
    events. Returns the raw per-sample times (ms) and the step's byte ledger."""
    from paged_gqa_decode_reshape_gb300 import ledger
    step = Step(w, dev, args.kv, args.qlen)
    calls = [step.calls()[k] for k in PASS_B_ORDER]  # launch order of the per-call pass
    present = [c is not None for c in step.calls()]  # in CALL_NAMES order
    stream = torch.cuda.current_stream(dev)
    run_step = step_runner(torch, step, args.serial)
    K = args.steps

    def head_start():
        if not args.no_head_start:
            torch.cuda._sleep(HEAD_START_CYCLES)

    for _ in range(max(3, args.warmup)):
        run_step()
    torch.cuda.synchronize(dev)
    sel_host = step.sel.cpu().numpy()
    fp8 = args.kv != "bf16"
    nb = ledger.step_bytes(w.context_lens, w.slot_mapping, w.Hq, w.Hkv, w.D, w.BS, w.topk,
                           selected=sel_host, elem_bytes=1 if fp8 else 2, q_rows=args.qlen,
                           block_scales=args.kv == "fp8_block")

    # Pass A (the timed region): whole steps, one event pair per step.
    # Kernels launch with programmatic stream serialization, so consecutive
    # launches overlap their start-up with the previous kernel's tail; the
    # Quest selection and sparse decode run beside the dense decode on a
    # second stream (step_runner).
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(gpu_id_for(torch, dev))
    if pgroup:
        pgroup.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        head_start()
        ev[i][0].record(stream)
        run_step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]

    # Pass B: the same steps on one stream with an event between consecutive
    # calls, for the per-call breakdown and the decode kernels' rooflines
    # (the extra events keep each call's launch gap inside its own interval).
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        head_start()
        evb[i][0].record(stream)
        for j, c in enumerate(calls):
            if c is not None:
                c()
            evb[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    per_call = np.array([[evb[i][j].elapsed_time(evb[i][j + 1]) for j in range(len(calls))]
                         for i in range(K)])              # ms, launch order
    per_call = per_call[:, np.argsort(PASS_B_ORDER)]     # ms, in CALL_NAMES order

    # Pass C: the step captured once in a CUDA graph and replayed.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_step()
    torch.cuda.synchronize(dev)
    for _ in range(3):
        graph.replay()
    evc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        head_start()
        evc[i][0].record(stream)
        graph.replay()
        evc[i][1].record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = [e0.elapsed_time(e1) for e0, e1 in evc]

    # end to end through the C ABI with host buffers: H2D of the step's inputs
    # (q, new K/V rows, slots, block tables, context lengths: one pinned
    # buffer) and D2H of its results (dense and sparse outputs, selection),
    # every step
    h_in = step.in_buf.cpu().pin_memory()
    h_out = torch.empty_like(step.out_buf, device="cpu").pin_memory()
    e2e_ms = []
    for i in range(K):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step.in_buf.copy_(h_in, non_blocking=True)
        run_step()
        h_out.copy_(step.out_buf, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    split, sms = (step.split_ctas() if not args.serial else 0), step.sms
    del graph, step
    torch.cuda.synchronize(dev)
    return dict(nb=nb, step_ms=step_ms, per_call=per_call, present=present, graph_ms=graph_ms, e2e_ms=e2e_ms,
                split=split, sms=sms,
                h2d=int(h_in.numel()), d2h=int(h_out.numel()), clocks=clocks, wall=wall)


def call_summary(m, peak: float) -> dict:
    """Per-call medians of pass B, their GB/s on the algorithmic bytes, and
    the fraction of the measured copy peak and of the nominal ~8 TB/s."""
    nb = m["nb"]
    wb = nb.reshape + nb.meta
    call_bytes = [wb, nb.dense, nb.select, nb.sparse, nb.select + nb.sparse, wb + nb.dense,
                  wb + nb.select + nb.sparse]
    med = np.median(m["per_call"], axis=0)
    out = {}
    for n, ms, b, here in zip(CALL_NAMES, med, call_bytes, m["present"]):
        if not here:
            continue
        gbs = b / (ms * 1e-3) / 1e9
        out[n] = {"us": round(float(ms) * 1e3, 2), "us_min": round(float(m["per_call"][:, CALL_NAMES.index(n)].min())
                                                                  * 1e3, 2),
                  "GBps": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 3),
                  "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 3), "bytes": int(b)}
    return out


def point_summary(m, peak: float, world: int) -> dict:
    """The metric's "µs/step dense vs Quest" at one context length: per-call
    medians (pass B), the dense step (write + dense decode) and the Quest step
    (write + quest_decode; and write + selection + sparse decode, unfused),
    and the whole step of pass A."""
    calls = call_summary(m, peak)
    dense_sep = calls["write"]["us"] + calls["dense"]["us"]
    quest_sep = calls["write"]["us"] + calls["quest"]["us"]
    dense_us = calls["dense_w"]["us"] if "dense_w" in calls else dense_sep
    quest_us = calls["quest_w"]["us"] if "quest_w" in calls else quest_sep
    return {
        "dense_step_us": round(dense_us, 2), "quest_step_us": round(quest_us, 2),
        "dense_step_separate_write_us": round(dense_sep, 2), "quest_step_separate_write_us": round(quest_sep, 2),
        "quest_step_unfused_us": round(calls["write"]["us"] + calls["select"]["us"] + calls["sparse"]["us"], 2),
        "dense_decode": calls["dense"], "quest_decode": calls["quest"], "sparse_decode": calls["sparse"],
        **{k: calls[k] for k in ("dense_w", "quest_w") if k in calls},
        "select": calls["select"], "write": calls["write"],
        "whole_step_us": stats_ms(np.asarray(m["step_ms"]) * 1e3),
        "whole_step_GBps": round(job_throughput(world, m["nb"].total, float(np.median(m["step_ms"]))), 1),
    }


def main():
    args = parse()
    world, rank, local, pgroup = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank, pgroup)

    import torch
    import paged_gqa_decode_reshape_gb300 as pg
    import paged_gqa_decode_reshape_gb300.build as pgb
    import workloads

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the native path has no CPU fallback)")
    pgb.build()
    pg.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.make(args.workload, poison=False)
    if args.qlen > 1 and (args.kv != "bf16" or w.B * args.qlen > 2048):
        raise SystemExit("--qlen > 1: bf16 cache and at most 2048 query rows")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    K = args.steps
    fp8 = args.kv != "bf16"
    sfx = "" if args.kv == "bf16" else "_" + args.kv
    peak, peak_kind = measured_peaks()

    m = measure(torch, pg, w, dev, args, flush, pgroup)
    # the metric's second context length, from the same run (one replica)
    m40 = None
    if args.workload == "quest_8k" and args.qlen == 1 and not args.no_long_point:
        m40 = measure(torch, pg, workloads.make("long_40k", poison=False), dev, args, flush, pgroup)

    mine = [float(np.median(m["step_ms"])), float(np.median(m["e2e_ms"])), float(np.median(m["graph_ms"]))]
    ms, e2e_ms_max, graph_ms_max = max_over_ranks(mine, pgroup)
    if rank != 0:
        return 0

    nb = m["nb"]
    value = job_throughput(world, nb.total, ms)
    point = point_summary(m, peak, world)
    dense = point["dense_decode"]
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 KV cache (per-block scales), bf16 q/out" if args.kv == "fp8_block" else
                  "e4m3 KV cache, bf16 q/out" if fp8 else "bf16"),
        "data": "synthetic",
        "config": config_of(w, args, world),
        "timing": ("value/ms_per_step: median over the timed steps of one event pair per step" +
                   ("" if args.serial else ", the Quest selection and sparse decode on a second stream "
                    "beside the dense decode") +
                   "; breakdown/roofline: medians of a second pass of the same steps on one stream with "
                   "an event between calls; L2 flushed before every timed sample "
                   f"({L2_FLUSH_BYTES >> 20} MiB write), outside the events" +
                   ("" if args.no_head_start else
                    f", then a {HEAD_START_CYCLES}-cycle spin kernel so the host has enqueued the step "
                    "before the GPU reaches it (device-timed passes; the e2e pass has none)")),
        "step_ms_stats": stats_ms(m["step_ms"]),
        "roofline": {
            "bound": "hbm",
            "kernel": ("pa_decode" + sfx if fp8 else "pa_decode_multi" if args.qlen > 1 else "pa_decode")
                      + " (split-KV decode + fused combine, 1 launch)",
            "achieved": dense["GBps"], "peak": peak, "unit": "GB/s",
            "frac": round(dense["GBps"] / peak, 4), "peak_kind": peak_kind,
            "frac_of_nominal_8tbs": round(dense["GBps"] / NOMINAL_HBM_GBS, 4),
            "traffic": (recorded_traffic("pa_decode" + sfx, args.workload) if args.qlen == 1 else None),
            "algorithmic_bytes_per_launch": int(nb.dense),
            "launch_us": {"median": dense["us"], "min": dense["us_min"]},
        },
        "roofline_sparse": {
            "bound": "hbm", "kernel": "quest_sparse_decode" + sfx,
            "achieved": point["sparse_decode"]["GBps"], "peak": peak, "unit": "GB/s",
            "frac": point["sparse_decode"]["frac_of_measured_peak"],
            "frac_of_nominal_8tbs": point["sparse_decode"]["frac_of_nominal_8tbs"],
            "algorithmic_bytes_per_launch": point["sparse_decode"]["bytes"],
        },
        "breakdown": {n: point[k] for n, k in (("write", "write"), ("dense", "dense_decode"),
                                               ("select", "select"), ("sparse", "sparse_decode"),
                                               ("quest", "quest_decode"), ("dense_w", "dense_w"),
                                               ("quest_w", "quest_w")) if k in point},
        "breakdown_steps": K,
        "dense_us_per_step": point["dense_step_us"],
        "quest_us_per_step": point["quest_step_us"],
        "quest_us_per_step_unfused": point["quest_step_unfused_us"],
        "dense_step": ("pa_reshape_and_decode (write folded into the decode launch, 1 launch)"
                       if "dense_w" in point else "write + pa_decode"),
        "quest_step": ("quest_reshape_and_decode (write folded into the score launch; then top-K and "
                       "sparse decode in one launch: 2 launches)" if "quest_w" in point else
                       "write + quest_decode (scores; then top-K and sparse decode in one launch)"),
        "dense_step_separate_write_us": point["dense_step_separate_write_us"],
        "quest_step_separate_write_us": point["quest_step_separate_write_us"],
        "quest_step_unfused": "write + quest_select_topk + quest_sparse_decode",
        "tokens_per_s": {"dense": round(world * w.B / (point["dense_step_us"] * 1e-6), 1),
                         "quest": round(world * w.B / (point["quest_step_us"] * 1e-6), 1)},
        "e2e": {"value": round(job_throughput(world, nb.total, e2e_ms_max), 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms_max, 5), "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"], "ms_stats": stats_ms(m["e2e_ms"])},
        "graph": {"value": round(job_throughput(world, nb.total, graph_ms_max), 2), "unit": UNIT,
                  "ms_per_step": round(graph_ms_max, 5), "ms_stats": stats_ms(m["graph_ms"]),
                  "how": "the step's calls captured once in a CUDA graph, replayed K times"},
        "two_stream_split": ({"sparse_ctas": m["split"], "dense_ctas": m["sms"] - m["split"]} if m["split"]
                             else None),
        "gpu_launches": int(K * (STEP_LAUNCHES_SERIAL if args.serial else STEP_LAUNCHES)),
        "wall_s_timed_region": round(m["wall"], 4),
        "clocks": m["clocks"],
    }
    if m40 is not None:
        line["context_points"] = {
            "8K": dict(workload=args.workload, **point),
            "40K": dict(workload="long_40k", **point_summary(m40, peak, world), clocks=m40["clocks"]),
        }
    if world == 1 and not args.no_cpu_baseline:
        b, s, seqs = OracleSampler(workloads.make(args.workload, poison=False), args.kv,
                                   args.qlen).sample(args.cpu_budget)
        line["cpu_baseline"] = {
            "value": round(b / s / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"write path for all {w.T} tokens + {seqs} of {w.B} sequences "
                      f"(dense, Quest select, sparse; all heads), {s:.1f} s of CPU time"}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
