"""Benchmark of the indexer hot path on GB300.

Default workload (the causal prefill indexer, the largest single-GPU
configuration): 4096 queries at positions 61440..65535 over 65536 shared bf16
index keys, H=64 heads, D=128, exact top-K=2048.  One step = score every
visible key (idx_score, 260 M (query, key) pairs) -> exact top-K
(idx_topk_scores).  The same line carries, as a nested `dosa` object, the
DoSA-pruned top-K (dosa_topk, 12288 cold-rule seeds, 16 retained heads) on
the same inputs: its step time, its speed-up over the unpruned step, its
candidate and survival rates, how many rows stayed pruned, and whether its
output equals the unpruned one bit for bit; `dosa_aligned` does the same on
the near-parallel-heads prefill, where the bound prunes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill|decode|ragged_fp8|prefill_dosa|prefill_dosa_aligned|
                              ragged_fp8_dosa|decode_prior|ragged_fp8_prior|block_select|tiny]

Prints ONE JSON line (rank 0).  `value` is queries*keys scored per second over
the whole job (inputs resident in HBM); `e2e` is the same metric through the
C ABI (idx_topk) with the inputs copied from pinned host memory and the top-K
ids copied back inside the timed region.  `roofline` is for the dominant
kernel, timed with CUDA events on its own stream inside the timed region.
`cpu_baseline` times the CPU oracle on a bounded sample of the same workload
on this host's cores (a process pool over every core this process may run
on, and one core).  `witness_vs_memcpy` times witness_merge against a
device-to-device copy of the same [rows, 2048] int32 buffer.
--impl reference times the oracle alone (the reference arm of this build).
Multi-GPU (torchrun): every rank runs its own independent batch (weak
scaling, no data-path collective); the time is the max over ranks.
"""
from __future__ import annotations

import os

# every CPU oracle process runs its BLAS on one thread, so a pool of N
# processes uses exactly N cores
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import multiprocessing as mp
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_attention_indexer_idx_gb300 import workloads as wl  # noqa: E402
from sparse_attention_indexer_idx_gb300.dist import job_step_ms, job_value, rank_seed  # noqa: E402

METRIC = "indexer queries*keys scored/sec"
# prefill queries: the heads of a query share one direction, q = |a| c_z + 0.05 eps
PREFILL_Q_NOISE = 0.05
UNIT = "pairs/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="idx_clocks_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        hi = max(sm)
        under = [x for x in sm if x >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(under), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- workloads --

def make_workload(name: str, rank: int, rows=None):
    """The workload's inputs; `rows` shrinks the batch (query rows) for profiling runs."""
    seed_shift = rank_seed(0, rank)
    kw = {}
    if name == "decode":
        if rows:
            kw["M"] = rows
        return wl.decode_bf16(seed=2 + seed_shift, **kw)
    if name in ("prefill", "prefill_dosa"):
        if rows:
            kw["n_queries"] = rows
        return wl.prefill_bf16(seed=3 + seed_shift, q_noise=PREFILL_Q_NOISE, **kw)
    if name == "prefill_dosa_aligned":
        if rows:
            kw["n_queries"] = rows
        return wl.prefill_bf16(seed=3 + seed_shift, q_noise=0.001, q_run=16, positive_w=True, **kw)
    if name == "decode_prior":
        if rows:
            kw["M"] = rows
        return wl.decode_bf16(seed=2 + seed_shift, **kw)
    if name in ("ragged_fp8", "ragged_fp8_dosa", "ragged_fp8_prior"):
        if rows:
            kw["M"] = rows
        return wl.ragged_fp8(seed=5 + seed_shift, **kw)
    if name == "tiny":
        return wl.tiny_fp32(seed=0 + seed_shift)
    if name == "block_select":
        if rows:
            kw["Q"] = rows
            kw["L"] = 128 * rows
        return wl.block_select(seed=4 + seed_shift, **kw)
    raise ValueError(name)


# workloads whose inputs exceed the 129 MB L2 (no flush between timed steps)
LARGE_INPUTS = ("decode", "ragged_fp8", "decode_prior", "ragged_fp8_prior")

# dram__bytes_read.sum + dram__bytes_write.sum of the score kernel per full launch: one ncu
# capture (a single pass) of the full-size workload, the kernel as built with this file
# (profiles/dram_traffic_full_size.md).  None where not captured.
SCORE_TRAFFIC = {"decode": 547.86e6, "ragged_fp8": 1158.60e6, "prefill": 1084.21e6}
# the same counters for one bt_max_kernel launch on the full block_select workload (the
# fp16 keys, 33.5 MB, dominate)
BLOCK_MAX_TRAFFIC = 37.66e6

WORKLOAD_TEXT = {
    "decode": "decode indexer bf16: 64 rows x 32768 own keys, H32 D128, top-2048, witness_merge S=16 (5% padding)",
    "prefill": "causal prefill bf16: 4096 queries over 65536 shared keys, H64 D128, top-2048 (unpruned)",
    "prefill_dosa": "causal prefill bf16 with DoSA pruning: 4096 queries, 65536 keys, H64 D128, K2048, 12288 seeds, R16",
    "prefill_dosa_aligned": "causal prefill bf16 with DoSA pruning, near-parallel heads: 4096 queries, 65536 keys, "
                            "H64 D128, K2048, 12288 seeds, R16; q_h = |a_h| c_z + 0.001 N(0,1), runs of 16 "
                            "queries share z, w = |N(0, 1/64)|",
    "ragged_fp8_dosa": "ragged decode FP8 with DoSA pruning: 128 rows, L_r~U[4096,131072], H64 D128, K2048, 8192 seeds/row, R20",
    "ragged_fp8": "ragged decode FP8 e4m3 keys + scale: 128 rows, L_r~U[4096,131072], H64 D128, top-2048, witness_merge S=32",
    "tiny": "tiny fp32 indexer: 8 rows, H4 D16, L512, K32, witness_merge S=4",
    "decode_prior": "decode indexer bf16 (as decode) ranked with a prior: the top-2048 of the two previous steps "
                    "(queries q + 0.3 N(0,1), one key fewer)",
    "ragged_fp8_prior": "ragged decode FP8 (as ragged_fp8) ranked with a prior: the top-2048 of the two previous "
                        "steps (queries q + 0.3 N(0,1), one key fewer)",
    "block_select": "MiniMax block select fp32: 1024 queries, 8 KV heads, D128, L131072, block 128, top 32, init 1, local 2",
}


# ---------------------------------------------------------------- our arm ----

class IndexerStep:
    """score -> top-K -> padding -> witness merge on device-resident inputs."""

    def __init__(self, B, wp, dev):
        self.B = B
        self.wp = wp
        self.dev = dev
        self.p = B.problem_to_device(wp, dev)
        self.K = wp.K
        self.ld = self.p.max_key_len
        self.scores = torch.empty((wp.M, self.ld), dtype=torch.float32, device=dev)
        self.tk_ws = torch.empty(max(1, B.idx_topk_scores_workspace_size(wp.M, self.ld, wp.K)), dtype=torch.uint8,
                                 device=dev)
        self.ids = torch.empty((wp.M, self.K), dtype=torch.int32, device=dev)
        self.S = wp.extras.get("S", 0)
        pm = wp.extras.get("pad_mask")
        self.pad = None if pm is None else torch.from_numpy(pm).to(dev)
        self.ctx = self.p.key_len
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        self.score_ms = []
        # score + top-K (filter and finish kernels) + witness merge
        self.launches = 1 + 2 + (1 if self.S else 0)

    def run(self, timed=False):
        """score -> top-K [-> padding -> witness merge].  The padding (5% of the
        learned slots set to -1, a torch op standing in for the learned
        selection's padding) lies between events 2 and 3, outside the step."""
        B, p = self.B, self.p
        if timed:
            self.ev[0].record()
        B.idx_score(p, self.scores, self.ld)
        if timed:
            self.ev[1].record()
        B.idx_topk_scores(self.scores, p.key_len, self.ld, self.K, self.ids, None, ld=self.ld, ws=self.tk_ws)
        if timed:
            self.ev[2].record()
        if self.S:
            if self.pad is not None:
                self.ids.masked_fill_(self.pad, -1)
            if timed:
                self.ev[3].record()
            B.witness_merge(self.ids, self.ctx, max(self.K - self.S, 0), self.S, self.S)
            if timed:
                self.ev[4].record()

    def collect(self):
        self.score_ms.append(self.ev[0].elapsed_time(self.ev[1]))

    def step_ms(self):
        ms = self.ev[0].elapsed_time(self.ev[2])
        if self.S:
            ms += self.ev[3].elapsed_time(self.ev[4])
        return ms

    def algorithmic_bytes(self):
        """Score kernel: every visible key row once, queries, weights, one fp32 score per pair."""
        wp = self.wp
        kb = {"bf16": 2, "f32": 4, "fp8": 1}[wp.dtype] * wp.D
        if wp.dtype == "fp8":
            kb += 4
        pairs = wp.pairs()
        if wp.key_off is None:
            key_bytes = int(np.max(wp.key_len)) * kb
        else:
            key_bytes = pairs * kb
        qb = wp.M * wp.H * wp.D * (4 if wp.dtype == "f32" else 2) + wp.M * wp.H * 4
        return key_bytes + qb + pairs * 4

    def flops(self):
        return 2.0 * self.wp.pairs() * self.wp.H * self.wp.D


class DosaStep:
    """DoSA-pruned top-K (dosa_topk) on device-resident inputs."""

    def __init__(self, B, wp, dev, R, n_seed, capacity=16384, group_stream=1):
        self.B = B
        self.wp = wp
        self.p = B.problem_to_device(wp, dev)
        self.K = wp.K
        self.dp = B.make_dosa_params(n_seed=n_seed, retained_heads=R, candidate_capacity=capacity,
                                     group_stream=group_stream)
        self.ids = torch.empty((wp.M, self.K), dtype=torch.int32, device=dev)
        self.sc = torch.empty((wp.M, self.K), dtype=torch.float32, device=dev)
        self.ws = torch.empty(B.dosa_topk_workspace_size(self.p, self.K, self.dp), dtype=torch.uint8, device=dev)
        self.stats = torch.zeros(B.DOSA_STATS_FIELDS, dtype=torch.int64, device=dev)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        self.score_ms = []
        # kernels dosa_topk enqueues per call: seeds, seed scores and top-K, planner,
        # bound scan, rescoring, merge, fallback and statistics (every top-K stage is
        # a filter and a finish kernel)
        two = lambda n: 2
        L = int(np.max(wp.key_len))
        NS = min(max(n_seed, wp.K), L)
        if wp.key_off is None:
            # + the group split and the shared-stream scoring (groups of four queries)
            grp = 2 if group_stream and wp.M >= 2 and wp.q.shape[1] in (16, 32, 64) else 0
            self.launches = 20 + grp + two(L) + two(NS) + two(wp.K + capacity) + two(L)
        else:
            self.launches = 13 + two(NS) + two(wp.K + capacity) + two(L)

    def run(self, timed=False):
        if timed:
            self.ev[0].record()
        self.B.dosa_topk(self.p, self.K, self.dp, self.ids, self.sc, self.ws, stats=self.stats)
        if timed:
            self.ev[1].record()

    def collect(self):
        self.score_ms.append(self.ev[0].elapsed_time(self.ev[1]))

    def step_ms(self):
        return self.ev[0].elapsed_time(self.ev[1])

    def info(self, stream, ref_ids=None, ref_sc=None):
        """One more call with fresh counters: candidate / survival rates, rows that
        stayed pruned, and (given the unpruned output) bit identity with it."""
        self.stats.zero_()
        rs = torch.full((self.wp.M,), -1, dtype=torch.int32, device=self.ids.device)
        with torch.cuda.stream(stream):
            self.B.dosa_topk(self.p, self.K, self.dp, self.ids, self.sc, self.ws, stats=self.stats, row_status=rs)
        torch.cuda.synchronize()
        st = self.stats.cpu().tolist()
        rs = rs.cpu().numpy()
        # rates over the non-seed pairs of the rows that ran the bound scan (row_status 0,
        # or 2: candidates over capacity), the seed pairs taken as evenly spread over the rows
        scanned = (rs == 0) | (rs == 2)
        lens = np.asarray(self.wp.key_len, dtype=np.int64)
        nonseed = float(lens[scanned].sum()) - float(st[1]) * float(scanned.sum()) / max(1, self.wp.M)
        rate = (lambda x: x / nonseed) if nonseed > 0 else (lambda x: None)
        out = {"pairs": st[0], "seed_pairs": st[1], "candidates": st[2], "survivors": st[3],
               "fallback_rows": st[4], "skipped_rows": st[5], "group_keys": st[6], "solo_keys": st[7],
               "group_stream": int(self.dp.group_stream),
               "rows_pruned": int((rs == 0).sum()), "rows": int(self.wp.M),
               "candidate_rate": rate(st[2]), "survival_rate": rate(st[3]),
               "rates_over": "non-seed pairs of the rows that ran the bound scan"}
        if ref_ids is not None:
            out["identical_to_unpruned"] = bool(torch.equal(self.ids, ref_ids) and
                                               torch.equal(self.sc.view(torch.int32), ref_sc.view(torch.int32)))
        return out


class BlockSelectStep:
    def __init__(self, B, bp, dev):
        self.B = B
        self.bp = bp
        self.q = torch.from_numpy(bp.index_q).to(dev)
        self.k = torch.from_numpy(bp.index_k).to(dev)
        self.pos = torch.from_numpy(bp.query_pos).to(dev)
        self.cfg = B.block_sparse_config(bp.block_size, bp.top_blocks, bp.init_blocks, bp.local_blocks)
        Q, n_kv, _ = bp.index_q.shape
        self.out = torch.empty((Q, n_kv, max(bp.top_blocks, bp.init_blocks + bp.local_blocks)), dtype=torch.int32,
                               device=dev)
        self.cnt = torch.empty((Q, n_kv), dtype=torch.int32, device=dev)
        self.ws = torch.empty(B.block_select_workspace_size(Q, n_kv, bp.index_k.shape[0], self.cfg),
                              dtype=torch.uint8, device=dev)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        self.score_ms = []          # the block-maxima kernel (bt_max_kernel)
        self.phase_ms = {k: [] for k in self.PHASES}
        self.launches = 5           # prep, block maxima, classify, rescoring, resolve

    PHASES = ("prep", "block_max", "classify", "rescore", "resolve")

    def run(self, timed=False):
        if timed:
            # events between the kernels, recorded by the library on the current stream
            self.B.block_select_events(self.q, self.k, self.pos, self.cfg, self.out, self.cnt, self.ws, self.ev,
                                       stream=torch.cuda.current_stream())
        else:
            self.B.block_select(self.q, self.k, self.pos, self.cfg, self.out, self.cnt, self.ws)

    def collect(self):
        for i, k in enumerate(self.PHASES):
            self.phase_ms[k].append(self.ev[i].elapsed_time(self.ev[i + 1]))
        self.score_ms.append(self.phase_ms["block_max"][-1])

    def step_ms(self):
        return self.ev[0].elapsed_time(self.ev[5])

    def bound_stats(self):
        st = self.B.block_select_stats_tensor()
        self.B.block_select(self.q, self.k, self.pos, self.cfg, self.out, self.cnt, self.ws, stats=st)
        torch.cuda.synchronize()
        return self.B.block_select_stats_read(st)

    def pairs(self):
        bs = self.bp.block_size
        L = self.bp.index_k.shape[0]
        return int(sum(min(int(p) + 1, L) for p in self.bp.query_pos)) * self.bp.index_q.shape[1]


class PriorStep:
    """Top-K with recent selections as a prior (idx_topk_prior) on device-resident inputs.
    The prior (the top-K of the two previous decode steps) is computed once, outside the
    timed region, by the unpruned top-K on the previous steps' queries."""

    PHASES = ("check", "prior_scores", "filter", "candidate_topk", "rest")

    def __init__(self, B, wp, dev, capacity):
        self.B = B
        self.wp = wp
        self.p = B.problem_to_device(wp, dev)
        self.K = K = wp.K
        M = wp.M
        priors = []
        for seed in (8, 9):
            prev = wl.previous_step(wp, seed=seed, noise=0.3)
            q = torch.from_numpy(np.ascontiguousarray(prev.q).view(np.int16)).to(dev).view(torch.bfloat16)
            pq = B.Problem(q, self.p.w, self.p.keys, torch.from_numpy(prev.key_len).to(dev), self.p.max_key_len,
                           self.p.key_off, self.p.key_scale)
            ids = torch.empty((M, K), dtype=torch.int32, device=dev)
            B.idx_topk(pq, K, ids, None, torch.empty(B.idx_topk_workspace_size(pq, K), dtype=torch.uint8, device=dev))
            priors.append(ids)
        self.prior = torch.cat(priors, dim=1).contiguous()
        self.cap = 4 * K
        self.ids = torch.empty((M, K), dtype=torch.int32, device=dev)
        self.sc = torch.empty((M, K), dtype=torch.float32, device=dev)
        self.ws = torch.empty(B.idx_topk_prior_workspace_size(self.p, K, self.prior.shape[1], self.cap),
                              dtype=torch.uint8, device=dev)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        self.score_ms = []          # the filtered score kernel
        self.phase_ms = {k: [] for k in self.PHASES}
        # check, prior scores, tau, filtered scores, route, candidate top-K (2), unpruned rows'
        # score and top-K (3, masked), counters
        self.launches = 11
        torch.cuda.synchronize()

    def run(self, timed=False):
        if timed:
            self.B.idx_topk_prior_events(self.p, self.K, self.prior, self.cap, self.ids, self.sc, self.ws, self.ev,
                                         stream=torch.cuda.current_stream())
        else:
            self.B.idx_topk_prior(self.p, self.K, self.prior, self.cap, self.ids, self.sc, self.ws)

    def collect(self):
        for i, k in enumerate(self.PHASES):
            self.phase_ms[k].append(self.ev[i].elapsed_time(self.ev[i + 1]))
        self.score_ms.append(self.phase_ms["filter"][-1])

    def step_ms(self):
        return self.ev[0].elapsed_time(self.ev[5])

    def algorithmic_bytes(self):
        """Filtered score kernel: every visible key row once, queries, weights (the candidates it
        writes are ~1% of that)."""
        wp = self.wp
        kb = {"bf16": 2, "fp8": 1}[wp.dtype] * wp.D + (4 if wp.dtype == "fp8" else 0)
        return wp.pairs() * kb + wp.M * wp.H * wp.D * 2 + wp.M * wp.H * 4

    def prior_stats(self):
        st = torch.zeros(3, dtype=torch.int64, device=self.ids.device)
        rs = torch.empty((self.wp.M,), dtype=torch.int32, device=self.ids.device)
        self.B.idx_topk_prior(self.p, self.K, self.prior, self.cap, self.ids, self.sc, self.ws, row_status=rs,
                              stats=st)
        torch.cuda.synchronize()
        s = st.cpu().tolist()
        return {"rows_filtered": s[0], "candidates_per_row": s[1] / max(1, s[0]), "dense_rows": s[2]}


def e2e_run(B, wp, dev, steps):
    """Same step through the C ABI from pinned host buffers: H2D of the step's
    inputs, score -> top-K -> witness merge, D2H of the top-K ids."""
    host = {}
    p_dev = B.problem_to_device(wp, dev)
    tens = {"q": p_dev.q, "w": p_dev.w, "keys": p_dev.keys, "key_len": p_dev.key_len}
    if p_dev.key_off is not None:
        tens["key_off"] = p_dev.key_off
    if p_dev.key_scale is not None:
        tens["key_scale"] = p_dev.key_scale
    for k, t in tens.items():
        host[k] = t.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    ids = torch.empty((wp.M, wp.K), dtype=torch.int32, device=dev)
    ids_host = torch.empty((wp.M, wp.K), dtype=torch.int32).pin_memory()
    d2h = ids_host.numel() * 4
    ws = torch.empty(B.idx_topk_workspace_size(p_dev, wp.K), dtype=torch.uint8, device=dev)
    S = wp.extras.get("S", 0)

    def one():
        for k, t in tens.items():
            t.copy_(host[k], non_blocking=True)
        B.idx_topk(p_dev, wp.K, ids, None, ws)
        if S:
            B.witness_merge(ids, p_dev.key_len, max(wp.K - S, 0), S, S)
        ids_host.copy_(ids, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


# ------------------------------------------------------------- CPU baseline --
# The oracle as it stands, run by a pool of worker processes (spawned, so that
# no worker inherits a CUDA context), one core each.  A worker holds a
# sub-problem with only the sampled rows (and the keys they read).

_ORACLE = None


def _oracle_init(problem):
    global _ORACLE
    _ORACLE = problem


def _oracle_indexer_row(task):
    """Score + exact top-K (+ witness merge) of one row: row `task` of the worker's
    problem, or row 0 of the one-row problem `task` (rows with their own keys)."""
    from oracle import dsa as odsa
    from oracle import witness as ow
    wp, m = (_ORACLE, task) if isinstance(task, int) else (task, 0)
    ids, _, _, _ = odsa.row_topk(wp, m, wp.K)
    S = wp.extras.get("S", 0)
    if S:
        ow.apply_topology_witnesses(ids, wp.K, [int(wp.key_len[m])], max(wp.K - S, 0), S, S)
    return int(wp.key_len[m])


def _oracle_block_query(i):
    """MiniMax selection of query i (all KV heads) of the worker's problem."""
    from oracle import block_select as obs
    bp = _ORACLE
    obs.block_sparse_select(bp.index_q[i], bp.index_k, int(bp.query_pos[i]), bp.block_size, bp.top_blocks,
                            bp.init_blocks, bp.local_blocks)
    return min(int(bp.query_pos[i]) + 1, bp.index_k.shape[0]) * bp.index_q.shape[1]


def _sub_indexer(wp, rows):
    """The rows `rows` of an indexer problem as a problem of their own (row i of it
    is row rows[i]); per-row keys are gathered, shared keys cut to what they see."""
    rows = np.asarray(rows, dtype=np.int64)
    key_len = np.asarray(wp.key_len)[rows].astype(np.int32)
    scale = None
    if wp.key_off is None:
        n = int(key_len.max()) if rows.size else 0
        keys, key_off = wp.keys[:n], None
        if wp.key_scale is not None:
            scale = wp.key_scale[:n]
    else:
        offs = np.asarray(wp.key_off)[rows]
        keys = np.concatenate([wp.keys[o:o + l] for o, l in zip(offs, key_len)])
        if wp.key_scale is not None:
            scale = np.concatenate([wp.key_scale[o:o + l] for o, l in zip(offs, key_len)])
        key_off = np.concatenate([[0], np.cumsum(key_len.astype(np.int64))[:-1]]).astype(np.int64)
    extras = {k: v for k, v in wp.extras.items() if k != "pad_mask"}
    return wl.IndexerProblem(wp.name, wp.dtype, wp.q[rows], wp.w[rows], keys, key_len, key_off, wp.K,
                             key_scale=scale, extras=extras)


def _sub_block(bp, queries):
    queries = np.asarray(queries, dtype=np.int64)
    pos = bp.query_pos[queries]
    n = min(int(pos.max()) + 1, bp.index_k.shape[0])
    return wl.BlockSelectProblem(bp.name, bp.index_q[queries], bp.index_k[:n], pos, bp.block_size, bp.top_blocks,
                                 bp.init_blocks, bp.local_blocks)


class OraclePool:
    """A bounded sample of the workload and the processes that run the oracle on it."""

    def __init__(self, wl_name, wp, cores):
        self.block = wl_name == "block_select"
        if self.block:
            Q = wp.index_q.shape[0]
            self.units = list(range(Q - 1, -1, -max(1, Q // 64)))          # 64 queries spread over [0, L)
            self.sub = _sub_block(wp, self.units)
            self.fn = _oracle_block_query
            self.sample = (f"{len(self.units)} of {Q} queries (all {wp.index_q.shape[1]} KV heads), "
                           "oracle.block_select (the page's sequential f32 dots)")
        else:
            stride = 16 if wp.M >= 1024 else 1                               # the prefill: every 16th query
            self.units = list(range(0, wp.M, stride))
            # shared keys travel to every worker once; rows with their own keys carry them in the task
            self.wp = wp
            self.per_row = wp.key_off is not None
            self.sub = None if self.per_row else _sub_indexer(wp, self.units)
            self.fn = _oracle_indexer_row
            S = wp.extras.get("S", 0)
            self.sample = (f"{'every 16th' if stride > 1 else 'every'} row ({len(self.units)} of {wp.M}): score + "
                           f"top-K{' + witness merge' if S else ''}, oracle.dsa fp64")
        self.cores = cores
        self.pool = None
        if cores > 1:
            self.pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_init, initargs=(self.sub,))

    def _tasks(self, idx):
        if not self.block and self.per_row:
            return [_sub_indexer(self.wp, [self.units[i]]) for i in idx]
        return list(idx)

    def run(self, idx):
        """Runs the sample's units `idx`; returns (pairs, seconds)."""
        tasks = self._tasks(idx)
        t0 = time.perf_counter()
        if self.pool is None:
            _oracle_init(self.sub)
            pairs = sum(self.fn(t) for t in tasks)
        else:
            pairs = sum(self.pool.map(self.fn, tasks, chunksize=1))
        return pairs, time.perf_counter() - t0

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool.join()


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl_name, wp, one_core_units=None):
    """The oracle as it stands on the sample, on every core of this host (a process
    pool) and on one core (the first `one_core_units` units of the sample)."""
    n = host_cores()
    pool = OraclePool(wl_name, wp, n)
    try:
        idx = list(range(len(pool.units)))
        pool.run(idx[:n])                       # workers started and warm
        pairs, dt = pool.run(idx)
    finally:
        pool.close()
    one = OraclePool(wl_name, wp, 1)
    k1 = one_core_units or max(1, len(one.units) // 8)
    p1, d1 = one.run(list(range(min(k1, len(one.units)))))
    return {"value": pairs / dt, "unit": UNIT, "cores": n, "kind": "oracle", "sample": pool.sample,
            "seconds": dt,
            "single_core": {"value": p1 / d1, "unit": UNIT, "cores": 1, "seconds": d1,
                            "sample": f"the first {min(k1, len(one.units))} units of the same sample"}}


# ------------------------------------------------------- witness vs memcpy --

def witness_vs_memcpy(B, dev, stream, reps=30):
    """witness_merge (S = 64, topk 2048, keep = topk - S, B = S: the page's
    setting) against a device-to-device copy of the same [rows, 2048] int32
    buffer (cudaMemcpyAsync through torch), each timed by CUDA events on the
    stream, median of `reps`; the merge runs on a fresh copy of the learned
    rows every time (the refresh lies outside its events).  A spin of the GPU
    (torch.cuda._sleep, outside the events) holds the stream while the host
    enqueues both timed calls, so that at a few rows the events measure the
    device time and not the host's submission gap."""
    out = {}
    topk, S = 2048, 64
    for rows in (32, 64, 128, 256, 512, 65536):
        learned, ctx = wl.witness_rows(seed=70 + rows, rows=rows, topk=topk, L_min=topk, L_max=131072)
        with torch.cuda.stream(stream):
            src = torch.from_numpy(learned).to(dev)
            work = torch.empty_like(src)
            dst = torch.empty_like(src)
            c = torch.from_numpy(ctx).to(dev)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            tw, tc = [], []
            for i in range(reps + 3):
                work.copy_(src)
                torch.cuda._sleep(200_000)
                ev[0].record(stream)
                B.witness_merge(work, c, topk - S, S, S, stream=stream)
                ev[1].record(stream)
                ev[2].record(stream)
                dst.copy_(src)
                ev[3].record(stream)
                torch.cuda.synchronize()
                if i >= 3:
                    tw.append(ev[0].elapsed_time(ev[1]))
                    tc.append(ev[2].elapsed_time(ev[3]))
        mw, mc = statistics.median(tw), statistics.median(tc)
        out[str(rows)] = {"witness_us": mw * 1e3, "memcpy_us": mc * 1e3, "ratio": mw / mc}
    return out


# --------------------------------------------------------------------- main --

def _timed_steps(step, stream, steps, flush):
    """`steps` calls of step.run(timed=True) on `stream`, each with its own events
    (created and recorded once before, so none is created in the timed region);
    returns the summed per-step milliseconds and the wall-clock region's."""
    per_step = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    for evs in per_step + [[t_start, t_end]]:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        step.ev = per_step[i]
        step.run(timed=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    total = 0.0
    for i in range(steps):
        step.ev = per_step[i]
        step.collect()
        total += step.step_ms()
    return total, t_start.elapsed_time(t_end)


def dosa_nested(B, wp, dev, stream, steps, warmup, unpruned_ms, ref_ids, ref_sc, flush, capacity, group_stream):
    """The DoSA-pruned top-K on the same inputs as the unpruned step."""
    with torch.cuda.stream(stream):
        d = DosaStep(B, wp, dev, R=wp.extras["R"], n_seed=wp.extras["n_seed"], capacity=capacity,
                     group_stream=group_stream)
        for _ in range(warmup):
            d.run()
        torch.cuda.synchronize()
        total, _ = _timed_steps(d, stream, steps, flush)
    ms = total / steps
    out = {"ms_per_step": ms, "speedup_vs_unpruned": unpruned_ms / ms,
           "pairs_per_s": wp.pairs() / (ms * 1e-3)}
    out.update(d.info(stream, ref_ids, ref_sc))
    return out


def reference_arm(args):
    """The CPU oracle on the machine's host cores, the same workload, metric and unit:
    W warm-up steps and K timed steps, each a bounded part of the sample."""
    wp = make_workload(args.workload, 0)
    n = host_cores()
    pool = OraclePool(args.workload, wp, n)
    units = list(range(len(pool.units)))
    per = max(n, min(len(units), 2 * n))       # units per step
    samples = []
    try:
        for i in range(args.warmup + args.steps):
            lo = (i * per) % len(units)
            idx = (units[lo:] + units[:lo])[:per]
            pairs, dt = pool.run(idx)
            if i >= args.warmup:
                samples.append(pairs / dt)
    finally:
        pool.close()
    v = statistics.median(samples)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "l2": _l2_text(args.workload)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": n, "kind": "oracle",
                             "sample": f"{per} units per step of: {pool.sample}"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _l2_text(name):
    return ("inputs larger than L2 (no flush)" if name in LARGE_INPUTS else
            "L2 flushed before every timed step (256 MB write outside the step's events)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill", choices=list(WORKLOAD_TEXT))
    ap.add_argument("--capacity", type=int, default=16384, help="DoSA candidate capacity per row")
    ap.add_argument("--group-stream", type=int, default=1, choices=[0, 1],
                    help="DoSA shared candidate stream for groups of four queries (shared keys)")
    ap.add_argument("--rows", type=int, default=0, help="smaller batch (query rows) for profiling runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the nested DoSA runs, the witness/memcpy leg and e2e (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # rank 0 alone; the other ranks of a torchrun launch exit at once
        if rank == 0:
            print(json.dumps(reference_arm(args)))
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    # the CPU baseline first: its worker processes are spawned before this
    # process touches the GPU
    wp = make_workload(args.workload, rank, args.rows or None)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.rows:
        cpu = cpu_baseline(args.workload, wp)

    from sparse_attention_indexer_idx_gb300 import binding as B
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B.lib()
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        if args.workload == "block_select":
            step = BlockSelectStep(B, wp, dev)
            pairs_per_step = step.pairs()
            rows_per_step = wp.index_q.shape[0] * wp.index_q.shape[1]
        elif args.workload in ("decode_prior", "ragged_fp8_prior"):
            step = PriorStep(B, wp, dev, args.capacity)
            pairs_per_step = wp.pairs()
            rows_per_step = wp.M
        elif args.workload in ("prefill_dosa", "prefill_dosa_aligned", "ragged_fp8_dosa"):
            step = DosaStep(B, wp, dev, R=wp.extras["R"], n_seed=wp.extras.get("n_seed", wp.extras.get("seed_cap", 8192)),
                            capacity=args.capacity, group_stream=args.group_stream)
            pairs_per_step = wp.pairs()
            rows_per_step = wp.M
        else:
            step = IndexerStep(B, wp, dev)
            pairs_per_step = wp.pairs()
            rows_per_step = wp.M
        for _ in range(args.warmup):
            step.run()
        torch.cuda.synchronize()
        assert B.device_error() == 0, "device error during warm-up"
        # inputs smaller than L2: a 256 MB write before every timed step evicts them; the
        # step is then timed by its own events, which the flush lies outside of
        flush = None if args.workload in LARGE_INPUTS else torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        clocks = Clocks(torch.cuda.current_device())
        clocks.start()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ms_total, _ = _timed_steps(step, stream, args.steps, flush)
        clock_info = clocks.stop()
    kernel_ms = step.score_ms
    ms_step = job_step_ms(ms_total / args.steps, device=dev)
    value = job_value(pairs_per_step, ms_step, world)

    hbm, bf16, bf16_sus, peak_src = _peaks()
    roof = None
    extra = {}
    if isinstance(step, IndexerStep):
        k_ms = statistics.median(kernel_ms)
        if wp.dtype in ("bf16", "fp8") and wp.key_off is None:
            ach = step.flops() / (k_ms * 1e-3) / 1e12
            roof = {"kernel": "score_tc_kernel", "bound": "tensor", "achieved": ach, "peak": bf16, "unit": "TFLOP/s",
                    "frac": ach / bf16, "traffic": SCORE_TRAFFIC.get(args.workload) if not args.rows else None,
                    "peak_source": f"{peak_src} bf16 burst", "kernel_ms": k_ms,
                    "algorithmic_flops": step.flops()}
        else:
            ach = step.algorithmic_bytes() / (k_ms * 1e-3) / 1e9
            traffic = SCORE_TRAFFIC.get(args.workload) if not args.rows else None
            roof = {"kernel": "score_tc_kernel" if wp.dtype != "f32" else "score_simt_kernel", "bound": "hbm",
                    "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": traffic,
                    "peak_source": f"{peak_src} hbm copy", "kernel_ms": k_ms,
                    "algorithmic_bytes": step.algorithmic_bytes()}
    elif isinstance(step, PriorStep):
        k_ms = statistics.median(kernel_ms)
        ach = step.algorithmic_bytes() / (k_ms * 1e-3) / 1e9
        roof = {"kernel": "score_tc_kernel (kFilter)", "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "traffic": None, "peak_source": f"{peak_src} hbm copy", "kernel_ms": k_ms,
                "algorithmic_bytes": step.algorithmic_bytes(),
                "phases_ms": {k: statistics.median(v) for k, v in step.phase_ms.items()}}
        with torch.cuda.stream(stream):
            roof["prior_stats"] = step.prior_stats()
    elif isinstance(step, BlockSelectStep):
        k_ms = statistics.median(kernel_ms)
        # the block maxima on the tensor cores: one multiply-add per visible (query, head,
        # position) and dimension (fp16 operands, fp32 accumulate; the fp16 dense rate is
        # the bf16 rate)
        flops = 2.0 * step.pairs() * wp.index_q.shape[2]
        ach = flops / (k_ms * 1e-3) / 1e12
        roof = {"kernel": "bt_max_kernel", "bound": "tensor", "achieved": ach, "peak": bf16, "unit": "TFLOP/s",
                "frac": ach / bf16, "traffic": BLOCK_MAX_TRAFFIC if not args.rows else None,
                "peak_source": f"{peak_src} bf16 burst (fp16 = bf16 rate)", "kernel_ms": k_ms,
                "algorithmic_flops": flops,
                "phases_ms": {k: statistics.median(v) for k, v in step.phase_ms.items()}}
        with torch.cuda.stream(stream):
            roof["bound_stats"] = step.bound_stats()
    else:
        k_ms = statistics.median(kernel_ms)
        roof = {"kernel": "dosa_topk (all kernels)", "bound": "tensor", "achieved": None, "peak": bf16,
                "unit": "TFLOP/s", "frac": None, "traffic": None, "kernel_ms": k_ms}
        extra["dosa"] = step.info(stream)

    e2e = None
    if isinstance(step, IndexerStep) and not args.no_extras:
        with torch.cuda.stream(stream):
            e_ms, h2d, d2h = e2e_run(B, wp, dev, max(3, min(args.steps, 10)))
        e2e = {"value": pairs_per_step * world / (e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms, "api": "idx_topk"}

    if isinstance(step, IndexerStep) and not args.no_extras and rank == 0:
        # the pruned path on the same inputs, and on the near-parallel-heads prefill
        if args.workload == "prefill" and not args.rows:
            ref_ids, ref_sc = _unpruned_topk(B, step, stream)
            extra["dosa"] = dosa_nested(B, wp, dev, stream, args.steps, args.warmup, ms_step, ref_ids, ref_sc,
                                        flush, args.capacity, args.group_stream)
            wa = make_workload("prefill_dosa_aligned", rank)
            sa = IndexerStep(B, wa, dev)
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    sa.run()
                torch.cuda.synchronize()
                ua, _ = _timed_steps(sa, stream, args.steps, flush)
            ra_ids, ra_sc = _unpruned_topk(B, sa, stream)
            extra["dosa_aligned"] = dosa_nested(B, wa, dev, stream, args.steps, args.warmup, ua / args.steps,
                                                ra_ids, ra_sc, flush, args.capacity, args.group_stream)
            extra["dosa_aligned"]["unpruned_ms_per_step"] = ua / args.steps
            extra["dosa_aligned"]["workload"] = WORKLOAD_TEXT["prefill_dosa_aligned"]
            del sa, wa
        extra["witness_vs_memcpy"] = witness_vs_memcpy(B, dev, stream)

    assert B.device_error() == 0, "device error during the timed region"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": {"f32": "f32", "bf16": "bf16", "fp8": "fp8e4m3"}.get(
                getattr(wp, "dtype", "f32"), "f32"),
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "l2": _l2_text(args.workload)},
            "rows_per_s": rows_per_step * world / (ms_step * 1e-3),
            "roofline": roof, "e2e": e2e, "clocks": clock_info,
            "gpu_launches": step.launches * args.steps}
    line.update(extra)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def _unpruned_topk(B, step, stream):
    """The unpruned top-K ids and scores of an IndexerStep's inputs (idx_topk)."""
    wp = step.wp
    with torch.cuda.stream(stream):
        ids = torch.empty((wp.M, wp.K), dtype=torch.int32, device=step.dev)
        sc = torch.empty((wp.M, wp.K), dtype=torch.float32, device=step.dev)
        ws = torch.empty(B.idx_topk_workspace_size(step.p, wp.K), dtype=torch.uint8, device=step.dev)
        B.idx_topk(step.p, wp.K, ids, sc, ws)
    torch.cuda.synchronize()
    del ws
    return ids, sc


if __name__ == "__main__":
    main()
