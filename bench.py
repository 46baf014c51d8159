"""Benchmark of the paged KV-cache hot path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long_gqa] [--batch B] [--no-extra]

A step is one pass of the whole path over one batch: paged_kv_append of the
step's new K/V rows at slot_mapping, then paged attention through
block_table (decode: one launch of the split-KV kernel, whose cut segments
are merged inside it).  The default workload is the largest single-GPU one:
long-context decode, 256 sequences with contexts U[1024, 32768], 32 query /
8 KV heads, head_dim 128, page_size 16 (about 17.7 GB of K/V read per step).
Inputs are synthetic, seeded, and resident in HBM; the L2 is flushed (256 MB
write, then 256 MB read of another buffer, both untimed) between timed
steps.  `value` is the decode KV-read throughput of the whole job: the
algorithmic K+V bytes every rank's step must read, divided by the mean step
time (max over ranks).

--impl reference times the fp64 CPU oracle (the only reference there is) on
the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from serving_slot_mapping_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attn decode KV-read GB/s (% of HBM peak), tokens/s; prefill TFLOP/s"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0


# ---------------------------------------------------------------------------
# plumbing
# ---------------------------------------------------------------------------

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_gqa")
    ap.add_argument("--batch", type=int, default=0,
                    help="decode workloads: keep only the first B sequences (a scaled-down case for "
                         "profiling; 0 = the workload as defined)")
    ap.add_argument("--cpu-oracle-json", default="", help=argparse.SUPPRESS)
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="oracle CPU-baseline sample length per thread setting; <= 0 skips it")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e leg")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="decode workloads: pool element type (e4m3: one scale per pool and tensor)")
    ap.add_argument("--decode", default="plain", choices=["plain", "fused", "csr", "cascade"],
                    help="decode workloads: the call a step makes (plain: append + decode; fused: "
                         "paged_attention_decode_append; csr: append + the CSR call; cascade: append + "
                         "cascade decode over the batch's shared prefix)")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


def file_hash(*paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def repeatability(times, repeats=5, limit=1.05):
    """The timed steps cut into ``repeats`` consecutive runs: the median of the
    runs' mean step times, their spread (slowest / fastest run) and whether the
    spread is within ``limit`` (a number whose runs disagree by more is flagged
    as not reportable)."""
    times = [float(t) for t in times]
    k = max(1, min(repeats, len(times)))
    if not times:
        return {"repeats": 0, "median_ms": None, "spread": None, "reportable": False}
    size = len(times) // k
    runs = [statistics.mean(times[i * size:(i + 1) * size if i < k - 1 else len(times)]) for i in range(k)]
    spread = max(runs) / min(runs) if min(runs) > 0 else None
    return {"repeats": k, "median_ms": round(statistics.median(runs), 5),
            "spread": round(spread, 4) if spread is not None else None,
            "reportable": spread is not None and spread <= limit}


def traffic_for(kernel_key: str):
    """Per-launch DRAM bytes from a committed ncu capture, if the kernel source
    is unchanged since the capture (else None)."""
    try:
        with open(TRAFFIC_PATH) as f:
            table = json.load(f)
        ent = table[kernel_key]
        if ent["source_hash"] != file_hash(*ent["sources"]):
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            text, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            text = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in text.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Untimed L2 flush between timed steps: write one buffer larger than L2,
    then read a second one, so the write-backs of the flush's own dirty lines
    happen here and the timed step starts from a clean L2 that holds none of
    its inputs."""

    def __init__(self, dev):
        n = L2_FLUSH_BYTES // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def timed_graph(graph, steps, flush, stream):
    """Replay `graph` `steps` times, flushing L2 between replays; per-replay ms."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            graph.replay()
            e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def capture(fn, stream, warm=3):
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def first_sequences(plan, batch: int):
    """The first ``batch`` sequences of a decode workload on a pool of their
    own (same lengths, heads, page size and share of free pages): the
    scaled-down case an ncu capture of a full-size workload is taken on."""
    if batch <= 0 or batch >= plan.batch:
        return plan
    if plan.kind != "decode" or wl.shared_prefix_pages(plan) > 0:
        raise ValueError(f"--batch applies to decode workloads without shared pages, not {plan.name}")
    free = 0.10 if plan.name.startswith("long") else 0.0
    return wl.plan_from_lengths(f"{plan.name}_first{batch}", plan.kind, plan.dtype, plan.num_q_heads,
                                plan.num_kv_heads, plan.head_dim, plan.page_size, plan.cached[:batch],
                                plan.new[:batch], plan.seed, free_frac=free, scale=plan.scale)


def rank_plan(name: str, rank: int, batch: int = 0):
    """The workload of one rank: same shapes, a rank-specific seed (weak scaling)."""
    if rank == 0:
        return first_sequences(wl.named_plan(name), batch)
    base = {"gqa_decode": lambda s: wl.gqa_decode_plan(seed=s),
            "shared_prefix": lambda s: wl.shared_prefix_plan(seed=s),
            "chunked_prefill": lambda s: wl.chunked_prefill_plan(seed=s),
            "long_gqa": lambda s: wl.long_context_plan(hkv=8, seed=s),
            "long_mqa": lambda s: wl.long_context_plan(hkv=1, seed=s)}[name]
    return first_sequences(base(1000 + 97 * rank), batch)


def measure_read_peak(dev, gib=4, reps=5):
    """Read-only HBM streaming rate (GB/s) of this GPU, measured live: the best
    of a few full reductions over a buffer far larger than L2 (torch's sum of
    an int64 view, which reads every byte once and writes one word).  A
    decode kernel only reads its K/V, so this is the bandwidth it can reach;
    the copy figure of the measured peaks moves each byte twice (read and
    write) and is lower."""
    try:
        x = torch.empty((gib << 30) // 8, dtype=torch.int64, device=dev)
        x.fill_(1)
        out = torch.empty((), dtype=torch.int64, device=dev)
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            torch.sum(x, dim=0, out=out)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        gbs = x.numel() * 8 / (best * 1e-3) / 1e9
        del x
        torch.cuda.empty_cache()
        return round(gbs, 1)
    except Exception:
        return None


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s figure the HBM3e of a GB300 is quoted at


def to_e4m3(pool, sc):
    """Pool codes from torch's own e4m3 conversion (test inputs only; the timed
    steps use the library's quantising append)."""
    out8 = torch.empty(pool.shape, dtype=torch.float8_e4m3fn, device=pool.device)
    step = max(1, (256 << 20) // max(1, pool[0].numel() * 4))
    for i in range(0, pool.shape[0], step):
        out8[i:i + step] = (pool[i:i + step].float() / sc).to(torch.float8_e4m3fn)
    return out8


class DecodeRig:
    """Device-resident decode workload.  A step consumes the tensors of
    ``inputs`` (q, this step's K/V rows and slots, the page table in the
    mode's form) and runs the mode's calls: append + decode (plain, csr,
    cascade) or the fused call."""

    E4M3_SCALE = 0.02

    def __init__(self, plan, dev, kv_dtype="bf16", mode="plain"):
        from serving_slot_mapping_gb300 import capi
        self.capi = capi
        self.plan = plan
        self.mode = mode
        self.st = wl.materialize(plan, dev)
        self.kv8 = kv_dtype == "e4m3"
        self.ks = self.vs = self.E4M3_SCALE if self.kv8 else 1.0
        if self.kv8 and mode == "cascade":
            raise ValueError("cascade decode takes bf16 pools")
        if self.kv8:
            self.st.key_pool = to_e4m3(self.st.key_pool, self.ks)
            self.st.value_pool = to_e4m3(self.st.value_pool, self.vs)
            torch.cuda.empty_cache()
        self.out = torch.empty_like(self.st.q)
        st = self.st
        self.inputs = {"q": st.q, "key": st.key, "value": st.value, "slot_mapping": st.slot_mapping}
        self.msl = int(plan.seq_lens.max())
        if mode == "csr":
            ip, ix, last = (torch.from_numpy(a).to(dev) for a in wl.csr_tables(plan))
            self.inputs.update(kv_indptr=ip, kv_indices=ix, kv_last_page_len=last)
        elif mode == "cascade":
            pages = wl.shared_prefix_pages(plan)
            if pages == 0:
                raise ValueError(f"{plan.name}: no page shared by the whole batch")
            pre, self.prefix_len, own_bt, own_lens = wl.cascade_tables(plan, pages, pages * plan.page_size)
            self.inputs.update(prefix_pages=torch.from_numpy(pre).to(dev),
                               block_table=torch.from_numpy(own_bt).to(dev),
                               seq_lens=torch.from_numpy(own_lens).to(dev))
            self.msl = int(own_lens.max())
        else:
            self.inputs.update(block_table=st.block_table, seq_lens=st.seq_lens)
        self.ws = (capi.cascade_workspace(plan.batch, plan.num_q_heads, st.key_pool) if mode == "cascade"
                   else capi.decode_workspace(plan.batch, plan.num_q_heads, st.key_pool))

    def kv_bytes(self):
        """Algorithmic K/V bytes a step's attention reads."""
        return wl.decode_kv_bytes(self.plan) // (2 if self.kv8 else 1)

    def append_with(self, t):
        st = self.st
        self.capi.paged_kv_append(st.key_pool, st.value_pool, t["key"], t["value"], t["slot_mapping"],
                                  k_scale=self.ks, v_scale=self.vs)

    def decode_with(self, t):
        st, c, p = self.st, self.capi, self.plan
        kw = dict(max_seq_len=self.msl, out=self.out, workspace=self.ws)
        if self.mode == "csr":
            c.paged_attention_decode_csr(st.key_pool, st.value_pool, t["q"], t["kv_indptr"], t["kv_indices"],
                                         t["kv_last_page_len"], p.scale, k_scale=self.ks, v_scale=self.vs, **kw)
        elif self.mode == "cascade":
            c.paged_attention_decode_cascade(st.key_pool, st.value_pool, t["q"], t["prefix_pages"],
                                             self.prefix_len, t["block_table"], t["seq_lens"], p.scale, **kw)
        else:
            c.paged_attention_decode(st.key_pool, st.value_pool, t["q"], t["block_table"], t["seq_lens"],
                                     p.scale, k_scale=self.ks, v_scale=self.vs, **kw)

    def step_with(self, t):
        if self.mode == "fused":
            st = self.st
            self.capi.paged_attention_decode_append(
                st.key_pool, st.value_pool, t["key"], t["value"], t["slot_mapping"], t["q"], t["block_table"],
                t["seq_lens"], self.plan.scale, max_seq_len=self.msl, out=self.out, workspace=self.ws,
                k_scale=self.ks, v_scale=self.vs)
        else:
            self.append_with(t)
            self.decode_with(t)

    def launches_per_step(self):
        return {"fused": 1, "cascade": 4}.get(self.mode, 2)  # cascade: append, prefix pass, split, combine

    # the device-resident forms
    def append(self):
        self.append_with(self.inputs)

    def decode(self):
        self.decode_with(self.inputs)

    def step(self):
        self.step_with(self.inputs)

    def fused_step(self):
        """The plain step as one call (one launch): append + decode."""
        st = self.st
        self.capi.paged_attention_decode_append(st.key_pool, st.value_pool, st.key, st.value,
                                                st.slot_mapping, st.q, st.block_table, st.seq_lens,
                                                self.plan.scale, max_seq_len=self.msl, out=self.out,
                                                workspace=self.ws, k_scale=self.ks, v_scale=self.vs)


class PrefillRig:
    """Device-resident prefill workload (bf16 pools, or e4m3 pools with one
    scale per pool and tensor): a step appends the new rows and prefills."""

    E4M3_SCALE = 0.02

    def __init__(self, plan, dev, kv_dtype="bf16"):
        from serving_slot_mapping_gb300 import capi
        self.capi = capi
        self.plan = plan
        self.st = wl.materialize(plan, dev)
        self.kv8 = kv_dtype == "e4m3"
        self.ks = self.vs = self.E4M3_SCALE if self.kv8 else 1.0
        if self.kv8:
            self.st.key_pool = to_e4m3(self.st.key_pool, self.ks)
            self.st.value_pool = to_e4m3(self.st.value_pool, self.vs)
        self.out = torch.empty_like(self.st.q)
        self.mql = int(plan.new.max())
        self.msl = int(plan.seq_lens.max())

    def append(self):
        st = self.st
        self.capi.paged_kv_append(st.key_pool, st.value_pool, st.key, st.value, st.slot_mapping,
                                  k_scale=self.ks, v_scale=self.vs)

    def prefill(self):
        st = self.st
        self.capi.paged_attention_prefill(st.key_pool, st.value_pool, st.q, st.query_start_loc,
                                          st.block_table, st.seq_lens, self.plan.scale,
                                          max_q_len=self.mql, max_seq_len=self.msl, out=self.out,
                                          k_scale=self.ks, v_scale=self.vs)

    def step(self):
        self.append()
        self.prefill()


def e2e_decode(rig: DecodeRig, steps, flush):
    """Same metric through the public API with host (pinned) inputs and output:
    H2D of the step's inputs (q, new K/V, slot_mapping, the page table in the
    mode's form); D2H of out."""
    host = {n: t.cpu().pin_memory() for n, t in rig.inputs.items()}
    dev = {n: torch.empty_like(t) for n, t in rig.inputs.items()}
    out_h = torch.empty(rig.out.shape, dtype=rig.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    stream = torch.cuda.current_stream()

    def one():
        for n in host:
            dev[n].copy_(host[n], non_blocking=True)
        rig.step_with(dev)
        out_h.copy_(rig.out, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        one()
        e.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(s.elapsed_time(e) for s, e in ev)
    return ms, h2d, d2h


class OracleRig:
    """The fp64 CPU oracle (as it stands) on a bounded sample of a decode
    workload: the first k sequences, with their own compact page pool (same
    lengths, heads, page size and value distribution).  One step = oracle
    append of the new rows + widening to fp64 + oracle decode."""

    unit = UNIT

    def __init__(self, plan, k):
        k = min(plan.batch, k)
        self.k = k
        self.plan = wl.plan_from_lengths(plan.name + "_sample", plan.kind, plan.dtype,
                                         plan.num_q_heads, plan.num_kv_heads, plan.head_dim,
                                         plan.page_size, plan.cached[:k], plan.new[:k],
                                         plan.seed, scale=plan.scale)
        st = wl.materialize(self.plan, "cpu")
        self.kb, self.vb = self._bits(st.key_pool), self._bits(st.value_pool)
        self.kn, self.vn = self._bits(st.key), self._bits(st.value)
        self.q = self._f64(self._bits(st.q))
        self.full_batch = plan.batch
        self.name = plan.name
        self.full_work = wl.decode_kv_bytes(plan)

    @staticmethod
    def _bits(t):
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
            else t.numpy()

    @staticmethod
    def _f64(a):
        if a.dtype == np.uint16:
            return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return a.astype(np.float64)

    def step(self):
        import oracle
        p = self.plan
        k2, v2 = oracle.paged_kv_append(self.kb, self.vb, self.kn, self.vn, p.slot_mapping)
        oracle.paged_attention_decode(self._f64(k2), self._f64(v2), self.q, p.block_table,
                                      p.seq_lens, p.scale)

    @property
    def work(self):
        """Algorithmic K/V bytes of the sample's decode."""
        return wl.decode_kv_bytes(self.plan)

    def rate(self, seconds_per_step):
        return self.work / seconds_per_step / 1e9

    def describe(self, reps, el):
        return (f"oracle append+decode of the first {self.k}/{self.full_batch} sequences of {self.name} "
                f"(compact pool of {self.plan.num_pages} pages), {reps} reps in {el:.1f}s; the rate is "
                f"the sample's KV bytes / its step time, extrapolated linearly to the whole batch")


class PrefillOracleRig(OracleRig):
    """The oracle on a bounded sample of a prefill workload: the first k
    sequences (all their new rows, after their cached context), on a compact
    pool.  One step = oracle append + widening + oracle varlen causal prefill."""

    unit = "TFLOP/s"

    def __init__(self, plan, k):
        k = min(plan.batch, k)
        self.k = k
        self.plan = wl.plan_from_lengths(plan.name + "_sample", plan.kind, plan.dtype,
                                         plan.num_q_heads, plan.num_kv_heads, plan.head_dim,
                                         plan.page_size, plan.cached[:k], plan.new[:k],
                                         plan.seed, scale=plan.scale)
        st = wl.materialize(self.plan, "cpu")
        self.kb, self.vb = self._bits(st.key_pool), self._bits(st.value_pool)
        self.kn, self.vn = self._bits(st.key), self._bits(st.value)
        self.q = self._f64(self._bits(st.q))
        self.full_batch = plan.batch
        self.name = plan.name
        self.full_work = wl.prefill_flops(plan)

    def step(self):
        import oracle
        p = self.plan
        k2, v2 = oracle.paged_kv_append(self.kb, self.vb, self.kn, self.vn, p.slot_mapping)
        oracle.paged_attention_prefill(self._f64(k2), self._f64(v2), self.q, p.query_start_loc,
                                       p.block_table, p.seq_lens, p.scale)

    @property
    def work(self):
        """FLOPs of the sample's visible (query, key) pairs."""
        return wl.prefill_flops(self.plan)

    def rate(self, seconds_per_step):
        return self.work / seconds_per_step / 1e12

    def describe(self, reps, el):
        return (f"oracle append+prefill of the first {self.k}/{self.full_batch} sequences of {self.name} "
                f"({self.plan.total_new} new rows), {reps} reps in {el:.1f}s; the rate is the sample's "
                f"visible-pair FLOPs / its step time, extrapolated linearly to the whole batch")


# sequences per oracle sample: CPU baseline (about ten seconds a leg) and
# reference arm (each of its steps; the whole --steps/--warmup run in minutes)
CPU_SAMPLE = {"decode": 16, "prefill": 2}
REF_SAMPLE = {"decode": 4, "prefill": 1}


def oracle_rig(plan, k):
    return (OracleRig if plan.kind == "decode" else PrefillOracleRig)(plan, k)


def time_oracle(rig, seconds: float):
    """Step the oracle for about `seconds` (at least once): (rate, s/step, reps, elapsed)."""
    reps = 0
    t0 = time.perf_counter()
    while True:
        rig.step()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    per = el / reps
    return rig.rate(per), per, reps, el


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def cpu_oracle_child(spec: str):
    """Body of the CPU-baseline subprocess: time the oracle on the sample and
    print one JSON object (the BLAS thread count was fixed by the parent
    through the environment, before numpy loaded)."""
    sp = json.loads(spec)
    plan = first_sequences(wl.named_plan(sp["workload"]), sp.get("batch", 0))
    rig = oracle_rig(plan, sp["sample"])
    rate, per, reps, el = time_oracle(rig, sp["seconds"])
    print(json.dumps({"value": rate, "unit": rig.unit, "s_per_step": per,
                      "full_step_s": per * rig.full_work / rig.work, "sample": rig.describe(reps, el)}))


def cpu_baseline(workload, batch, seconds, kind):
    """The oracle timed on the host cores in a subprocess per thread setting:
    every core of this process's affinity mask, then one thread.  Returns the
    cpu_baseline object of the JSON line (None if it could not run)."""
    cores = cpu_cores()
    legs = {}
    for threads in (cores, 1):
        env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
        for v in THREAD_VARS:
            env[v] = str(threads)
        spec = json.dumps({"workload": workload, "batch": batch, "seconds": seconds,
                           "sample": CPU_SAMPLE[kind]})
        try:
            r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-oracle-json", spec],
                               env=env, capture_output=True, text=True, timeout=900, cwd=ROOT)
            legs[threads] = json.loads(r.stdout.strip().splitlines()[-1])
        except Exception as ex:
            legs[threads] = {"error": repr(ex)[:200]}
    full = legs.get(cores, {})
    one = legs.get(1, {})
    if "value" not in full:
        return {"error": full.get("error", "no result"), "kind": "oracle", "cores": cores}
    digits = 4 if full["unit"] == UNIT else 6
    return {"value": round(full["value"], digits), "unit": full["unit"], "cores": cores, "kind": "oracle",
            "sample": full["sample"] + f"; BLAS threads = {cores} (the process's affinity mask)",
            "s_per_step": round(full["s_per_step"], 3),
            "full_step_s_extrapolated": round(full["full_step_s"], 2),
            "one_thread": ({"value": round(one["value"], digits), "cores": 1,
                            "s_per_step": round(one["s_per_step"], 3)} if "value" in one else one)}


REPEAT_RUNS, REPEAT_REPLAYS = 5, 50  # repeatability: runs x replays, whatever --steps is


def hbm_fractions(achieved, hbm, read_peak):
    """achieved GB/s against the measured copy peak, the live read-only peak
    and the nominal 8 TB/s."""
    return {"frac_of_copy_peak": round(achieved / hbm, 4),
            "read_peak": read_peak,
            "frac_of_read_peak": round(achieved / read_peak, 4) if read_peak else None,
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}


def run_ours(args, rank, world, local):
    from serving_slot_mapping_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    read_peak = measure_read_peak(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)

    plan = rank_plan(args.workload, rank, args.batch)
    if plan.kind == "prefill":
        return run_prefill_line(args, rank, world, local, plan, dev, flush, stream, bf16, bf16_sus, peak_src)
    rig = DecodeRig(plan, dev, args.kv_dtype, args.decode)
    g_step = capture(rig.step, stream)
    # the attention call alone (fused: the step is that one call)
    g_dec = capture(rig.step if args.decode == "fused" else rig.decode, stream)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    times = timed_graph(g_step, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    # the attention call alone (plain: one launch, merges included), same flushing
    dec_times = timed_graph(g_dec, max(50, args.steps), flush, stream)
    clocks = sampler.stop()
    # repeatability of the step on runs long enough to mean something
    rep_times = timed_graph(g_step, REPEAT_RUNS * REPEAT_REPLAYS, flush, stream)

    ms_step = max_over_ranks(statistics.mean(times), world)
    kv_bytes = rig.kv_bytes()
    total_kv = sum_over_ranks(float(kv_bytes), world)
    value = total_kv / (ms_step * 1e-3) / 1e9
    tokens_s = sum_over_ranks(float(plan.batch), world) / (ms_step * 1e-3)

    dec_ms = statistics.mean(dec_times)
    # algorithmic bytes of the attention call: cascade reads the shared prefix once
    unique = wl.decode_unique_kv_bytes(plan) if args.decode == "cascade" else None
    dec_bytes = (unique if unique is not None else kv_bytes) + wl.decode_io_bytes(plan)
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    variant = "" if (args.kv_dtype, args.decode) == ("bf16", "plain") else f":{args.kv_dtype}:{args.decode}"
    traffic = traffic_for(f"decode_split:{plan.name}{variant}")
    call = {"plain": "paged_attention_decode (decode_split_kernel, in-kernel merges)",
            "fused": "paged_attention_decode_append (decode_split_kernel, fused append)",
            "csr": "paged_attention_decode_csr (decode_split_kernel)",
            "cascade": "paged_attention_decode_cascade"}[args.decode]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "kernel": call + (" on e4m3 pools" if rig.kv8 else ""),
                "algorithmic_bytes_per_launch": dec_bytes,
                "ms_per_launch": round(dec_ms, 5), "peak_source": peak_src + " (copy: read + write)"}
    roofline.update(hbm_fractions(achieved, hbm, read_peak))

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_decode(rig, max(20, min(args.steps, 200)), flush)
        e2e_ms = max_over_ranks(e2e_ms, world)
        e2e = {"value": round(total_kv / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 5)}

    extra = {}
    if not args.no_extra and rank == 0:
        extra = run_extra(dev, flush, stream, hbm, bf16, bf16_sus, read_peak)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(args.workload, args.batch, args.cpu_seconds, "decode")

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_median": round(max_over_ranks(statistics.median(times), world), 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV, f16 products" if rig.kv8 else "bf16",
        "data": "synthetic",
        "config": {"workload": plan.name, "batch": plan.batch, "num_q_heads": plan.num_q_heads,
                   "num_kv_heads": plan.num_kv_heads, "head_dim": plan.head_dim,
                   "page_size": plan.page_size,
                   "context": f"{int(plan.seq_lens.min())}..{int(plan.seq_lens.max())} keys",
                   "kv_dtype": args.kv_dtype, "decode_call": args.decode,
                   "kv_bytes_per_step": kv_bytes,
                   "unique_kv_bytes_per_step": wl.decode_unique_kv_bytes(plan) // (2 if rig.kv8 else 1),
                   "step": "append 1 token/seq + decode" + (" (one call)" if args.decode == "fused" else ""),
                   "l2": "flushed between timed steps (256 MB write + 256 MB read, untimed)",
                   "timing": "mean of the timed steps (CUDA events, one graph replay each; the event "
                             "clock ticks in ~2 us steps, which a mean averages out and a median does not)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tokens_per_s": round(tokens_s, 1),
        "pct_of_hbm_peak": round(100.0 * value / (hbm * world), 2),
        "repeatability": dict(repeatability(rep_times, REPEAT_RUNS),
                              replays_per_run=REPEAT_REPLAYS),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": rig.launches_per_step() * args.steps,
        "extra": extra,
    }
    return line


def e2e_prefill(rig, steps, flush):
    """The prefill step through the public API with host (pinned) inputs and
    output: H2D of q, the new K/V rows, slot_mapping and the page metadata;
    D2H of out."""
    st = rig.st
    names = ("q", "key", "value", "slot_mapping", "query_start_loc", "block_table", "seq_lens")
    host = {n: getattr(st, n).cpu().pin_memory() for n in names}
    dev = {n: torch.empty_like(getattr(st, n)) for n in names}
    out_h = torch.empty(rig.out.shape, dtype=rig.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    stream = torch.cuda.current_stream()
    c, p = rig.capi, rig.plan

    def one():
        for n in host:
            dev[n].copy_(host[n], non_blocking=True)
        c.paged_kv_append(st.key_pool, st.value_pool, dev["key"], dev["value"], dev["slot_mapping"],
                          k_scale=rig.ks, v_scale=rig.vs)
        c.paged_attention_prefill(st.key_pool, st.value_pool, dev["q"], dev["query_start_loc"],
                                  dev["block_table"], dev["seq_lens"], p.scale, max_q_len=rig.mql,
                                  max_seq_len=rig.msl, out=rig.out, k_scale=rig.ks, v_scale=rig.vs)
        out_h.copy_(rig.out, non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_, e_ in ev:
        flush.zero_()
        s_.record(stream)
        one()
        e_.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s_.elapsed_time(e_) for s_, e_ in ev), h2d, d2h


def run_prefill_line(args, rank, world, local, plan, dev, flush, stream, bf16, bf16_sus, peak_src):
    """Main line for a prefill workload: append of the new tokens + varlen
    causal prefill per step; value in TFLOP/s of visible (query, key) pairs."""
    rig = PrefillRig(plan, dev, args.kv_dtype)
    g_step = capture(rig.step, stream)
    g_pf = capture(rig.prefill, stream)
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    times = timed_graph(g_step, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    pf_times = timed_graph(g_pf, max(20, args.steps), flush, stream)
    clocks = sampler.stop()
    rep_times = timed_graph(g_step, REPEAT_RUNS * REPEAT_REPLAYS, flush, stream)
    ms_step = max_over_ranks(statistics.mean(times), world)
    flops = wl.prefill_flops(plan)
    total_flops = sum_over_ranks(float(flops), world)
    value = total_flops / (ms_step * 1e-3) / 1e12
    pf_ms = statistics.mean(pf_times)
    achieved = flops / (pf_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_prefill(rig, max(20, min(args.steps, 100)), flush)
        e2e_ms = max_over_ranks(e2e_ms, world)
        e2e = {"value": round(total_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)}
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(args.workload, 0, args.cpu_seconds, "prefill")
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_median": round(max_over_ranks(statistics.median(times), world), 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV, f16 products" if rig.kv8 else "bf16",
        "data": "synthetic",
        "config": {"workload": plan.name, "batch": plan.batch, "num_q_heads": plan.num_q_heads,
                   "num_kv_heads": plan.num_kv_heads, "head_dim": plan.head_dim,
                   "page_size": plan.page_size, "kv_dtype": args.kv_dtype, "new_tokens": plan.total_new,
                   "visible_pairs": wl.prefill_visible_pairs(plan), "flops_per_step": flops,
                   "step": "append new tokens + varlen causal prefill",
                   "l2": "flushed between timed steps (256 MB write + 256 MB read, untimed)",
                   "timing": "mean of the timed steps (CUDA events, one graph replay each)"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16, 4),
                     "traffic": traffic_for(f"prefill:{plan.name}" + (":e4m3" if rig.kv8 else "")),
                     "kernel": "paged_attention_prefill (prefill_tc_kernel" + (", e4m3 pools)" if rig.kv8 else ")"),
                     "ms_per_launch": round(pf_ms, 5),
                     "peak_source": peak_src + " (bf16 burst)", "peak_sustained": bf16_sus,
                     "frac_of_sustained": round(achieved / bf16_sus, 4)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks, "gpu_launches": 2 * args.steps,
        "repeatability": dict(repeatability(rep_times, REPEAT_RUNS), replays_per_run=REPEAT_REPLAYS),
    }


def run_extra(dev, flush, stream, hbm, bf16, bf16_sus, read_peak, steps=30):
    """The other workloads, one number each (same flushing, CUDA graphs,
    median of the replays)."""
    res = {}
    for name in ["gqa_decode", "shared_prefix", "long_mqa"]:
        try:
            plan = wl.named_plan(name)
            rig = DecodeRig(plan, dev)
            g = capture(rig.decode, stream)
            ms = statistics.mean(timed_graph(g, max(steps, 100), flush, stream))
            kvb = wl.decode_kv_bytes(plan)
            io = wl.decode_io_bytes(plan)
            gbs = (kvb + io) / (ms * 1e-3) / 1e9
            ent = {"decode_ms": round(ms, 5), "kv_GBps": round(gbs, 1),
                   "frac_hbm": round(gbs / hbm, 4),
                   "tokens_per_s": round(plan.batch / (ms * 1e-3), 1)}
            ent.update(hbm_fractions(gbs, hbm, read_peak))
            if name == "shared_prefix":
                ub = wl.decode_unique_kv_bytes(plan)
                ent["unique_kv_GBps"] = round(ub / (ms * 1e-3) / 1e9, 1)
                ent["unique_frac_hbm"] = round(ub / (ms * 1e-3) / 1e9 / hbm, 4)
                # the same batch through cascade decode: the shared prefix read once
                pages = wl.shared_prefix_pages(plan)
                pre, plen, own_bt, own_lens = wl.cascade_tables(plan, pages, pages * plan.page_size)
                cw = rig.capi.cascade_workspace(plan.batch, plan.num_q_heads, rig.st.key_pool)
                pre_t = torch.from_numpy(pre).to(dev)
                bt_t = torch.from_numpy(own_bt).to(dev)
                sl_t = torch.from_numpy(own_lens).to(dev)
                msl = int(own_lens.max())

                def cascade():
                    rig.capi.paged_attention_decode_cascade(
                        rig.st.key_pool, rig.st.value_pool, rig.st.q, pre_t, plen, bt_t, sl_t,
                        plan.scale, max_seq_len=msl, out=rig.out, workspace=cw)
                gc = capture(cascade, stream)
                cms = statistics.mean(timed_graph(gc, max(steps, 100), flush, stream))
                ent["cascade_ms"] = round(cms, 5)
                ent["cascade_unique_GBps"] = round(ub / (cms * 1e-3) / 1e9, 1)
                ent["cascade_unique_frac_hbm"] = round(ub / (cms * 1e-3) / 1e9 / hbm, 4)
                ent["cascade_tokens_per_s"] = round(plan.batch / (cms * 1e-3), 1)
                del gc
            res[name] = ent
            del rig, g
            torch.cuda.empty_cache()
        except Exception as ex:  # report, do not hide
            res[name] = {"error": repr(ex)[:200]}
    for name in ["gqa_decode", "long_gqa", "long_mqa"]:  # the same batches on e4m3 pools
        try:
            plan = wl.named_plan(name)
            rig = DecodeRig(plan, dev, "e4m3")
            g = capture(rig.decode, stream)
            ms = statistics.mean(timed_graph(g, steps, flush, stream))
            kvb = wl.decode_kv_bytes(plan) // 2 + wl.decode_io_bytes(plan)
            res[name + "_fp8"] = {"decode_ms": round(ms, 5), "kv_GBps": round(kvb / (ms * 1e-3) / 1e9, 1),
                                  "frac_hbm": round(kvb / (ms * 1e-3) / 1e9 / hbm, 4),
                                  "tokens_per_s": round(plan.batch / (ms * 1e-3), 1),
                                  "speedup_vs_bf16_pool": None}
            bf = res.get(name, {}).get("decode_ms")
            if bf is None:  # long_gqa is the main line: time its bf16 decode here too
                rig16 = DecodeRig(plan, dev)
                g16 = capture(rig16.decode, stream)
                bf = statistics.mean(timed_graph(g16, steps, flush, stream))
                del rig16, g16
                torch.cuda.empty_cache()
            res[name + "_fp8"]["bf16_pool_decode_ms"] = round(bf, 5)
            res[name + "_fp8"]["speedup_vs_bf16_pool"] = round(bf / ms, 3)
            del rig, g
            torch.cuda.empty_cache()
        except Exception as ex:
            res[name + "_fp8"] = {"error": repr(ex)[:200]}
    for name in ["gqa_decode", "long_gqa"]:  # append + decode as one call vs two
        try:
            plan = wl.named_plan(name)
            rig = DecodeRig(plan, dev)
            g2 = capture(rig.step, stream)
            g1 = capture(rig.fused_step, stream)
            ms2 = statistics.mean(timed_graph(g2, steps, flush, stream))
            ms1 = statistics.mean(timed_graph(g1, steps, flush, stream))
            kvb = wl.decode_kv_bytes(plan)
            res[name + "_fused_step"] = {"step_ms": round(ms1, 5), "two_call_step_ms": round(ms2, 5),
                                         "kv_GBps": round(kvb / (ms1 * 1e-3) / 1e9, 1),
                                         "frac_hbm": round(kvb / (ms1 * 1e-3) / 1e9 / hbm, 4),
                                         "speedup_vs_two_calls": round(ms2 / ms1, 3)}
            del rig, g1, g2
            torch.cuda.empty_cache()
        except Exception as ex:
            res[name + "_fused_step"] = {"error": repr(ex)[:200]}
    try:  # the GQA decode batch with its page table in CSR form
        plan = wl.named_plan("gqa_decode")
        rig = DecodeRig(plan, dev)
        rig.append()
        ip, ix, last = (torch.from_numpy(a).to(dev) for a in wl.csr_tables(plan))
        msl = int(plan.seq_lens.max())

        def decode_csr():
            rig.capi.paged_attention_decode_csr(rig.st.key_pool, rig.st.value_pool, rig.st.q, ip, ix, last,
                                                plan.scale, max_seq_len=msl, out=rig.out, workspace=rig.ws)
        g = capture(decode_csr, stream)
        ms = statistics.mean(timed_graph(g, max(steps, 100), flush, stream))
        kvb = wl.decode_kv_bytes(plan) + wl.decode_io_bytes(plan)
        res["gqa_decode_csr"] = {"decode_ms": round(ms, 5), "kv_GBps": round(kvb / (ms * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(kvb / (ms * 1e-3) / 1e9 / hbm, 4)}
        del rig, g
    except Exception as ex:
        res["gqa_decode_csr"] = {"error": repr(ex)[:200]}
    try:
        plan = wl.named_plan("chunked_prefill")
        rig = PrefillRig(plan, dev)
        g = capture(rig.prefill, stream)
        ms = statistics.mean(timed_graph(g, steps, flush, stream))
        ga = capture(rig.append, stream)
        ams = statistics.mean(timed_graph(ga, max(steps, 100), flush, stream))
        fl = wl.prefill_flops(plan)
        tf = fl / (ms * 1e-3) / 1e12
        ab = wl.append_bytes(plan)
        res["chunked_prefill"] = {
            "prefill_ms": round(ms, 4), "TFLOPs": round(tf, 1),
            "frac_bf16_burst": round(tf / bf16, 4), "frac_bf16_sustained": round(tf / bf16_sus, 4),
            "visible_pairs": wl.prefill_visible_pairs(plan), "flops": fl,
            "append_ms": round(ams, 5), "append_GBps": round(ab / (ams * 1e-3) / 1e9, 1),
            "append_frac_hbm": round(ab / (ams * 1e-3) / 1e9 / hbm, 4)}
    except Exception as ex:
        res["chunked_prefill"] = {"error": repr(ex)[:200]}
    try:  # the same prefill on e4m3 pools (f16 products; codes converted in shared memory)
        plan = wl.named_plan("chunked_prefill")
        rig8 = PrefillRig(plan, dev, "e4m3")
        g = capture(rig8.prefill, stream)
        ms8 = statistics.mean(timed_graph(g, steps, flush, stream))
        tf8 = wl.prefill_flops(plan) / (ms8 * 1e-3) / 1e12
        ent = {"prefill_ms": round(ms8, 4), "TFLOPs": round(tf8, 1), "frac_bf16_burst": round(tf8 / bf16, 4)}
        if "prefill_ms" in res.get("chunked_prefill", {}):
            ent["time_vs_bf16_pool"] = round(ms8 / res["chunked_prefill"]["prefill_ms"], 3)
        res["chunked_prefill_fp8"] = ent
        del rig8, g
        torch.cuda.empty_cache()
    except Exception as ex:
        res["chunked_prefill_fp8"] = {"error": repr(ex)[:200]}
    return res


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return None
    plan = first_sequences(wl.named_plan(args.workload), args.batch)
    rig = oracle_rig(plan, REF_SAMPLE[plan.kind])   # each step: a bounded sample of the workload
    for _ in range(args.warmup):
        rig.step()
    pers = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        rig.step()
        pers.append(time.perf_counter() - t0)
    el = time.perf_counter() - t_all
    per = statistics.median(pers)
    value = rig.rate(per)
    digits = 4 if rig.unit == UNIT else 6
    cores = cpu_cores()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, digits), "unit": rig.unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": plan.name, "batch": plan.batch, "num_q_heads": plan.num_q_heads,
                   "num_kv_heads": plan.num_kv_heads, "head_dim": plan.head_dim,
                   "page_size": plan.page_size, "sample_sequences": rig.k},
        "cpu_baseline": {"value": round(value, digits), "unit": rig.unit, "cores": cores, "kind": "oracle",
                         "sample": rig.describe(len(pers), el)},
        "e2e": {"value": round(value, digits), "unit": rig.unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.cpu_oracle_json:   # the CPU-baseline subprocess (no GPU)
        cpu_oracle_child(args.cpu_oracle_json)
        return
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit at once without work
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup()
    line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
