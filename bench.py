"""Benchmark of one decode step of paged attention on GB300.

A step is one pass of the hot path over one batch: the append of the step's
K/V row for every (sequence, kv head) and decode attention over the L + 1
valid tokens, issued as one paged_attention_decode_append launch (or, with
--unfused and for split-KV workloads, paged_kv_append followed by
paged_attention_decode / the partial + reduce pair).  The default workload is the Llama-7B-like layer: 64 sequences,
32 heads (MHA), head_dim 128, fp16, block_size 16, lengths uniform in
450..520, 4096-block pool with shuffled ids.

Metric: algorithmic bytes of the step / step time in GB/s, where the bytes
are the valid K/V rows read (never padding), the block_table entries the
step needs, seq_lens, Q and O, plus the append's reads and writes.  Also
reported: query tokens/s, microseconds per layer-step, the decode kernel's
fraction of measured HBM bandwidth, an end-to-end figure with host buffers,
and the CPU oracle's throughput on the host cores.

The kernel's duration comes from a pass of 64 isolated launches after the
timed region (each bracketed by its own events, one launch after a
synchronize discarded), so it does not depend on --steps.  A one-GPU run
then measures the other configurations of the report the same way (the
five workloads, the long tail at block sizes 8/16/32/64, the GQA layer at
16/256, the int8 and fp8 caches, a pool 16 bytes off the 128-byte boundary)
and adds them to the same JSON line under "per_workload".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I]
       [--block-size BS] [--impl reference]
Under torchrun (N > 1) every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path
from types import SimpleNamespace

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

METRIC = "paged decode KV-read GB/s (% of GB300 HBM peak); attention tokens/s"
UNIT = "GB/s"
DTYPE_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
SPLIT_PTOK = {5: 1024}          # workloads timed through split-KV partitions
SHARED_PREFIX = {5: 4096}       # ... or with the shared prefix read once per group (partition)
SHARED_PREFIX_CODES = {5: 2048}  # the same over an int8 / fp8 cache (measured best of 1024-4096)
PROFILE_DIR = ROOT / "profiles"
KERNEL_SOURCES = {"decode_simt": "decode_simt.cu", "decode_gqa_tc": "decode_gqa_tc.cu",
                  "decode_gqa_umma": "decode_gqa_umma.cu",
                  "decode_simt_balanced": "decode_balanced_simt.cu",
                  "decode_tc_balanced": "decode_balanced_tc.cu",
                  "decode_int8": "decode_int8.cu",
                  "decode_int8_tc": "decode_int8_tc.cu",
                  "decode_fp8_tc": "decode_int8_tc.cu",
                  "decode_fp8": "decode_int8.cu",
                  "decode_prefix_tc": "decode_prefix_tc.cu",
                  "decode_prefix_int8_tc": "decode_int8_tc.cu",
                  "decode_prefix_fp8_tc": "decode_int8_tc.cu",
                  "append_tokens": "append.cu"}


# ---------------------------------------------------------------------------
# algorithmic byte counts
# ---------------------------------------------------------------------------

def decode_bytes(w, lens_after, window: int = 0) -> int:
    """Valid K/V rows + needed table entries + seq_lens + Q + O of one decode.

    Blocks shared by several table rows are counted once (they need to cross
    HBM once).  With a sliding window only the last `window` rows count.
    """
    s = w.q.element_size()
    s_kv = w.pool.element_size()           # 1 for an int8 or fp8 cache
    lens = [int(x) for x in lens_after]
    tab = w.block_table.cpu()
    row_bytes = w.Hkv * w.D * s_kv         # one token, all kv heads, K or V
    rows = {}                              # (block, slot) rows read, shared ones once
    tables = 0
    for b, L in enumerate(lens):
        lo = max(0, L - window) if window > 0 else 0
        j0, j1 = lo // w.bs, -(-L // w.bs)
        tables += j1 - j0
        for j in range(j0, j1):
            blk = int(tab[b, j])
            a, e = max(lo, j * w.bs) - j * w.bs, min(L, (j + 1) * w.bs) - j * w.bs
            cur = rows.get(blk)
            rows[blk] = (a, e) if cur is None else (min(cur[0], a), max(cur[1], e))
    kv = 2 * row_bytes * sum(e - a for a, e in rows.values())
    # a quantised cache also reads the K and V scales of every block it touches
    scales = 2 * 4 * w.Hkv * len(rows) if getattr(w, "scales", None) is not None else 0
    return kv + scales + 4 * tables + 4 * w.B + 2 * w.B * w.H * w.D * s


def prefill_bytes(w) -> int:
    """Prompt write of every sequence's L tokens: read the padded batch's
    valid rows, write them into the pool, plus positions, counts and the
    table entries the write needs."""
    s = w.q.element_size()
    lens = [int(x) for x in w.lens]
    rows = sum(lens)
    tables = sum(-(-L // w.bs) for L in lens)
    return 2 * 2 * rows * w.Hkv * w.D * s + 8 * w.B + 4 * tables


def logical_kv_bytes(w, lens_after) -> int:
    s = w.pool.element_size()
    return 2 * w.Hkv * w.D * s * sum(int(x) for x in lens_after)


def append_bytes(w) -> int:
    """Read the new K/V rows, write them into the pool (as codes for a quantised
    cache, which also reads the target blocks' scales), plus positions and
    table entries."""
    s = w.k_new.element_size()
    s_kv = w.pool.element_size()
    scales = 2 * 4 * w.B * w.Hkv if getattr(w, "scales", None) is not None else 0
    return 2 * w.B * w.Hkv * w.D * (s + s_kv) + scales + 4 * w.B + 4 * w.B


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                "clocks.mem")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict | None:
        if self.proc is None:
            return None
        sm, mx, mem, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "out", "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                if len(f) > 9:
                    mem.append(float(f[9]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "mem_mhz": statistics.median(mem) if mem else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def source_digest(name: str) -> str:
    """sha256 over a kernel source file and every header it includes from the
    tree (recursively), so that a change to shared device code also marks the
    counters taken on the old build as stale."""
    dirs = [ROOT / "pagedattention_decode_paged_gb300" / "csrc", ROOT / "include"]
    seen, order, todo = set(), [], [name]
    while todo:
        n = todo.pop(0)
        path = next((d / n for d in dirs if (d / n).exists()), None)
        if path is None or n in seen:
            continue
        seen.add(n)
        order.append(path)
        todo += re.findall(r'^#include "([^"]+)"', path.read_text(), flags=re.M)
    h = hashlib.sha256()
    for path in order:
        h.update(path.read_bytes())
    return h.hexdigest()


def kernel_traffic(kernel: str, workload: str, fused: bool = False) -> int | None:
    """DRAM bytes per launch from a committed ncu summary, if still current.

    Summaries are named <kernel>__<description>_<workload>[_fused].md.  Each
    records the source_digest() of its kernel at capture time; when the
    sources have changed since, the figure is stale and None is returned.
    """
    digest = source_digest(KERNEL_SOURCES[kernel])
    pat = re.compile(rf"^{re.escape(kernel)}__.*_{re.escape(workload)}(_fused)?\.md$")
    for f in sorted(PROFILE_DIR.glob(f"{kernel}__*.md")):
        m = pat.match(f.name)
        if m is None or (m.group(1) is not None) != fused:
            continue
        text = f.read_text()
        m_src = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
        if m_src and m_tr and m_src.group(1) == digest:
            return int(m_tr.group(1))
    return None


def replica_seed(workload: int, rank: int) -> int:
    """Seed of rank `rank`'s replica of a workload: every rank holds its own
    independent data (weak scaling, no collective on the data path)."""
    return 1000 + workload + 7 * rank


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of the ranks' values (the elapsed time a multi-rank run
    reports); `dist` is torch.distributed or None for one rank."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job GB/s: the bytes every rank moved in a step over the slowest
    rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def local_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


def describe(w, index) -> dict:
    lens = [int(x) for x in w.lens]
    return {"workload": f"{w.name} (workload {index})", "batch": w.B, "num_heads": w.H,
            "num_kv_heads": w.Hkv, "head_dim": w.D, "block_size": w.bs, "num_blocks": w.NB,
            "seq_len_min": min(lens) + 1, "seq_len_max": max(lens) + 1,
            "seq_len_mean": round(sum(lens) / len(lens) + 1, 1),
            "split_kv_partition": None}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def step_options(**over) -> SimpleNamespace:
    """The step-shaping flags of the command line, with their defaults."""
    o = dict(unfused=False, window=0, balanced=False, prefill=False, split_tokens=None,
             shared_prefix=None, int8=False, fp8=False, graph=0, long_seq=0, pool_offset=0, batch=None)
    o.update(over)
    return SimpleNamespace(**o)


def make_bench_workload(index, o, dev, rank=0, block_size=None, batch=None):
    """Workload `index` on `dev` as the options shape it: another batch size,
    a long request beside the batch, an int8 or fp8 cache (codes drawn on the
    device), or a pool moved `pool_offset` bytes off its 512-byte aligned
    allocation."""
    batch = o.batch if batch is None else batch
    w = workloads.make_workload(index, block_size=block_size, device=dev,
                                seed=replica_seed(index, rank), batch=batch)
    if o.long_seq:
        w = workloads.with_long_sequence(w, o.long_seq, seed=7 + rank, device=dev)
    if o.int8 and o.fp8:
        raise SystemExit("--int8 and --fp8 are two cache formats: pick one")
    if o.int8 or o.fp8:
        if o.prefill or o.window or o.balanced or o.graph:
            raise SystemExit("--int8 / --fp8 time the quantising append + decode pair only")
        w = (workloads.to_fp8(w, seed=19 + rank, device=dev) if o.fp8
             else workloads.to_int8(w, seed=17 + rank, device=dev))
    if o.pool_offset:
        es = w.pool.element_size()
        if o.pool_offset % 16 or o.pool_offset % es:
            raise SystemExit("--pool-offset must keep the 16-byte alignment the library requires")
        n = w.pool.numel()
        buf = torch.empty(n + 1024 // es, dtype=w.pool.dtype, device=dev)
        off = o.pool_offset // es
        buf[off:off + n].copy_(w.pool.view(-1))
        w.pool = buf[off:off + n].view(w.pool.shape)
    return w


class StepPlan:
    """One step of the hot path over workload `w` through the C ABI: the calls,
    the kernel they centre on and the bytes they move.

    A step is the append of the step's K/V row for every (sequence, kv head)
    and decode attention over the L + 1 valid tokens: one fused
    paged_attention_decode_append launch by default; append + decode (or the
    split-KV pair, or the shared-prefix split) as separate launches otherwise;
    the prompt write of every sequence for --prefill.
    """

    def __init__(self, pa, w, index, o, dev, stream):
        self.pa, self.w, self.index, self.o, self.stream = pa, w, index, o, stream
        kw = dict(block_size=w.bs, num_blocks=w.NB, block_stride=w.block_stride)
        self.kw = kw
        shape = pa.make_shape(batch=w.B, num_heads=w.H, num_kv_heads=w.Hkv, head_dim=w.D,
                              block_size=w.bs, max_blocks_per_seq=w.MB, num_blocks=w.NB,
                              block_stride=w.block_stride, dtype=w.dtype)
        which = pa.paged_attention_decode_kernel(shape, o.window or 0, 0)
        kernel = {pa.PA_KERNEL_TCGEN05: "decode_gqa_umma", pa.PA_KERNEL_MMA_SYNC: "decode_gqa_tc"}.get(
            which, "decode_simt")
        self.quant = "fp8" if o.fp8 else "int8" if o.int8 else None
        if o.int8:
            # grouped-query shapes with 16-bit queries and head_dim 64/128 run on
            # the tensor cores (the rule of paged_attention_decode_int8)
            tc8 = w.H // w.Hkv >= 2 and w.D in (64, 128) and w.dtype in (torch.float16, torch.bfloat16)
            kernel = "decode_int8_tc" if tc8 else "decode_int8"
        if o.fp8:
            # grouped-query shapes at head_dim 64/128 on the tensor cores, the
            # rest on the CUDA cores (the rule of paged_attention_decode_fp8)
            kernel = "decode_fp8_tc" if w.H // w.Hkv >= 2 and w.D in (64, 128) else "decode_fp8"
        if o.prefill:
            kernel = "append_tokens"
        ptok = SPLIT_PTOK.get(index) if o.split_tokens is None else (o.split_tokens or None)
        self.positions = w.lens.clone()
        self.lens_after = (w.lens + 1).clone()
        self.out = torch.empty_like(w.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = pa.workspace_for(w.q, w.block_table, ptok, num_kv_heads=w.Hkv, **kw) if ptok else None
        fused = not ptok and not o.unfused and not self.quant
        window = o.window or 0
        if window and not o.balanced:
            fused = False
        if self.quant:
            ptok = None
        groups = None
        shared = o.shared_prefix
        if shared is None:
            shared = index in SHARED_PREFIX and not o.balanced and not o.long_seq \
                and not o.prefill and not window
        if shared:
            if "shared_blocks" not in w.meta:
                raise SystemExit("--shared-prefix needs a workload with a shared prefix (workload 5)")
            groups = {"first": [0, w.B], "shared": [w.meta["shared_blocks"] * w.bs]}
            ptok = o.split_tokens or (SHARED_PREFIX_CODES if self.quant else SHARED_PREFIX).get(index, 4096)
            ws = pa.workspace_for(w.q, w.block_table, ptok, num_kv_heads=w.Hkv, **kw)
            fused = False
            kernel = {"fp8": "decode_prefix_fp8_tc", "int8": "decode_prefix_int8_tc"}.get(
                self.quant, "decode_prefix_tc")
        bws = None
        if o.balanced:
            ptok = None
            fused = not o.unfused
            kernel = kernel.replace("decode_gqa_umma", "decode_tc").replace("decode_gqa_tc", "decode_tc") + "_balanced"
            bws = pa.balanced_workspace_for(w.q, w.block_table, num_kv_heads=w.Hkv, **kw)
        prefill = None
        if o.prefill:
            # the padded batch of whole prompts, lengths = the workload's lengths
            T = int(w.lens.max())
            gen = torch.Generator(device=dev).manual_seed(99)
            prefill = {
                "k": torch.randn((w.B, T, w.Hkv, w.D), generator=gen, device=dev).to(w.dtype),
                "v": torch.randn((w.B, T, w.Hkv, w.D), generator=gen, device=dev).to(w.dtype),
                "start": torch.zeros(w.B, dtype=torch.int32, device=dev),
            }
            fused = False
        if ptok and not shared and not o.balanced and not self.quant and not o.prefill:
            which = pa.paged_attention_decode_kernel(shape, 0, ptok)
            kernel = {pa.PA_KERNEL_TCGEN05: "decode_gqa_umma", pa.PA_KERNEL_MMA_SYNC: "decode_gqa_tc"}.get(
                which, "decode_simt")
        self.kernel, self.fused, self.ptok, self.window = kernel, fused, ptok, window
        self.shared, self.groups, self.ws, self.bws, self.prefill = shared, groups, ws, bws, prefill
        self.main_calls, self.app_calls = self.make_calls(prepared=True)

    def make_calls(self, prepared: bool, t=None):
        """The step's C-ABI calls on the tensors `t` (default: the workload's
        own q, k_new, v_new, block_table, positions, lens_after and out).
        Prepared calls marshal their arguments once (a serving loop reuses
        its buffers every step) and are bound to the bench stream; graph
        capture needs calls on the capture stream."""
        pa, w, o, kw = self.pa, self.w, self.o, self.kw
        t = t or dict(q=w.q, k_new=w.k_new, v_new=w.v_new, block_table=w.block_table,
                      positions=self.positions, lens_after=self.lens_after, out=self.out)
        ptok, ws, bws, groups, window = self.ptok, self.ws, self.bws, self.groups, self.window
        kflat, vflat = w.k_flat(), w.v_flat()
        opt = dict(err_word=self.err, prepare=prepared,
                   stream=self.stream.cuda_stream if prepared else None)

        def bind(fn, *a, **k):
            c = fn(*a, **k, **opt)
            return c if prepared else (lambda: fn(*a, **k, **dict(opt, prepare=False)))

        if self.prefill is not None:
            p = self.prefill
            return [bind(pa.paged_kv_append_tokens, p["k"], p["v"], kflat, vflat, w.block_table, p["start"],
                         w.lens, **kw)], []
        if self.shared and self.quant:
            fn = (pa.paged_attention_decode_shared_prefix_fp8 if o.fp8
                  else pa.paged_attention_decode_shared_prefix_int8)
            app_fn = pa.paged_kv_append_fp8 if o.fp8 else pa.paged_kv_append_int8
            return ([bind(fn, t["out"], t["q"], kflat, vflat, w.scales, t["block_table"], t["lens_after"],
                          w.scale, ptok, ws, group_first=groups["first"], shared_tokens=groups["shared"],
                          num_kv_heads=w.Hkv, **kw)],
                    [bind(app_fn, t["k_new"], t["v_new"], kflat, vflat, w.scales, t["block_table"],
                          t["positions"], **kw)])
        if self.shared:
            return ([bind(pa.paged_attention_decode_shared_prefix, t["out"], t["q"], kflat, vflat,
                          t["block_table"], t["lens_after"], w.scale, ptok, ws, group_first=groups["first"],
                          shared_tokens=groups["shared"], num_kv_heads=w.Hkv, **kw)],
                    [bind(pa.paged_kv_append, t["k_new"], t["v_new"], kflat, vflat, t["block_table"],
                          t["positions"], **kw)])
        if self.quant:
            dec = pa.paged_attention_decode_fp8 if o.fp8 else pa.paged_attention_decode_int8
            app_fn = pa.paged_kv_append_fp8 if o.fp8 else pa.paged_kv_append_int8
            return ([bind(dec, t["out"], t["q"], kflat, vflat, w.scales, t["block_table"], t["lens_after"],
                          w.scale, num_kv_heads=w.Hkv, **kw)],
                    [bind(app_fn, t["k_new"], t["v_new"], kflat, vflat, w.scales, t["block_table"],
                          t["positions"], **kw)])
        app = [bind(pa.paged_kv_append, t["k_new"], t["v_new"], kflat, vflat, t["block_table"],
                    t["positions"], **kw)]
        if o.balanced:
            if self.fused:
                return [bind(pa.paged_attention_decode_balanced, t["out"], t["q"], kflat, vflat,
                             t["block_table"], w.scale, bws, positions=t["positions"], k_new=t["k_new"],
                             v_new=t["v_new"], window=window, num_kv_heads=w.Hkv, **kw)], []
            return [bind(pa.paged_attention_decode_balanced, t["out"], t["q"], kflat, vflat,
                         t["block_table"], w.scale, bws, seq_lens=t["lens_after"], window=window,
                         num_kv_heads=w.Hkv, **kw)], app
        if self.fused:
            return [bind(pa.paged_attention_decode_append, t["out"], t["q"], t["k_new"], t["v_new"], kflat,
                         vflat, t["block_table"], t["positions"], w.scale, num_kv_heads=w.Hkv, **kw)], []
        if window:
            return [bind(pa.paged_attention_decode_window, t["out"], t["q"], kflat, vflat, t["block_table"],
                         t["lens_after"], w.scale, window, num_kv_heads=w.Hkv, **kw)], app
        if ptok:
            return [bind(pa.paged_attention_decode_partial, t["q"], kflat, vflat, t["block_table"],
                         t["lens_after"], w.scale, ptok, ws, num_kv_heads=w.Hkv, **kw),
                    bind(pa.paged_attention_decode_reduce, t["out"], ws, t["lens_after"], ptok,
                         num_kv_heads=w.Hkv, max_blocks_per_seq=w.MB, **kw)], app
        return [bind(pa.paged_attention_decode, t["out"], t["q"], kflat, vflat, t["block_table"],
                     t["lens_after"], w.scale, num_kv_heads=w.Hkv, **kw)], app

    def append(self):
        for c in self.app_calls:
            c()

    def decode(self):
        for c in self.main_calls:
            c()

    def step(self):
        self.append()
        self.decode()

    @property
    def launches_per_step(self) -> int:
        return len(self.main_calls) + len(self.app_calls)

    def check_err(self, when: str) -> None:
        if int(self.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(self.err.item())} during {when}")

    def byte_counts(self):
        """(decode bytes, step bytes, bytes of the timed kernel launch(es))."""
        w = self.w
        if self.prefill is not None:
            b = prefill_bytes(w)
            return b, b, b
        dbytes = decode_bytes(w, self.lens_after, self.window)
        # the fused kernel also writes the appended rows into the pool
        kbytes = dbytes + (2 * w.B * w.Hkv * w.D * w.q.element_size() if self.fused else 0)
        return dbytes, dbytes + append_bytes(w), kbytes


def time_steps(plan: StepPlan, K: int, stream) -> float:
    """Milliseconds of K back-to-back steps, bracketed by events on `stream`
    after a synchronize (no events between the steps, so that programmatic
    dependent launch overlaps one step's tail with the next one's start)."""
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(K):
        plan.step()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


KERNEL_PASS = 64


def kernel_pass(plan: StepPlan, stream, n: int = KERNEL_PASS) -> list[float]:
    """Durations (us) of n launches of the step's timed kernel(s), each
    bracketed by its own pair of events on the launching stream, so that no
    launch overlaps a neighbour: the whole launch, ramp-up and drain
    included, as ncu's gpu__time_duration counts it.  One more launch runs
    first, right after a synchronize, and is discarded; the pass does not
    depend on the number of timed steps."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n + 1)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        plan.decode()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev[1:]]


def spread(samples: list[float]) -> dict:
    s = sorted(samples)
    return {"mean": round(statistics.fmean(s), 3), "median": round(statistics.median(s), 3),
            "p10": round(s[len(s) // 10], 3), "p90": round(s[(9 * len(s)) // 10], 3), "samples": len(s)}


DEFAULT_BLOCK_SIZE = {1: 16, 2: 16, 3: 16, 4: 16, 5: 32}


def workload_key(index, o, block_size=None) -> str:
    """The key profile summaries are filed under: workload, block size when
    it is not the workload's default, batch when given, cache variant, skew
    and pool offset."""
    key = f"w{index}"
    if block_size and block_size != DEFAULT_BLOCK_SIZE.get(index):
        key += f"_bs{block_size}"
    if o.batch:
        key += f"_b{o.batch}"
    if o.long_seq:
        key += f"_long{o.long_seq}"
    key += "_fp8" if o.fp8 else "_int8" if o.int8 else ""
    return key + (f"_pool_off{o.pool_offset}" if o.pool_offset else "")


# Configurations measured beside the headline step in the same run (one
# entry each): the five workloads of the report, the block-size sweep of the
# long tail and of the GQA layer, the GQA layer at batch 4, 16 and 64 (where
# the tcgen05 kernel runs: clusters of CTAs per unit, one CTA per unit, several
# units per CTA), the quantised caches, and a pool that is 16- but not 128-byte
# aligned.
PER_WORKLOAD = [
    ("w1", 1, None, {}),
    ("w2", 2, None, {}),
    ("w3_bs8", 3, 8, {}), ("w3_bs16", 3, 16, {}), ("w3_bs32", 3, 32, {}), ("w3_bs64", 3, 64, {}),
    ("w4_bs16", 4, 16, {}), ("w4_bs256", 4, 256, {}),
    ("w4_b4", 4, 16, {"batch": 4}), ("w4_b16", 4, 16, {"batch": 16}), ("w4_b64", 4, 16, {"batch": 64}),
    ("w5", 5, None, {}),
    ("w2_int8", 2, None, {"int8": True}), ("w4_int8", 4, 16, {"int8": True}),
    ("w5_int8", 5, None, {"int8": True}),
    ("w2_fp8", 2, None, {"fp8": True}), ("w4_fp8", 4, 16, {"fp8": True}),
    ("w5_fp8", 5, None, {"fp8": True}),
    ("w2_pool_off16", 2, None, {"pool_offset": 16}),
]


def measure_entry(pa, index, block_size, o, dev, stream, seconds: float, peaks: dict) -> dict:
    """One configuration: a few warm-up steps, about `seconds` of timed
    steps, then the kernel pass; the same figures as the headline line."""
    w = make_bench_workload(index, o, dev, block_size=block_size)
    plan = StepPlan(pa, w, index, o, dev, stream)
    for _ in range(5):
        plan.step()
    torch.cuda.synchronize()
    plan.check_err("warm-up")
    probe_ms = time_steps(plan, 10, stream) / 10
    K = int(min(20000, max(20, seconds * 1e3 / max(probe_ms, 1e-3))))
    ms_step = time_steps(plan, K, stream) / K
    samples = kernel_pass(plan, stream)
    torch.cuda.synchronize()
    plan.check_err("timing")
    dbytes, step_bytes, kbytes = plan.byte_counts()
    kd = spread(samples)
    achieved = kbytes / (kd["mean"] * 1e-6) / 1e9
    lens = [int(x) for x in w.lens]
    entry = {
        "workload": f"{w.name} (workload {index})", "batch": w.B, "num_heads": w.H,
        "num_kv_heads": w.Hkv, "head_dim": w.D, "block_size": w.bs, "cache": plan.quant or DTYPE_NAME[w.dtype],
        "seq_len_mean": round(sum(lens) / len(lens) + 1, 1), "steps": K,
        "us_per_layer_step": round(ms_step * 1e3, 3),
        "gbs": round(step_bytes / (ms_step * 1e-3) / 1e9, 1),
        "tokens_per_s": round(w.B / (ms_step * 1e-3), 1),
        "kernel": plan.kernel, "launches_per_step": plan.launches_per_step,
        "kernel_us": kd, "kernel_bytes": kbytes,
        "kernel_gbs": round(achieved, 1), "frac": round(achieved / peaks["hbm_gbs"], 4),
        "traffic": kernel_traffic(plan.kernel, workload_key(index, o, block_size), plan.fused),
        "step": ("fused append + decode" if plan.fused else
                 "append + shared-prefix split" if plan.shared else
                 "append + decode" if not plan.ptok else "append + split-KV pair"),
    }
    if plan.ptok:
        entry["split_kv_partition"] = plan.ptok
    if o.pool_offset:
        entry["pool_base_mod_128"] = w.pool.data_ptr() % 128
    if index == 5:
        lb = logical_kv_bytes(w, plan.lens_after)
        entry["logical_kv_gbs"] = round(lb / (ms_step * 1e-3) / 1e9, 1)
        entry["bytes_note"] = "unique bytes: shared blocks counted once"
    del plan, w
    torch.cuda.empty_cache()
    return entry


def per_workload_summary(entries: dict) -> dict:
    """Derived comparisons that the pages quote figures for (on their own
    hardware, as context): the cost of address translation at small blocks
    ("KV Cache and BlockManager" s2: 12% at block_size 8, 3.7% at 32 on an
    A100) and of a block start off the 128-byte boundary ("KV Block design"
    s3.7: about 15%)."""
    notes = {}
    t = {k: e["us_per_layer_step"] for k, e in entries.items() if "us_per_layer_step" in e}
    if "w3_bs8" in t and "w3_bs32" in t:
        notes["long_tail_bs8_over_bs32"] = round(t["w3_bs8"] / t["w3_bs32"] - 1, 4)
    if "w3_bs16" in t and "w3_bs64" in t:
        notes["long_tail_bs64_over_bs16"] = round(t["w3_bs64"] / t["w3_bs16"] - 1, 4)
    if "w2" in t and "w2_pool_off16" in t:
        notes["pool_16_not_128_aligned_over_aligned"] = round(t["w2_pool_off16"] / t["w2"] - 1, 4)
    return notes


def run_gpu(args) -> None:
    import pagedattention_decode_paged_gb300 as pa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pa.load()
    stream = torch.cuda.current_stream()
    o = step_options(unfused=args.unfused, window=args.window, balanced=args.balanced,
                     prefill=args.prefill, split_tokens=args.split_tokens,
                     shared_prefix=args.shared_prefix, int8=args.int8, fp8=args.fp8,
                     graph=args.graph, long_seq=args.long_seq, pool_offset=args.pool_offset,
                     batch=args.batch)

    # each rank holds its own replica of the workload (weak scaling)
    w = make_bench_workload(args.workload, o, dev, rank=rank, block_size=args.block_size,
                            batch=args.batch)
    plan = StepPlan(pa, w, args.workload, o, dev, stream)
    main_key = workload_key(args.workload, o, args.block_size)
    for _ in range(args.warmup):
        plan.step()
    torch.cuda.synchronize()
    plan.check_err("warm-up")

    K = args.steps
    graph = None
    if args.graph:
        # capture args.graph steps into one CUDA graph; the timed region
        # replays it K / args.graph times (K is rounded up to a multiple)
        K = -(-K // args.graph) * args.graph
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            plan.step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g_main, g_app = plan.make_calls(prepared=False)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.graph):
                for c in g_app + g_main:
                    c()
        graph.replay()
        torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_gpu_index(local_rank)) as clk:
        t0.record(stream)
        for _ in range(K // args.graph if graph is not None else 0):
            graph.replay()
        for _ in range(0 if graph is not None else K):
            plan.step()
        t1.record(stream)
        torch.cuda.synchronize()
        # the kernel's launch duration, outside the timed region: isolated
        # launches, each bracketed by its own events
        samples = kernel_pass(plan, stream)
    if dist:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    kd = spread(samples)
    decode_ms = kd["mean"] * 1e-3
    total_ms = max_over_ranks(total_ms, dist, dev)

    # end to end through the C ABI with host buffers: every step copies its
    # inputs (q, k_new, v_new, block_table, positions, lengths) from pinned
    # host memory, runs the step and reads the output back.  The inputs sit
    # in one pinned buffer and one device buffer per slot (one copy each
    # way), and two slots are double-buffered on two copy streams: the H2D
    # of step i+1 and the D2H of step i-1 overlap step i, the pipelining a
    # serving loop would use.  Graph and prefill runs copy in line.
    names = ("q", "k_new", "v_new", "block_table", "positions", "lens_after")
    src = dict(q=w.q, k_new=w.k_new, v_new=w.v_new, block_table=w.block_table,
               positions=plan.positions, lens_after=plan.lens_after)
    out = plan.out
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += -(-src[n].numel() * src[n].element_size() // 256) * 256
    h2d = sum(src[n].numel() * src[n].element_size() for n in names)
    d2h = out.numel() * out.element_size()
    host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n in names:
        nb = src[n].numel() * src[n].element_size()
        host_in[offs[n]:offs[n] + nb].copy_(src[n].contiguous().view(-1).view(torch.uint8).cpu())
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    Ke = max(3, min(K, 2000))
    pipelined = graph is None and plan.prefill is None
    if pipelined:
        dev_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        slots = []
        for buf in dev_in:
            t = {n: buf[offs[n]:offs[n] + src[n].numel() * src[n].element_size()]
                 .view(src[n].dtype).view(src[n].shape) for n in names}
            t["out"] = torch.empty_like(out)
            slots.append((buf, t, plan.make_calls(prepared=True, t=t)))
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        done = [torch.cuda.Event() for _ in range(2)]      # step in slot b finished
        loaded = [torch.cuda.Event() for _ in range(2)]    # inputs of slot b copied
        read = [torch.cuda.Event() for _ in range(2)]      # output of slot b copied back
        for b in range(2):
            done[b].record(stream)
            read[b].record(stream)

        def e2e_run(n):
            for i in range(n):
                b = i % 2
                buf, t, (m_calls, a_calls) = slots[b]
                h2d_stream.wait_event(done[b])
                with torch.cuda.stream(h2d_stream):
                    buf.copy_(host_in, non_blocking=True)
                loaded[b].record(h2d_stream)
                stream.wait_event(loaded[b])
                stream.wait_event(read[b])
                for c in a_calls + m_calls:
                    c()
                done[b].record(stream)
                d2h_stream.wait_event(done[b])
                with torch.cuda.stream(d2h_stream):
                    host_out[b].copy_(t["out"], non_blocking=True)
                read[b].record(d2h_stream)
            for b in range(2):
                stream.wait_event(read[b])
    else:
        host_views = {n: host_in[offs[n]:offs[n] + src[n].numel() * src[n].element_size()]
                      .view(src[n].dtype).view(src[n].shape) for n in names}

        def e2e_run(n):
            for _ in range(n):
                for name in names:
                    src[name].copy_(host_views[name], non_blocking=True)
                plan.step()
                host_out[0].copy_(out, non_blocking=True)

    e2e_run(3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if pipelined:
        h2d_stream.wait_event(e0)
    e2e_run(Ke)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    # the copies really landed: the last output read back equals the step's
    # (a prefill run writes no output)
    out_checked = (None if plan.prefill is not None else
                   bool(torch.equal(host_out[(Ke - 1) % 2 if pipelined else 0].to(dev), out)))
    plan.check_err("timing")

    dbytes, step_bytes, kbytes = plan.byte_counts()
    peaks = measured_peaks()
    achieved = kbytes / (decode_ms * 1e-3) / 1e9
    ms_step = total_ms / K
    value = job_throughput(world, step_bytes, ms_step)
    e2e_value = job_throughput(world, step_bytes, e2e_ms / Ke)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w.to("cpu"), plan.lens_after.cpu(), budget_s=args.cpu_seconds)

    line = None
    if rank == 0:
        cfg = describe(w, args.workload)
        cfg["split_kv_partition"] = plan.ptok
        cfg["l2"] = ("inputs larger than L2: %.0f MB of K/V read per step vs 129 MB L2; no flush"
                     % (dbytes / 1e6)) if dbytes > 2 * 129e6 else "L2 flushed: no (small workload)"
        cfg["parallelism"] = f"replicas x{world}"
        if o.pool_offset:
            cfg["pool_offset_bytes"] = o.pool_offset
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[w.dtype], "data": "synthetic (seeded N(0,1) Q/K/V, shuffled block ids)",
            "config": cfg,
            "tokens_per_s": round(world * w.B / (ms_step * 1e-3), 1),
            "us_per_layer_step": round(ms_step * 1e3, 3),
            "decode_us": kd["mean"], "decode_us_median": kd["median"],
            "decode_us_spread": kd,
            "decode_bytes": dbytes, "kernel_bytes": kbytes,
            "logical_kv_bytes": logical_kv_bytes(w, plan.lens_after),
            "decode_path": plan.kernel, "fused_append": plan.fused, "cuda_graph_steps": args.graph or None,
            "window": plan.window or None, "schedule": "balanced" if o.balanced else "one CTA per unit",
            "op": "prefill write" if plan.prefill is not None else "decode step",
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": kernel_traffic(plan.kernel, main_key, plan.fused),
                         "kernel": plan.kernel, "timed_launches": len(samples),
                         "kernel_timing": f"{len(samples)} isolated launches after the timed region, "
                                          "each bracketed by its own events on the launching "
                                          "stream; one launch after a synchronize discarded"},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": Ke,
                    "ms_per_step": round(e2e_ms / Ke, 6),
                    "copies": ("one H2D and one D2H per step, double-buffered on two copy streams"
                               if pipelined else "in line with the step"),
                    "output_read_back_matches": out_checked},
            "gpu_launches": K * plan.launches_per_step,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
    del plan, w, src, out
    if pipelined:
        del slots, dev_in
    torch.cuda.empty_cache()

    # the other configurations, one after another on the same GPU (rank 0 of
    # a one-GPU run only: every entry is a single-GPU measurement)
    if line is not None and world == 1 and not args.no_per_workload:
        peaks = measured_peaks()
        entries = {}
        # a plain run (no flag that reshapes the step) already measured its own entry
        plain = not (o.unfused or o.window or o.balanced or o.prefill or o.graph or o.long_seq or
                     o.split_tokens is not None or o.shared_prefix is not None or args.batch)
        with ClockSampler(local_gpu_index(local_rank)) as pclk:
            for key, index, bs, over in PER_WORKLOAD:
                ovr = step_options(**over)
                if plain and workload_key(index, ovr, bs) == main_key:
                    # the headline line itself: its figures, not a second run
                    entries[key] = {"headline": True, "us_per_layer_step": line["us_per_layer_step"],
                                    "gbs": line["value"], "kernel": line["decode_path"],
                                    "kernel_us": line["decode_us_spread"],
                                    "frac": line["roofline"]["frac"], "traffic": line["roofline"]["traffic"]}
                    continue
                try:
                    entries[key] = measure_entry(pa, index, bs, ovr, dev, stream,
                                                 args.per_workload_seconds, peaks)
                except (RuntimeError, torch.cuda.OutOfMemoryError) as exc:   # report, keep going
                    entries[key] = {"error": str(exc).splitlines()[0][:200]}
        line["per_workload"] = {
            "entries": entries,
            "notes": per_workload_summary(entries),
            "clocks": pclk.summary(),
            "timing": f"each entry: 5 warm-up steps, about {args.per_workload_seconds} s of back-to-back "
                      f"steps, then {KERNEL_PASS} isolated launches of its kernel(s); not part of the "
                      "headline's timed region"}
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# the CPU oracle, timed on the host cores
# ---------------------------------------------------------------------------

def _oracle_sample(w, lens_after, seqs, threads=None):
    """Oracle decode of the sequences `seqs` (all heads) on `threads` host
    threads (default: every core); returns bytes read and seconds."""
    threads = threads or os.cpu_count() or 1
    import oracle
    sub = torch.tensor(seqs, dtype=torch.long)
    q = w.q.index_select(0, sub).contiguous()
    table = w.block_table.index_select(0, sub).contiguous()
    lens = lens_after.index_select(0, sub).contiguous()
    flat = w.pool.view(-1)
    t = time.perf_counter()
    if getattr(w, "scales", None) is not None and w.pool.dtype == torch.uint8:
        oracle.attention_decode_fp8(q, flat, flat[w.v_offset:], w.scales, table, lens, w.scale,
                                    num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride,
                                    num_blocks=w.NB, threads=threads)
    elif getattr(w, "scales", None) is not None:
        oracle.attention_decode_i8(q, flat, flat[w.v_offset:], w.scales, table, lens, w.scale,
                                   num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride,
                                   num_blocks=w.NB, threads=threads)
    else:
        oracle.attention_decode(q, flat, flat[w.v_offset:], table, lens, w.scale,
                                num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride,
                                num_blocks=w.NB, threads=threads)
    dt = time.perf_counter() - t
    s = w.pool.element_size()
    sq = w.q.element_size()
    nbytes = sum(2 * w.Hkv * w.D * s * int(L) + 4 * -(-int(L) // w.bs) + 4 + 2 * w.H * w.D * sq
                 for L in lens)
    return nbytes, dt


def cpu_baseline(w, lens_after, budget_s=10.0) -> dict:
    def run(threads, budget):
        done_bytes, done_s, seqs = 0, 0.0, 0
        while done_s < budget:
            nbytes, dt = _oracle_sample(w, lens_after, [seqs % w.B], threads)
            done_bytes += nbytes
            done_s += dt
            seqs += 1
        return done_bytes / done_s / 1e9, seqs, done_s

    value, seqs, done_s = run(os.cpu_count() or 1, budget_s)
    value1, seqs1, done1 = run(1, budget_s / 4)
    return {"value": round(value, 4), "unit": UNIT,
            "cores": os.cpu_count() or 1, "kind": "oracle",
            "value_1_thread": round(value1, 4),
            "sample": f"{seqs} sequence decodes (all {w.H} heads each) of the same workload, "
                      f"fp64 C oracle with OpenMP over (sequence, kv head), {done_s:.1f} s; "
                      f"one thread: {seqs1} decodes, {done1:.1f} s"}


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    w = workloads.make_workload(args.workload, block_size=args.block_size, device="cpu",
                                batch=args.batch)
    if args.long_seq:
        w = workloads.with_long_sequence(w, args.long_seq)
    if args.int8:
        w = workloads.to_int8(w)
    if args.fp8:
        w = workloads.to_fp8(w)
    lens_after = w.lens + 1
    for i in range(args.warmup):
        _oracle_sample(w, lens_after, [i % w.B])
    total_bytes, total_s = 0, 0.0
    t_start = time.perf_counter()
    for i in range(args.steps):
        nbytes, dt = _oracle_sample(w, lens_after, [i % w.B])
        total_bytes += nbytes
        total_s += dt
    wall = time.perf_counter() - t_start
    value = total_bytes / total_s / 1e9
    cfg = describe(w, args.workload)
    cfg["parallelism"] = "host cores"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[w.dtype],
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled block ids)", "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": os.cpu_count() or 1,
                         "kind": "oracle",
                         "sample": "each step: the fp64 C oracle's decode of one sequence "
                                   f"(all {w.H} heads) of the workload, cycling through the batch"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--block-size", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (workloads 2-4)")
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window decode over the last W tokens (append + window decode)")
    ap.add_argument("--prefill", action="store_true",
                    help="time the prompt write of every sequence's full length instead")
    ap.add_argument("--graph", type=int, default=0,
                    help="capture this many steps into one CUDA graph and replay it")
    ap.add_argument("--long-seq", type=int, default=0,
                    help="replace the last sequence by one of this many tokens (skewed batch)")
    ap.add_argument("--shared-prefix", action=argparse.BooleanOptionalAction, default=None,
                    help="paged_attention_decode_shared_prefix (shared blocks read once per "
                         "group; the default for workload 5)")
    ap.add_argument("--fp8", action="store_true",
                    help="fp8 (E4M3) cache with per-block scales (paged_kv_append_fp8 + "
                         "paged_attention_decode_fp8)")
    ap.add_argument("--int8", action="store_true",
                    help="int8 cache with per-block scales (paged_kv_append_int8 + "
                         "paged_attention_decode_int8)")
    ap.add_argument("--balanced", action="store_true",
                    help="time paged_attention_decode_balanced (persistent load-balanced grid)")
    ap.add_argument("--unfused", action="store_true",
                    help="time paged_kv_append and paged_attention_decode as two launches")
    ap.add_argument("--split-tokens", type=int, default=None,
                    help="split-KV partition size (0: single-pass decode); default per workload")
    ap.add_argument("--pool-offset", type=int, default=0,
                    help="move the pool this many bytes (a multiple of 16) off its 512-byte aligned "
                         "allocation: the cost of block starts off the 128-byte boundary")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the other configurations measured after the headline")
    ap.add_argument("--per-workload-seconds", type=float, default=0.3,
                    help="timed seconds per configuration of the per_workload object")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
