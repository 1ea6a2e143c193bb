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

    # each rank holds its own replica of the workload (weak scaling)
    w = workloads.make_workload(args.workload, block_size=args.block_size, device=dev,
                                seed=replica_seed(args.workload, rank), batch=args.batch)
    workload_key = f"w{args.workload}" + (f"_bs{args.block_size}" if args.block_size else "")
    if args.long_seq:
        w = workloads.with_long_sequence(w, args.long_seq, seed=7 + rank, device=dev)
        workload_key += f"_long{args.long_seq}"
    if args.int8 and args.fp8:
        raise SystemExit("--int8 and --fp8 are two cache formats: pick one")
    if args.int8 or args.fp8:
        if args.prefill or args.window or args.balanced or args.graph:
            raise SystemExit("--int8 / --fp8 time the quantising append + decode pair only")
        w = (workloads.to_fp8(w, seed=19 + rank) if args.fp8 else workloads.to_int8(w, seed=17 + rank)).to(dev)
        workload_key += "_fp8" if args.fp8 else "_int8"
    kw = dict(block_size=w.bs, num_blocks=w.NB, block_stride=w.block_stride)
    shape = pa.make_shape(batch=w.B, num_heads=w.H, num_kv_heads=w.Hkv, head_dim=w.D,
                          block_size=w.bs, max_blocks_per_seq=w.MB, num_blocks=w.NB,
                          block_stride=w.block_stride, dtype=w.dtype)
    path = pa.paged_attention_decode_path(shape)
    kernel = "decode_gqa_tc" if path == pa.PA_PATH_TENSOR_GQA else "decode_simt"
    if args.int8:
        # grouped-query shapes with 16-bit queries and head_dim 64/128 run on
        # the tensor cores (the rule of paged_attention_decode_int8)
        tc8 = w.H // w.Hkv >= 2 and w.D in (64, 128) and w.dtype in (torch.float16, torch.bfloat16)
        kernel = "decode_int8_tc" if tc8 else "decode_int8"
    if args.fp8:
        # grouped-query shapes at head_dim 64/128 on the tensor cores, the
        # rest on the CUDA cores (the rule of paged_attention_decode_fp8)
        kernel = "decode_fp8_tc" if w.H // w.Hkv >= 2 and w.D in (64, 128) else "decode_fp8"
    if args.prefill:
        kernel = "append_tokens"
    ptok = SPLIT_PTOK.get(args.workload) if args.split_tokens is None else (args.split_tokens or None)
    positions = w.lens.clone()
    lens_after = (w.lens + 1).clone()
    out = torch.empty_like(w.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = (pa.workspace_for(w.q, w.block_table, ptok, num_kv_heads=w.Hkv, **kw)
          if ptok else None)
    stream = torch.cuda.current_stream()

    quant = args.int8 or args.fp8
    fused = not ptok and not args.unfused and not quant

    window = args.window or 0
    balanced = args.balanced
    if window and not balanced:
        fused = False
    bws = None
    if quant:
        ptok = None
    groups = None
    if args.shared_prefix is None:
        args.shared_prefix = args.workload in SHARED_PREFIX and not args.balanced \
            and not args.long_seq and not args.prefill and not window
    if args.shared_prefix:
        if "shared_blocks" not in w.meta:
            raise SystemExit("--shared-prefix needs a workload with a shared prefix (workload 5)")
        groups = {"first": [0, w.B], "shared": [w.meta["shared_blocks"] * w.bs]}
        ptok = args.split_tokens or (SHARED_PREFIX_CODES if quant else SHARED_PREFIX).get(args.workload, 4096)
        ws = pa.workspace_for(w.q, w.block_table, ptok, num_kv_heads=w.Hkv, **kw)
        fused = False
        kernel = "decode_prefix_fp8_tc" if args.fp8 else "decode_prefix_int8_tc" if args.int8 else "decode_prefix_tc"
    if balanced:
        ptok = None
        fused = not args.unfused
        kernel = kernel.replace("decode_gqa_tc", "decode_tc") + "_balanced"
        bws = pa.balanced_workspace_for(w.q, w.block_table, num_kv_heads=w.Hkv, **kw)
    prefill = None
    if args.prefill:
        # the padded batch of whole prompts, lengths = the workload's lengths
        T = int(w.lens.max())
        gen = torch.Generator(device=dev).manual_seed(99)
        prefill = {
            "k": torch.randn((w.B, T, w.Hkv, w.D), generator=gen, device=dev).to(w.dtype),
            "v": torch.randn((w.B, T, w.Hkv, w.D), generator=gen, device=dev).to(w.dtype),
            "start": torch.zeros(w.B, dtype=torch.int32, device=dev),
        }
        fused = False
    kflat, vflat = w.k_flat(), w.v_flat()

    def make_calls(prepared: bool, t=None):
        """The step's C-ABI calls on the tensors `t` (default: the workload's
        own q, k_new, v_new, block_table, positions, lens_after and out).
        Prepared calls marshal their arguments once (a serving loop reuses
        its buffers every step) and are bound to the bench stream; graph
        capture needs calls on the capture stream."""
        t = t or dict(q=w.q, k_new=w.k_new, v_new=w.v_new, block_table=w.block_table,
                      positions=positions, lens_after=lens_after, out=out)
        o = dict(err_word=err, prepare=prepared,
                 stream=stream.cuda_stream if prepared else None)

        def bind(fn, *a, **k):
            c = fn(*a, **k, **o)
            return c if prepared else (lambda: fn(*a, **k, **dict(o, prepare=False)))

        calls = []
        if prefill is not None:
            calls.append(bind(pa.paged_kv_append_tokens, prefill["k"], prefill["v"], kflat, vflat,
                              w.block_table, prefill["start"], w.lens, **kw))
            return calls, []
        if args.shared_prefix and quant:
            fn = (pa.paged_attention_decode_shared_prefix_fp8 if args.fp8
                  else pa.paged_attention_decode_shared_prefix_int8)
            calls.append(bind(fn, t["out"], t["q"], kflat, vflat, w.scales, t["block_table"], t["lens_after"],
                              w.scale, ptok, ws, group_first=groups["first"], shared_tokens=groups["shared"],
                              num_kv_heads=w.Hkv, **kw))
            app_fn = pa.paged_kv_append_fp8 if args.fp8 else pa.paged_kv_append_int8
            return calls, [bind(app_fn, t["k_new"], t["v_new"], kflat, vflat, w.scales, t["block_table"],
                                t["positions"], **kw)]
        if args.shared_prefix:
            calls.append(bind(pa.paged_attention_decode_shared_prefix, t["out"], t["q"], kflat, vflat,
                              t["block_table"], t["lens_after"], w.scale, ptok, ws,
                              group_first=groups["first"], shared_tokens=groups["shared"],
                              num_kv_heads=w.Hkv, **kw))
            return calls, [bind(pa.paged_kv_append, t["k_new"], t["v_new"], kflat, vflat, t["block_table"],
                                t["positions"], **kw)]
        if args.fp8:
            calls.append(bind(pa.paged_attention_decode_fp8, t["out"], t["q"], kflat, vflat, w.scales,
                              t["block_table"], t["lens_after"], w.scale, num_kv_heads=w.Hkv, **kw))
            return calls, [bind(pa.paged_kv_append_fp8, t["k_new"], t["v_new"], kflat, vflat, w.scales,
                                t["block_table"], t["positions"], **kw)]
        if args.int8:
            calls.append(bind(pa.paged_attention_decode_int8, t["out"], t["q"], kflat, vflat, w.scales,
                              t["block_table"], t["lens_after"], w.scale, num_kv_heads=w.Hkv, **kw))
            return calls, [bind(pa.paged_kv_append_int8, t["k_new"], t["v_new"], kflat, vflat, w.scales,
                                t["block_table"], t["positions"], **kw)]
        if balanced:
            if fused:
                calls.append(bind(pa.paged_attention_decode_balanced, t["out"], t["q"], kflat, vflat,
                                  t["block_table"], w.scale, bws, positions=t["positions"], k_new=t["k_new"],
                                  v_new=t["v_new"], window=window, num_kv_heads=w.Hkv, **kw))
                return calls, []
            calls.append(bind(pa.paged_attention_decode_balanced, t["out"], t["q"], kflat, vflat,
                              t["block_table"], w.scale, bws, seq_lens=t["lens_after"], window=window,
                              num_kv_heads=w.Hkv, **kw))
            return calls, [bind(pa.paged_kv_append, t["k_new"], t["v_new"], kflat, vflat, t["block_table"],
                                t["positions"], **kw)]
        if fused:
            calls.append(bind(pa.paged_attention_decode_append, t["out"], t["q"], t["k_new"], t["v_new"], kflat,
                              vflat, t["block_table"], t["positions"], w.scale, num_kv_heads=w.Hkv, **kw))
            return calls, []
        app = [bind(pa.paged_kv_append, t["k_new"], t["v_new"], kflat, vflat, t["block_table"], t["positions"],
                    **kw)]
        if window:
            calls.append(bind(pa.paged_attention_decode_window, t["out"], t["q"], kflat, vflat,
                              t["block_table"], t["lens_after"], w.scale, window, num_kv_heads=w.Hkv, **kw))
        elif ptok:
            calls.append(bind(pa.paged_attention_decode_partial, t["q"], kflat, vflat, t["block_table"],
                              t["lens_after"], w.scale, ptok, ws, num_kv_heads=w.Hkv, **kw))
            calls.append(bind(pa.paged_attention_decode_reduce, t["out"], ws, t["lens_after"], ptok,
                              num_kv_heads=w.Hkv, max_blocks_per_seq=w.MB, **kw))
        else:
            calls.append(bind(pa.paged_attention_decode, t["out"], t["q"], kflat, vflat, t["block_table"],
                              t["lens_after"], w.scale, num_kv_heads=w.Hkv, **kw))
        return calls, app

    main_calls, app_calls = make_calls(prepared=True)

    def append():
        for c in app_calls:
            c()

    def decode():
        for c in main_calls:
            c()

    def step():
        append()
        decode()

    launches_per_step = len(main_calls) + len(app_calls)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during warm-up")

    K = args.steps
    graph = None
    if args.graph:
        # capture args.graph steps into one CUDA graph; the timed region
        # replays it K / args.graph times (K is rounded up to a multiple)
        K = -(-K // args.graph) * args.graph
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g_main, g_app = make_calls(prepared=False)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.graph):
                for c in g_app + g_main:
                    c()
        graph.replay()
        torch.cuda.synchronize()
    # kernel durations are sampled live on every EVERY-th step of the timed
    # region (events bracket those launches on the launching stream); the
    # other steps run back to back, so that events do not sit between kernels
    EVERY = 16
    sampled = [] if graph is not None else list(range(0, K, EVERY))
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for i in sampled}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_gpu_index(local_rank)) as clk:
        t0.record(stream)
        for i in range(K // args.graph if graph is not None else 0):
            graph.replay()
        for i in range(0 if graph is not None else K):
            e = ev.get(i)
            if e is None:
                step()
                continue
            e[0].record(stream)
            append()
            e[1].record(stream)
            decode()
            e[2].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    if graph is not None:
        # no events inside the graph: the step time bounds the kernel time
        decode_ms = append_ms = total_ms / K
    else:
        decode_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev.values())
        append_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev.values())
    # spread of the bracketed decode launches: p10 / median / p90 (us)
    dsamples = sorted(e[1].elapsed_time(e[2]) * 1e3 for e in ev.values()) if graph is None else []
    dspread = ({"p10": round(dsamples[len(dsamples) // 10], 3),
                "median": round(statistics.median(dsamples), 3),
                "p90": round(dsamples[(9 * len(dsamples)) // 10], 3), "samples": len(dsamples)}
               if dsamples else None)
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
               positions=positions, lens_after=lens_after)
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
    pipelined = graph is None and prefill is None
    if pipelined:
        dev_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        slots = []
        for buf in dev_in:
            t = {n: buf[offs[n]:offs[n] + src[n].numel() * src[n].element_size()]
                 .view(src[n].dtype).view(src[n].shape) for n in names}
            t["out"] = torch.empty_like(out)
            slots.append((buf, t, make_calls(prepared=True, t=t)))
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
                step()
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
    out_checked = (None if prefill is not None else
                   bool(torch.equal(host_out[(Ke - 1) % 2 if pipelined else 0].to(dev), out)))
    if int(err.item()) != 0:
        raise RuntimeError(f"device error bits {int(err.item())} during timing")

    if prefill is not None:
        dbytes = step_bytes = kbytes = prefill_bytes(w)
    else:
        dbytes = decode_bytes(w, lens_after, window)
        step_bytes = dbytes + append_bytes(w)
        # the fused kernel also writes the appended rows into the pool
        kbytes = dbytes + (2 * w.B * w.Hkv * w.D * w.q.element_size() if fused else 0)
    peaks = measured_peaks()
    achieved = kbytes / (decode_ms * 1e-3) / 1e9
    ms_step = total_ms / K
    value = job_throughput(world, step_bytes, ms_step)
    e2e_value = job_throughput(world, step_bytes, e2e_ms / Ke)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w.to("cpu"), lens_after.cpu(), budget_s=args.cpu_seconds)

    if rank == 0:
        cfg = describe(w, args.workload)
        cfg["split_kv_partition"] = ptok
        cfg["l2"] = ("inputs larger than L2: %.0f MB of K/V read per step vs 129 MB L2; no flush"
                     % (dbytes / 1e6)) if dbytes > 2 * 129e6 else "L2 flushed: no (small workload)"
        cfg["parallelism"] = f"replicas x{world}"
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[w.dtype], "data": "synthetic (seeded N(0,1) Q/K/V, shuffled block ids)",
            "config": cfg,
            "tokens_per_s": round(world * w.B / (ms_step * 1e-3), 1),
            "us_per_layer_step": round(ms_step * 1e3, 3),
            "decode_us": round(decode_ms * 1e3, 3), "append_us": round(append_ms * 1e3, 3),
            "decode_us_spread": dspread,
            "decode_bytes": dbytes, "kernel_bytes": kbytes,
            "logical_kv_bytes": logical_kv_bytes(w, lens_after),
            "decode_path": kernel, "fused_append": fused, "cuda_graph_steps": args.graph or None,
            "window": window or None, "schedule": "balanced" if balanced else "one CTA per unit",
            "op": "prefill write" if prefill is not None else "decode step",
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": kernel_traffic(kernel, workload_key, fused),
                         "kernel": kernel, "timed_launches": len(sampled),
                         "kernel_timing": "graph step" if graph is not None else "events"},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": Ke,
                    "ms_per_step": round(e2e_ms / Ke, 6),
                    "copies": ("one H2D and one D2H per step, double-buffered on two copy streams"
                               if pipelined else "in line with the step"),
                    "output_read_back_matches": out_checked},
            "gpu_launches": K * launches_per_step,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
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
