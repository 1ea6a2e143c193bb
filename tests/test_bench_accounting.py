"""The host-side parts of bench.py, on CPU: the algorithmic byte counts
that the roofline fraction divides by (valid rows only, shared blocks once,
the window's rows, the scales of a quantised cache), the lookup of DRAM
traffic from the committed ncu summaries, which must refuse a summary whose
kernel sources have changed, and the JSON line of the reference arm (the
oracle on the host cores), which runs without a GPU."""
import json
import os
import subprocess
import sys

import pytest

import bench
import workloads


def _tiny(lens, bs=4, H=4, Hkv=2, D=16):
    return workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=D, bs=bs, dtype=workloads.torch.float16,
                                  lens=lens, seed=1, poison=False)


def test_decode_bytes_counts_valid_rows_tables_and_q_out():
    w = _tiny([5, 0, 9])
    lens = [5, 0, 9]
    s = 2   # fp16
    kv = 2 * w.Hkv * w.D * s * sum(lens)
    tables = sum(-(-L // w.bs) for L in lens)
    want = kv + 4 * tables + 4 * w.B + 2 * w.B * w.H * w.D * s
    assert bench.decode_bytes(w, lens) == want
    assert bench.logical_kv_bytes(w, lens) == kv


def test_decode_bytes_window_counts_only_the_last_rows():
    w = _tiny([9, 3])
    # window 4 over lengths 9 and 3: rows 5..8 of sequence 0 (blocks 1 and 2),
    # rows 0..2 of sequence 1 (block 0)
    s = 2
    rows = 4 + 3
    tables = 2 + 1
    want = 2 * w.Hkv * w.D * s * rows + 4 * tables + 4 * w.B + 2 * w.B * w.H * w.D * s
    assert bench.decode_bytes(w, [9, 3], window=4) == want


def test_decode_bytes_reads_shared_blocks_once():
    w = _tiny([8, 8])
    w.block_table[1, :2] = w.block_table[0, :2]   # both sequences share their two blocks
    s = 2
    want = 2 * w.Hkv * w.D * s * 8 + 4 * 4 + 4 * w.B + 2 * w.B * w.H * w.D * s
    assert bench.decode_bytes(w, [8, 8]) == want


def test_quantised_cache_counts_one_byte_per_element_and_the_scales():
    for conv in (workloads.to_int8, workloads.to_fp8):
        w = conv(_tiny([5, 9]))
        lens = [5, 9]
        blocks = sum(-(-L // w.bs) for L in lens)
        kv = 2 * w.Hkv * w.D * 1 * sum(lens)
        want = kv + 2 * 4 * w.Hkv * blocks + 4 * blocks + 4 * w.B + 2 * w.B * w.H * w.D * 2
        assert bench.decode_bytes(w, lens) == want
        # the append reads the 16-bit rows and their block's two scales and
        # writes one byte per element
        assert bench.append_bytes(w) == 2 * w.B * w.Hkv * w.D * (2 + 1) + 2 * 4 * w.B * w.Hkv + 8 * w.B


def test_quantised_cache_reads_shared_blocks_and_their_scales_once():
    """The shared-beam figures over an int8 or fp8 cache divide by unique
    bytes: a block named by several rows adds its codes and its K and V
    scales once."""
    for conv in (workloads.to_int8, workloads.to_fp8):
        w16 = _tiny([8, 8, 5])
        w16.block_table[1, :2] = w16.block_table[0, :2]   # rows 0 and 1 share their two blocks
        w = conv(w16)
        unique_rows = 8 + 5
        unique_blocks = 2 + 2
        tables = 2 + 2 + 2
        want = (2 * w.Hkv * w.D * unique_rows + 2 * 4 * w.Hkv * unique_blocks + 4 * tables + 4 * w.B
                + 2 * w.B * w.H * w.D * 2)
        assert bench.decode_bytes(w, [8, 8, 5]) == want
        assert bench.logical_kv_bytes(w, [8, 8, 5]) == 2 * w.Hkv * w.D * (8 + 8 + 5)


def test_kernel_traffic_refuses_a_stale_summary(tmp_path, monkeypatch):
    digest = bench.source_digest(bench.KERNEL_SOURCES["decode_simt"])
    good = tmp_path / "decode_simt__tiny_w9_fused.md"
    good.write_text(f"source_sha256: {digest}\ndram_bytes_per_launch: 1234\n")
    stale = tmp_path / "decode_simt__tiny_w8_fused.md"
    stale.write_text("source_sha256: " + "0" * 64 + "\ndram_bytes_per_launch: 999\n")
    monkeypatch.setattr(bench, "PROFILE_DIR", tmp_path)
    assert bench.kernel_traffic("decode_simt", "w9", fused=True) == 1234
    assert bench.kernel_traffic("decode_simt", "w9", fused=False) is None   # no unfused summary
    assert bench.kernel_traffic("decode_simt", "w8", fused=True) is None    # sources changed since


def test_every_profiled_kernel_has_a_source():
    """Each kernel bench.py can name maps to a source file whose digest can
    be taken, and every committed summary names a known kernel."""
    for name, src in bench.KERNEL_SOURCES.items():
        assert (bench.ROOT / "pagedattention_decode_paged_gb300" / "csrc" / src).exists(), name
        assert len(bench.source_digest(src)) == 64
    for f in bench.PROFILE_DIR.glob("*.md"):
        kernel = f.name.split("__")[0]
        assert kernel == "launches" or kernel in bench.KERNEL_SOURCES, f.name


@pytest.mark.parametrize("extra", [[], ["--int8"], ["--fp8"]])
def test_reference_arm_prints_the_contract_line(extra):
    cmd = [sys.executable, str(bench.ROOT / "bench.py"), "--impl", "reference", "--workload", "1",
           "--steps", "3", "--warmup", "3", *extra]
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=bench.ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 3, 3)
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("tiny")


def test_workload_keys_and_per_workload_table():
    """Profile keys drop the default block size and name the cache variant;
    the per_workload table has unique labels, covers workloads 1-5, the
    long tail at block sizes 8/16/32/64 and the GQA layer at 16/256, and each
    label's key is distinct (no configuration measured twice); the GQA layer
    also runs at batch 4, 16 and 64."""
    o = bench.step_options()
    assert bench.workload_key(4, o, 16) == bench.workload_key(4, o) == "w4"
    assert bench.workload_key(4, o, 256) == "w4_bs256"
    assert bench.workload_key(3, bench.step_options(int8=True), 8) == "w3_bs8_int8"
    assert bench.workload_key(2, bench.step_options(pool_offset=16)) == "w2_pool_off16"
    assert bench.workload_key(4, bench.step_options(batch=64), 16) == "w4_b64"
    labels = [e[0] for e in bench.PER_WORKLOAD]
    assert len(labels) == len(set(labels))
    keys = [bench.workload_key(i, bench.step_options(**over), bs) for _, i, bs, over in bench.PER_WORKLOAD]
    assert len(keys) == len(set(keys))
    assert {i for _, i, _, _ in bench.PER_WORKLOAD} == {1, 2, 3, 4, 5}
    assert {bs for _, i, bs, _ in bench.PER_WORKLOAD if i == 3} == {8, 16, 32, 64}
    assert {bs for _, i, bs, over in bench.PER_WORKLOAD if i == 4 and not over} == {16, 256}
    assert {over.get("batch") for _, i, _, over in bench.PER_WORKLOAD if i == 4} >= {None, 4, 16, 64}


def test_per_workload_notes():
    e = {"w3_bs8": {"us_per_layer_step": 112.0}, "w3_bs32": {"us_per_layer_step": 100.0},
         "w3_bs16": {"us_per_layer_step": 105.0}, "w3_bs64": {"us_per_layer_step": 110.25},
         "w2": {"us_per_layer_step": 80.0}, "w2_pool_off16": {"us_per_layer_step": 84.0},
         "w4_bs16": {"error": "x"}}
    n = bench.per_workload_summary(e)
    assert n == {"long_tail_bs8_over_bs32": 0.12, "long_tail_bs64_over_bs16": 0.05,
                 "pool_16_not_128_aligned_over_aligned": 0.05}
    assert bench.per_workload_summary({}) == {}


def test_spread_of_kernel_samples():
    s = bench.spread([float(x) for x in range(1, 65)])
    assert s["samples"] == 64 and s["mean"] == 32.5 and s["median"] == 32.5
    assert s["p10"] == 7.0 and s["p90"] == 58.0
