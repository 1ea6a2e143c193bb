"""paged_attention_decode_split_static: split-KV decode for callers that
cannot allocate device memory.

Some callers of this library are not allowed to allocate: code running inside
a memory pool or allocator callback, a plugin that a host framework hands only
its input and output buffers, or work being captured into a CUDA graph where
an allocation would break the capture.  For them the library keeps the
split-KV partial results in a fixed scratch array of its own.  These tests
call that entry point through the C ABI, twice in a row on different shapes
(the array keeps whatever the previous call left), and compare each result
with the CPU oracle and with paged_attention_decode on the same inputs; they
also probe the size limit at the exact shape where the workspace stops
fitting.

This file is named so that pytest collects it last.
"""
import ctypes
import re
from pathlib import Path

import pytest
import torch

import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu

HEADER = Path(__file__).resolve().parent.parent / "include" / "pagedattn.h"


def scratch_bytes() -> int:
    """PA_STATIC_SCRATCH_BYTES as include/pagedattn.h defines it."""
    m = re.search(r"#define\s+PA_STATIC_SCRATCH_BYTES\s+\((\d+)u?\s*<<\s*(\d+)\)", HEADER.read_text())
    assert m, "PA_STATIC_SCRATCH_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


def _entry():
    lib = pa.load()
    f = lib.paged_attention_decode_split_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(pa.Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    return f


def _call(f, g, lens, ptok, out, err):
    shape = hz.shape_of(g)
    return f(ctypes.byref(shape), out.data_ptr(), g.q.data_ptr(), g.k_flat().data_ptr(),
             g.v_flat().data_ptr(), g.block_table.data_ptr(), lens.data_ptr(), g.scale, ptok,
             err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _check_against_both(f, w, ptok):
    """One static call on w (no append; attention over w.lens) against the
    oracle and against paged_attention_decode, each with its own err word."""
    g = w.to("cuda")
    err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_gpu = hz.gpu_decode(g, g.lens, err_ref)
    torch.cuda.synchronize()
    assert int(err_ref.item()) == 0, f"paged_attention_decode raised device bits {int(err_ref.item())}"
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(g.q, float("nan"))
    st = _call(f, g, g.lens, ptok, out, err)
    assert st == pa.PA_OK, pa.status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"split_static raised device bits {int(err.item())}"
    ref, e = hz.oracle_decode(w, w.pool, w.lens)
    assert not e.any()
    hz.assert_close(out, ref, w.dtype, f"{w.name} split_static vs oracle")
    atol, rtol = hz.TOL[w.dtype]
    diff = (out.float() - ref_gpu.float()).abs()
    assert bool((diff <= atol + rtol * ref_gpu.float().abs()).all()), float(diff.max())


def test_static_scratch_split_matches_oracle_twice_in_a_row(cuda_ok):
    f = _entry()
    limit = scratch_bytes()
    cases = [
        (workloads.make_workload(5, max_len=6000, poison=True), 1024),        # MHA, shared prefix
        (workloads.make_workload(4, batch=6, max_len=900, poison=True), 256),  # GQA, tensor cores
    ]
    for w, ptok in cases:
        assert 0 < pa.paged_attention_partial_workspace(hz.shape_of(w), ptok) <= limit
        _check_against_both(f, w, ptok)


def _boundary_workload(mb: int):
    """One sequence of 40 tokens whose table row holds mb entries (the rest
    -1), so that the split-KV workspace grows with mb at 16-token partitions."""
    w = workloads.make_generic(B=1, H=4, Hkv=4, D=128, bs=16, dtype=torch.bfloat16,
                               lens=[40], seed=5, poison=True)
    assert mb >= w.MB
    table = torch.full((1, mb), -1, dtype=torch.int32)
    table[0, :w.MB] = w.block_table[0]
    w.block_table = table
    w.MB = mb
    return w


def test_static_scratch_size_limit_is_exact(cuda_ok):
    f = _entry()
    limit = scratch_bytes()
    ptok = 16
    # largest row length whose workspace still fits (workspace grows with it)
    ws = lambda mb: pa.paged_attention_partial_workspace(hz.shape_of(_boundary_workload(mb)), ptok)  # noqa: E731
    lo, hi = 16, 1 << 16             # rows of at least 16 entries hold the sequence's 3 blocks
    assert ws(lo) <= limit < ws(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if ws(mid) <= limit else (lo, mid)
    assert ws(lo) <= limit < ws(lo + 1)
    _check_against_both(f, _boundary_workload(lo), ptok)            # at the limit: runs
    g = _boundary_workload(lo + 1).to("cuda")                       # one partition more: rejected
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(f, g, g.lens, ptok, out, err) == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_static_scratch_rejects_shapes_beyond_its_size(cuda_ok):
    f = _entry()
    w = workloads.make_generic(B=64, H=64, Hkv=8, D=128, bs=16, dtype=torch.bfloat16,
                               lens=[3] * 64, poison=False)
    w.MB = 4096                      # room for 65536 tokens per sequence
    w.block_table = torch.full((w.B, w.MB), -1, dtype=torch.int32)
    g = w.to("cuda")
    assert pa.paged_attention_partial_workspace(hz.shape_of(g), 16) > scratch_bytes()
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(f, g, g.lens, 16, out, err) == pa.PA_ERR_WORKSPACE
