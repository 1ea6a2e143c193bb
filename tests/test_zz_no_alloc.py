"""paged_attention_decode_split_static: split-KV decode for callers that
cannot allocate device memory.

Some callers of this library are not allowed to allocate: code running inside
a memory pool or allocator callback, a plugin that a host framework hands only
its input and output buffers, or work being captured into a CUDA graph where
an allocation would break the capture.  For them the library keeps the
split-KV partial results in a fixed scratch array of its own.  These tests
call that entry point through the C ABI, twice in a row on different shapes
(the array keeps whatever the previous call left), and compare each result
with paged_attention_decode on the same inputs.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20      # PA_STATIC_SCRATCH_BYTES in include/pagedattn.h


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


def test_static_scratch_split_matches_decode_twice_in_a_row(cuda_ok):
    f = _entry()
    cases = [
        (workloads.make_workload(5, max_len=6000, poison=True), 1024),        # MHA, shared prefix
        (workloads.make_workload(4, batch=6, max_len=900, poison=True), 256),  # GQA, tensor cores
    ]
    for w, ptok in cases:
        g = w.to("cuda")
        shape = hz.shape_of(g)
        assert 0 < pa.paged_attention_partial_workspace(shape, ptok) <= SCRATCH_BYTES
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = hz.gpu_decode(g, g.lens, err)
        out = torch.full_like(g.q, float("nan"))
        st = _call(f, g, g.lens, ptok, out, err)
        assert st == pa.PA_OK, pa.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        atol, rtol = hz.TOL[w.dtype]
        diff = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert bool((diff <= atol + rtol * ref.float().abs()).all()), float(diff.max())


def test_static_scratch_rejects_shapes_beyond_its_size(cuda_ok):
    f = _entry()
    w = workloads.make_generic(B=64, H=64, Hkv=8, D=128, bs=16, dtype=torch.bfloat16,
                               lens=[3] * 64, poison=False)
    w.MB = 4096                      # room for 65536 tokens per sequence
    w.block_table = torch.full((w.B, w.MB), -1, dtype=torch.int32)
    g = w.to("cuda")
    assert pa.paged_attention_partial_workspace(hz.shape_of(g), 16) > SCRATCH_BYTES
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(f, g, g.lens, 16, out, err) == pa.PA_ERR_WORKSPACE
