"""Shared helpers for the GPU parity tests: run a decode step through the C
ABI and the same step through the CPU oracle, then compare.

Tolerances: appends are compared bit for bit; attention outputs must satisfy
|gpu - ref| <= 2e-3 + 1e-2*|ref| for fp16/bf16 caches and <= 1e-5 for fp32
(fp32 accumulation on the GPU, fp64 in the oracle).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pagedattention_decode_paged_gb300 as pa

TOL = {torch.float32: (1e-5, 0.0), torch.float16: (2e-3, 1e-2), torch.bfloat16: (2e-3, 1e-2)}


def int_view(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def kw(w):
    return dict(block_size=w.bs, num_blocks=w.NB, block_stride=w.block_stride)


def shape_of(w, batch=None):
    return pa.make_shape(batch=w.B if batch is None else batch, num_heads=w.H,
                         num_kv_heads=w.Hkv, head_dim=w.D, block_size=w.bs,
                         max_blocks_per_seq=w.MB, num_blocks=w.NB, block_stride=w.block_stride,
                         dtype=w.dtype)


def gpu_append(g, positions, err):
    pa.paged_kv_append(g.k_new, g.v_new, g.k_flat(), g.v_flat(), g.block_table, positions,
                       err_word=err, **kw(g))


def gpu_decode(g, lens, err, out=None):
    out = torch.empty_like(g.q) if out is None else out
    pa.paged_attention_decode(out, g.q, g.k_flat(), g.v_flat(), g.block_table, lens, g.scale,
                              num_kv_heads=g.Hkv, err_word=err, **kw(g))
    return out


def gpu_split(g, lens, ptok, err, out=None):
    ws = pa.workspace_for(g.q, g.block_table, ptok, num_kv_heads=g.Hkv, **kw(g))
    ws.fill_(0xFF)  # NaN pattern: any slot the reduce reads without a write shows up
    out = torch.empty_like(g.q) if out is None else out
    pa.paged_attention_decode_partial(g.q, g.k_flat(), g.v_flat(), g.block_table, lens, g.scale,
                                      ptok, ws, num_kv_heads=g.Hkv, err_word=err, **kw(g))
    pa.paged_attention_decode_reduce(out, ws, lens, ptok, num_kv_heads=g.Hkv,
                                     max_blocks_per_seq=g.MB, err_word=err, **kw(g))
    return out, ws


def oracle_append(w):
    """Oracle pool after appending w.k_new/w.v_new at w.lens (copy of the pool)."""
    pool = w.pool.clone()
    flat = pool.view(-1)
    err = oracle.kv_append(w.k_new, w.v_new, flat, flat[w.v_offset:], w.block_table, w.lens, **kw(w))
    return pool, err


def oracle_decode(w, pool, lens, threads=0):
    flat = pool.view(-1)
    return oracle.attention_decode(w.q, flat, flat[w.v_offset:], w.block_table, lens, w.scale,
                                   num_kv_heads=w.Hkv, threads=threads, **kw(w))


def assert_close(got: torch.Tensor, ref: np.ndarray, dtype, what=""):
    atol, rtol = TOL[dtype]
    g = got.detach().float().cpu().double().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def run_step_and_check(w, *, split_ptok=None):
    """Append + decode (or split decode) on the GPU vs the oracle; returns max error."""
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append(g, g.lens, err)
    lens = g.lens + 1
    if split_ptok is None:
        out = gpu_decode(g, lens, err)
    else:
        out, _ = gpu_split(g, lens, split_ptok, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    ref_pool, e = oracle_append(w)
    assert not e.any()
    assert torch.equal(int_view(g.pool.cpu()), int_view(ref_pool)), "append not bit-exact"
    ref, e = oracle_decode(w, ref_pool, w.lens + 1)
    assert not e.any()
    return assert_close(out, ref, w.dtype, w.name)


def gpu_fused(g, positions, err, out=None):
    out = torch.empty_like(g.q) if out is None else out
    pa.paged_attention_decode_append(out, g.q, g.k_new, g.v_new, g.k_flat(), g.v_flat(),
                                     g.block_table, positions, g.scale, num_kv_heads=g.Hkv,
                                     err_word=err, **kw(g))
    return out


def run_fused_step_and_check(w):
    """paged_attention_decode_append on the GPU vs the oracle's append then decode."""
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_fused(g, g.lens, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    ref_pool, e = oracle_append(w)
    assert not e.any()
    assert torch.equal(int_view(g.pool.cpu()), int_view(ref_pool)), "append not bit-exact"
    ref, e = oracle_decode(w, ref_pool, w.lens + 1)
    assert not e.any()
    return out, assert_close(out, ref, w.dtype, w.name)


def balanced_ws(g):
    return pa.balanced_workspace_for(g.q, g.block_table, num_kv_heads=g.Hkv, **kw(g))


def balanced_counters(g, ws):
    """The per-item counters at the end of a balanced workspace (int32)."""
    n = pa.paged_attention_balanced_workspace(shape_of(g))
    if pa.paged_attention_decode_path(shape_of(g)) == pa.PA_PATH_TENSOR_GQA:
        items = g.B * g.Hkv * ((g.H // g.Hkv + 15) // 16)
    else:
        items = g.B * g.H
    return ws[n - 4 * items:n].view(torch.int32)


def gpu_balanced(g, err, *, lens=None, positions=None, window=0, ws=None, out=None):
    """One step through paged_attention_decode_balanced: plain decode over
    `lens`, or the fused append at `positions` then decode."""
    ws = balanced_ws(g) if ws is None else ws
    out = torch.empty_like(g.q) if out is None else out
    fused = positions is not None
    pa.paged_attention_decode_balanced(out, g.q, g.k_flat(), g.v_flat(), g.block_table, g.scale, ws,
                                       seq_lens=None if fused else lens, positions=positions,
                                       k_new=g.k_new if fused else None,
                                       v_new=g.v_new if fused else None, window=window,
                                       num_kv_heads=g.Hkv, err_word=err, **kw(g))
    return out, ws
