"""GPU parity of the shared-prefix split-KV pair over the quantised caches
(paged_attention_decode_shared_prefix_int8 / _fp8) against the CPU oracle:
the shared-beams workload at full size, groups of several sizes next to
ungrouped sequences on each supported head_dim, query dtype and block size
(tensor boxes, and row copies for block sizes that boxes cannot tile),
partitions that straddle the end of the shared prefix, agreement with the
single-pass decode of the same cache, the device check of the declared
sharing, a bad block inside a per-sequence partition, and the shapes the
entry points reject."""
from dataclasses import dataclass
from typing import Callable

import pytest
import torch

import oracle
import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu

F32, F16, BF16 = torch.float32, torch.float16, torch.bfloat16


@dataclass(frozen=True)
class Fmt:
    convert: Callable
    append: Callable
    decode: Callable
    prefix: Callable
    oracle_append: Callable
    oracle_decode: Callable


FMTS = {
    "int8": Fmt(workloads.to_int8, pa.paged_kv_append_int8, pa.paged_attention_decode_int8,
                pa.paged_attention_decode_shared_prefix_int8, oracle.kv_append_i8, oracle.attention_decode_i8),
    "fp8": Fmt(workloads.to_fp8, pa.paged_kv_append_fp8, pa.paged_attention_decode_fp8,
               pa.paged_attention_decode_shared_prefix_fp8, oracle.kv_append_fp8, oracle.attention_decode_fp8),
}


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()


def kwp(w):
    return dict(block_size=w.bs, num_blocks=w.NB, block_stride=w.block_stride)


def gpu_prefix(fmt, g, lens, ptok, err, group_first, shared_tokens):
    ws = pa.workspace_for(g.q, g.block_table, ptok, num_kv_heads=g.Hkv, **kwp(g))
    ws.fill_(0xFF)   # NaN pattern: a slot the reduce reads without a write shows up
    out = torch.empty_like(g.q)
    FMTS[fmt].prefix(out, g.q, g.k_flat(), g.v_flat(), g.scales, g.block_table, lens, g.scale, ptok, ws,
                     group_first=group_first, shared_tokens=shared_tokens, num_kv_heads=g.Hkv,
                     err_word=err, **kwp(g))
    return out


def oracle_decode(fmt, w, pool, lens):
    flat = pool.view(-1)
    return FMTS[fmt].oracle_decode(w.q, flat, flat[w.v_offset:], w.scales, w.block_table, lens, w.scale,
                                   num_kv_heads=w.Hkv, **kwp(w))


def check(fmt, w16, ptok, group_first, shared_tokens, seed=17):
    """Quantising append, then the shared-prefix decode over L + 1 tokens, vs
    the oracle (codes bit-exact, outputs within the 16-bit tolerance that a
    quantised cache is held to whatever the query dtype)."""
    f = FMTS[fmt]
    w = f.convert(w16, seed=seed)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    f.append(g.k_new, g.v_new, g.k_flat(), g.v_flat(), g.scales, g.block_table, g.lens, err_word=err,
             **kwp(g))
    out = gpu_prefix(fmt, g, g.lens + 1, ptok, err, group_first, shared_tokens)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    pool = w.pool.clone()
    flat = pool.view(-1)
    e = f.oracle_append(w.k_new, w.v_new, flat, flat[w.v_offset:], w.scales, w.block_table, w.lens, **kwp(w))
    assert not e.any()
    assert torch.equal(g.pool.cpu(), pool), "append codes differ"
    ref, e = oracle_decode(fmt, w, pool, w.lens + 1)
    assert not e.any()
    return hz.assert_close(out, ref, F16, w.name)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("ptok", [1024, 4096])
def test_shared_beams_full_size(fmt, ptok):
    w = workloads.make_workload(5)
    shared = w.meta["shared_blocks"] * w.bs
    check(fmt, w, ptok, [0, w.B], [shared])


SHAPES = [(4, 4, BF16, 128, 16), (16, 2, F16, 128, 16), (8, 8, BF16, 64, 32), (16, 4, BF16, 128, 8),
          (4, 2, F16, 64, 24), (2, 1, BF16, 128, 48)]


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("H,Hkv,dtype,D,bs", SHAPES)
@pytest.mark.parametrize("ptok", [16, 256])
def test_groups_next_to_ungrouped_sequences(fmt, H, Hkv, dtype, D, bs, ptok):
    g = H // Hkv
    big = max(1, min(4, 16 // g))
    sizes = [big, 1, 2, 1]
    w = workloads.make_prefix_groups(group_sizes=sizes, shared_blocks=[600 // bs + 1, 0, 300 // bs, 2],
                                     tails=[3, 17, 40, 9, 0, 33, 5, 71][:sum(sizes)], H=H, Hkv=Hkv, D=D,
                                     bs=bs, dtype=dtype, seed=H + D + bs, poison=False)
    check(fmt, w, ptok, w.meta["group_first"], w.meta["shared_tokens"], seed=H + bs)


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_fp32_queries(D):
    w = workloads.make_prefix_groups(group_sizes=[3, 1], shared_blocks=[30, 0], tails=[4, 0, 21, 50],
                                     H=4, Hkv=4, D=D, bs=16, dtype=F32, seed=D, poison=False)
    check("fp8", w, 64, w.meta["group_first"], w.meta["shared_tokens"])


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_equals_the_single_pass_decode(fmt):
    f = FMTS[fmt]
    w = f.convert(workloads.make_prefix_groups(group_sizes=[4, 3], shared_blocks=[40, 25],
                                               tails=[5, 9, 100, 0, 31, 64, 2], H=32, Hkv=32, D=128, bs=16,
                                               dtype=BF16, seed=3, poison=False))
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = gpu_prefix(fmt, g, g.lens, 128, err, w.meta["group_first"], w.meta["shared_tokens"])
    b = torch.empty_like(g.q)
    f.decode(b, g.q, g.k_flat(), g.v_flat(), g.scales, g.block_table, g.lens, g.scale, num_kv_heads=g.Hkv,
             err_word=err, **kwp(g))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hz.assert_close(a, b.double().cpu().numpy(), F16)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_declared_sharing_is_checked(fmt):
    """A member whose table leaves the shared blocks, or whose length does not
    cover the declared prefix, turns its group's outputs to zeros with
    PA_DEVERR_BAD_PREFIX; other groups are unaffected."""
    w = FMTS[fmt].convert(workloads.make_prefix_groups(group_sizes=[3, 2], shared_blocks=[20, 20],
                                                       tails=[5, 9, 7, 3, 4], H=4, Hkv=4, D=128, bs=16,
                                                       dtype=BF16, seed=4, poison=False))
    ref, _ = oracle_decode(fmt, w, w.pool, w.lens)
    g = w.to("cuda")
    g.block_table[1, 3] = g.block_table[3, 3]   # group 0: member 1 names another (valid) block
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_prefix(fmt, g, g.lens, 64, err, w.meta["group_first"], w.meta["shared_tokens"])
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_PREFIX
    assert not out[0:3].any()
    hz.assert_close(out[3:5], ref[3:5], F16)
    g2 = w.to("cuda")                            # group 1 declares more than member 4 holds
    err.zero_()
    lens = g2.lens.clone()
    lens[4] = 100
    out = gpu_prefix(fmt, g2, lens, 64, err, w.meta["group_first"], w.meta["shared_tokens"])
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_PREFIX
    assert not out[3:5].any()
    hz.assert_close(out[0:3], ref[0:3], F16)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_bad_block_in_a_private_partition(fmt):
    """A hole in an ungrouped sequence's table sets PA_DEVERR_BAD_BLOCK and
    zeros that sequence only."""
    w = FMTS[fmt].convert(workloads.make_prefix_groups(group_sizes=[2, 1], shared_blocks=[12, 0],
                                                       tails=[6, 30, 90], H=8, Hkv=2, D=64, bs=16, dtype=F16,
                                                       seed=6, poison=False))
    ref, _ = oracle_decode(fmt, w, w.pool, w.lens)
    g = w.to("cuda")
    g.block_table[2, 3] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_prefix(fmt, g, g.lens, 32, err, w.meta["group_first"], w.meta["shared_tokens"])
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_BLOCK
    assert not out[2].any()
    hz.assert_close(out[0:2], ref[0:2], F16)


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_rejects_what_it_cannot_run(fmt):
    f = FMTS[fmt]
    w = f.convert(workloads.make_prefix_groups(group_sizes=[5], shared_blocks=[4], tails=[1, 2, 3, 4, 5],
                                               H=8, Hkv=2, D=128, bs=16, dtype=BF16, seed=5, poison=False))
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as ei:   # 5 members x 4 heads > 16 columns
        gpu_prefix(fmt, g, g.lens, 64, err, [0, 5], [64])
    assert ei.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PagedAttnError) as ei:   # not ascending
        gpu_prefix(fmt, g, g.lens, 64, err, [0, 3, 2], [64, 0])
    assert ei.value.status == pa.PA_ERR_INVALID_ARG
    w256 = f.convert(workloads.make_prefix_groups(group_sizes=[2], shared_blocks=[2], tails=[1, 2], H=2,
                                                  Hkv=2, D=256, bs=16, dtype=BF16, seed=5, poison=False))
    g = w256.to("cuda")
    with pytest.raises(pa.PagedAttnError) as ei:   # head_dim 256: no tensor-core code kernel
        gpu_prefix(fmt, g, g.lens, 32, err, [0, 2], [32])
    assert ei.value.status == pa.PA_ERR_UNSUPPORTED
    if fmt == "int8":
        w32 = f.convert(workloads.make_prefix_groups(group_sizes=[2], shared_blocks=[2], tails=[1, 2], H=2,
                                                     Hkv=2, D=128, bs=16, dtype=F32, seed=5, poison=False))
        g = w32.to("cuda")
        with pytest.raises(pa.PagedAttnError) as ei:   # fp32 queries over int8: no tensor-core kernel
            gpu_prefix(fmt, g, g.lens, 32, err, [0, 2], [32])
        assert ei.value.status == pa.PA_ERR_UNSUPPORTED
