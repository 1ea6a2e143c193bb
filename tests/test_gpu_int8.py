"""GPU parity of the int8 cache (quantised blocks with per-(block, kv head)
scales) against the CPU oracle: the quantising append is compared code for
code (the rounding rule decides integers, so it must be bit-exact, including
ties, clamped values and NaN), and decode attention over the codes within
the 16-bit tolerance, on the five workloads' shapes, ragged lengths, every
supported head_dim and query dtype, GQA through the CUDA-core path, and the
device-side error handling."""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu

F32, F16, BF16 = torch.float32, torch.float16, torch.bfloat16


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()


def kw8(w):
    return dict(block_size=w.bs, num_blocks=w.NB, block_stride=w.block_stride)


def gpu_append8(g, positions, err):
    pa.paged_kv_append_int8(g.k_new, g.v_new, g.k_flat(), g.v_flat(), g.scales, g.block_table,
                            positions, err_word=err, **kw8(g))


def gpu_decode8(g, lens, err):
    out = torch.empty_like(g.q)
    pa.paged_attention_decode_int8(out, g.q, g.k_flat(), g.v_flat(), g.scales, g.block_table, lens,
                                   g.scale, num_kv_heads=g.Hkv, err_word=err, **kw8(g))
    return out


def oracle_append8(w, positions=None):
    pool = w.pool.clone()
    flat = pool.view(-1)
    e = oracle.kv_append_i8(w.k_new, w.v_new, flat, flat[w.v_offset:], w.scales, w.block_table,
                            w.lens if positions is None else positions, **kw8(w))
    return pool, e


def oracle_decode8(w, pool, lens):
    flat = pool.view(-1)
    return oracle.attention_decode_i8(w.q, flat, flat[w.v_offset:], w.scales, w.block_table, lens,
                                      w.scale, num_kv_heads=w.Hkv, **kw8(w))


def run_step8(w):
    """Quantising append then decode over L + 1 tokens, vs the oracle."""
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append8(g, g.lens, err)
    out = gpu_decode8(g, g.lens + 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    ref_pool, e = oracle_append8(w)
    assert not e.any()
    assert torch.equal(g.pool.cpu(), ref_pool), "int8 append codes differ"
    ref, e = oracle_decode8(w, ref_pool, w.lens + 1)
    assert not e.any()
    # an int8 cache is held to the 16-bit tolerance whatever the query dtype
    return hz.assert_close(out, ref, F16, w.name)


@pytest.mark.parametrize("index,bs", [(1, None), (2, None), (3, 16), (3, 8), (4, 16), (5, None)])
def test_int8_workloads_full_size(index, bs):
    w = workloads.to_int8(workloads.make_workload(index, block_size=bs))
    run_step8(w)


LENS = [0, 1, 15, 16, 17, 31, 33, 64, 100, 257]


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_int8_every_head_dim_and_query_dtype(dtype, D):
    w = workloads.to_int8(workloads.make_generic(B=len(LENS), H=3, Hkv=3, D=D, bs=16, dtype=dtype,
                                                 lens=LENS, seed=D, poison=False), seed=D)
    run_step8(w)


@pytest.mark.parametrize("bs", [1, 3, 8, 24, 32, 128])
def test_int8_block_sizes(bs):
    w = workloads.to_int8(workloads.make_generic(B=len(LENS), H=2, Hkv=2, D=128, bs=bs, dtype=BF16,
                                                 lens=LENS, seed=bs, poison=False), seed=bs)
    run_step8(w)


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(8, 2, BF16, 128, 16), (16, 1, BF16, 128, 16),
                                              (64, 8, BF16, 128, 16), (48, 2, F16, 128, 16),
                                              (16, 2, F16, 64, 8), (8, 1, F16, 64, 16),
                                              (8, 2, BF16, 128, 3), (8, 2, F32, 128, 16)])
def test_int8_grouped_query(H, Hkv, dtype, D, bs):
    """Tensor-core int8 path (16-bit queries, head_dim 64/128, any block
    size) and the CUDA-core one for fp32 queries."""
    w = workloads.to_int8(workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype,
                                                 lens=LENS, seed=H + bs, poison=False), seed=H)
    run_step8(w)


@pytest.mark.parametrize("D,H,Hkv", [(64, 8, 2), (128, 8, 2), (128, 2, 2), (256, 3, 3)])
def test_int8_grouped_query_long_sequences(D, H, Hkv):
    """Sequences with more blocks than the kernels stage in shared memory
    (the rest of the table and its scales come from global memory); with
    few (sequence, head) units the CUDA-core kernel spreads each over a
    thread-block cluster."""
    lens = [9000, 17, 8200]
    w = workloads.to_int8(workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=D, bs=16, dtype=BF16,
                                                 lens=lens, seed=D + 1, poison=False), seed=D)
    run_step8(w)


def test_int8_append_rounding_edges():
    """Ties, clamped values, infinities and NaN through the quantising append."""
    B, Hkv, D, bs = 4, 2, 64, 16
    w = workloads.to_int8(workloads.make_generic(B=B, H=Hkv, Hkv=Hkv, D=D, bs=bs, dtype=F32,
                                                 lens=[5, 16, 31, 0], seed=3, poison=False), seed=3)
    # power-of-two scales make (k + 0.5) * s exact ties in binary32
    w.scales = (2.0 ** torch.randint(-9, -3, w.scales.shape, generator=torch.Generator().manual_seed(1))).float()
    k = torch.arange(-140, 140, dtype=torch.float32)
    vals = torch.cat([k + 0.5, k])[: B * Hkv * D].reshape(B, Hkv, D)
    s_first = w.scales[0, 0, 0]
    kn = vals * s_first
    kn[0, 0, :4] = torch.tensor([float("inf"), float("-inf"), float("nan"), 1e30])
    w.k_new = kn.contiguous()
    w.v_new = (-kn).contiguous()
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append8(g, g.lens, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_pool, _ = oracle_append8(w)
    assert torch.equal(g.pool.cpu(), ref_pool)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_int8_errors_reported_and_zeroed(H, Hkv):
    lens = [40, 40, 40, 40]
    w = workloads.to_int8(workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens,
                                                 seed=9, poison=False), seed=9)
    w.block_table[1, 1] = -1                 # hole inside the valid range
    w.block_table[2, 0] = w.NB + 2           # id past the pool
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_lens = torch.tensor([40, 40, 40, w.MB * w.bs + 1], dtype=torch.int32, device="cuda")
    out = gpu_decode8(g, bad_lens, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_BLOCK and e & pa.DEVERR_BAD_LEN
    assert not out[1].any() and not out[2].any() and not out[3].any()
    ref, _ = oracle_decode8(w, w.pool, torch.tensor(lens, dtype=torch.int32))
    hz.assert_close(out[0:1], ref[0:1], F16)
    # the append skips a bad position and an unallocated target, writing the rest
    before = g.pool.clone()
    pos = torch.tensor([40, w.MB * w.bs, 40, 40], dtype=torch.int32, device="cuda")
    g.block_table[3, 2] = -1
    err.zero_()
    gpu_append8(g, pos, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_POS and e & pa.DEVERR_BAD_BLOCK
    changed = (g.pool != before).reshape(w.NB, -1).any(1)
    assert set(torch.nonzero(changed).flatten().tolist()) == {int(w.block_table[0, 2]),
                                                               int(w.block_table[2, 2])}
