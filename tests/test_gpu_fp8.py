"""GPU parity of the fp8 cache (OCP FP8 E4M3 codes with per-(block, kv head)
scales) against the CPU oracle: the quantising append is compared code for
code (the rounding rule decides the codes, so it must be bit-exact,
including ties, subnormals and saturated values), and decode attention over
the codes within the 16-bit tolerance, on the five workloads' shapes,
ragged lengths, every head_dim and query dtype, both kernels (tensor cores
for grouped queries, CUDA cores for MHA and head_dim 256), odd block sizes
(row-by-row copies), NaN codes past the length, long sequences and the
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


def gpu_append(g, positions, err):
    pa.paged_kv_append_fp8(g.k_new, g.v_new, g.k_flat(), g.v_flat(), g.scales, g.block_table,
                           positions, err_word=err, **kw8(g))


def gpu_decode(g, lens, err):
    out = torch.empty_like(g.q)
    pa.paged_attention_decode_fp8(out, g.q, g.k_flat(), g.v_flat(), g.scales, g.block_table, lens,
                                  g.scale, num_kv_heads=g.Hkv, err_word=err, **kw8(g))
    return out


def oracle_append(w, positions=None):
    pool = w.pool.clone()
    flat = pool.view(-1)
    e = oracle.kv_append_fp8(w.k_new, w.v_new, flat, flat[w.v_offset:], w.scales, w.block_table,
                             w.lens if positions is None else positions, **kw8(w))
    return pool, e


def oracle_decode(w, pool, lens):
    flat = pool.view(-1)
    return oracle.attention_decode_fp8(w.q, flat, flat[w.v_offset:], w.scales, w.block_table, lens,
                                       w.scale, num_kv_heads=w.Hkv, **kw8(w))


def run_step(w):
    """Quantising append then decode over L + 1 tokens, vs the oracle."""
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append(g, g.lens, err)
    out = gpu_decode(g, g.lens + 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    ref_pool, e = oracle_append(w)
    assert not e.any()
    assert torch.equal(g.pool.cpu(), ref_pool), "fp8 append codes differ"
    ref, e = oracle_decode(w, ref_pool, w.lens + 1)
    assert not e.any()
    # an fp8 cache is held to the 16-bit tolerance whatever the query dtype
    return hz.assert_close(out, ref, F16, w.name)


@pytest.mark.parametrize("index,bs", [(1, None), (2, None), (3, 16), (3, 8), (4, 16), (4, 256), (5, None)])
def test_fp8_workloads_full_size(index, bs):
    w = workloads.to_fp8(workloads.make_workload(index, block_size=bs))
    run_step(w)


LENS = [0, 1, 15, 16, 17, 31, 33, 64, 100, 257]


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp8_every_head_dim_and_query_dtype(dtype, D):
    w = workloads.to_fp8(workloads.make_generic(B=len(LENS), H=3, Hkv=3, D=D, bs=16, dtype=dtype,
                                                lens=LENS, seed=D, poison=False), seed=D)
    run_step(w)


@pytest.mark.parametrize("bs", [1, 3, 8, 24, 32, 128])
def test_fp8_block_sizes(bs):
    w = workloads.to_fp8(workloads.make_generic(B=len(LENS), H=4, Hkv=2, D=128, bs=bs, dtype=BF16,
                                                lens=LENS, seed=bs, poison=False), seed=bs)
    run_step(w)


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(8, 2, BF16, 128, 16), (16, 1, BF16, 128, 16),
                                              (64, 8, BF16, 128, 16), (48, 2, F16, 128, 16),
                                              (16, 2, F16, 64, 8), (8, 1, F16, 64, 16),
                                              (8, 2, BF16, 128, 3), (8, 2, F32, 128, 16),
                                              (8, 2, BF16, 256, 16)])
def test_fp8_grouped_query(H, Hkv, dtype, D, bs):
    w = workloads.to_fp8(workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype,
                                                lens=LENS, seed=H + bs, poison=False), seed=H)
    run_step(w)


@pytest.mark.parametrize("D,H,Hkv", [(64, 8, 2), (128, 8, 2), (128, 2, 2), (256, 3, 3), (64, 2, 2)])
def test_fp8_long_sequences(D, H, Hkv):
    """More blocks than the kernels stage in shared memory."""
    lens = [9000, 17, 8200]
    w = workloads.to_fp8(workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=D, bs=16, dtype=BF16,
                                                lens=lens, seed=D + 1, poison=False), seed=D)
    run_step(w)


def test_fp8_append_rounding_edges():
    """Ties between neighbouring codes, subnormals, saturation and
    infinities through the quantising append, with power-of-two scales so
    that the binary32 quotient is exact."""
    B, Hkv, D, bs = 4, 2, 64, 16
    w = workloads.to_fp8(workloads.make_generic(B=B, H=Hkv, Hkv=Hkv, D=D, bs=bs, dtype=F32,
                                                lens=[5, 16, 31, 0], seed=3, poison=False), seed=3)
    w.scales = (2.0 ** torch.randint(-9, -3, w.scales.shape, generator=torch.Generator().manual_seed(1))).float()
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    fin = vals[torch.isfinite(vals) & (vals >= 0)].sort().values
    mids = (fin[1:] + fin[:-1]) / 2                         # exact ties between neighbours
    extra = torch.tensor([500.0, -500.0, 1e30, -1e30, float("inf"), float("-inf"), 449.0, -463.0,
                          2.0 ** -10, 3 * 2.0 ** -10, -(2.0 ** -11), 0.0, -0.0])
    pool_vals = torch.cat([mids, -mids, fin, extra])
    n = B * Hkv * D
    pool_vals = pool_vals.repeat(n // pool_vals.numel() + 1)[:n].reshape(B, Hkv, D)
    pos = w.lens
    kn = torch.empty(B, Hkv, D)
    vn = torch.empty(B, Hkv, D)
    for b in range(B):
        blk = int(w.block_table[b, int(pos[b]) // bs])
        for hk in range(Hkv):
            kn[b, hk] = pool_vals[b, hk] * w.scales[blk, 0, hk]
            vn[b, hk] = pool_vals[(b + 1) % B, hk] * w.scales[blk, 1, hk]
    w.k_new = kn.contiguous()
    w.v_new = vn.contiguous()
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_append(g, g.lens, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_pool, _ = oracle_append(w)
    assert torch.equal(g.pool.cpu(), ref_pool)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_fp8_errors_reported_and_zeroed(H, Hkv):
    lens = [40, 40, 40, 40]
    w = workloads.to_fp8(workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens,
                                                seed=9, poison=False), seed=9)
    w.block_table[1, 1] = -1                 # hole inside the valid range
    w.block_table[2, 0] = w.NB + 2           # id past the pool
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_lens = torch.tensor([40, 40, 40, w.MB * w.bs + 1], dtype=torch.int32, device="cuda")
    out = gpu_decode(g, bad_lens, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_BLOCK and e & pa.DEVERR_BAD_LEN
    assert not out[1].any() and not out[2].any() and not out[3].any()
    ref, _ = oracle_decode(w, w.pool, torch.tensor(lens, dtype=torch.int32))
    hz.assert_close(out[0:1], ref[0:1], F16)
    before = g.pool.clone()
    pos = torch.tensor([40, w.MB * w.bs, 40, 40], dtype=torch.int32, device="cuda")
    g.block_table[3, 2] = -1
    err.zero_()
    gpu_append(g, pos, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_POS and e & pa.DEVERR_BAD_BLOCK
    changed = (g.pool != before).reshape(w.NB, -1).any(1)
    assert set(torch.nonzero(changed).flatten().tolist()) == {int(w.block_table[0, 2]),
                                                               int(w.block_table[2, 2])}


def test_fp8_equals_16bit_decode_on_exactly_representable_values():
    """Codes times power-of-two scales are exact in fp16: the fp8 path and
    the 16-bit tensor-core path see the same K/V values, so they agree to
    rounding (both within tolerance of each other)."""
    w16 = workloads.make_workload(4, batch=4)
    w = workloads.to_fp8(w16, seed=5)
    w.scales = (2.0 ** torch.randint(-8, -6, w.scales.shape, generator=torch.Generator().manual_seed(2))).float()
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)
    deq = vals[w.pool.long()] * w.scales[:, :, :, None, None]
    w16.pool = deq.to(w16.dtype).reshape(w16.pool.shape)
    assert torch.equal(w16.pool.float().reshape(deq.shape), deq)   # exact in bf16
    g8, g16 = w.to("cuda"), w16.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = gpu_decode(g8, g8.lens, err)
    b = torch.empty_like(g16.q)
    pa.paged_attention_decode(b, g16.q, g16.k_flat(), g16.v_flat(), g16.block_table, g16.lens, g16.scale,
                              num_kv_heads=g16.Hkv, err_word=err, **hz.kw(g16))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hz.assert_close(a, b.double().cpu().numpy(), BF16, "fp8 vs bf16 path")


@pytest.mark.parametrize("bs,H,Hkv", [(16, 4, 4), (8, 8, 2), (3, 8, 2), (32, 16, 2), (8, 4, 4), (3, 2, 2)])
def test_fp8_nan_codes_past_the_length_are_ignored(bs, H, Hkv):
    """Slots past each sequence's length (in its last block, and in blocks
    nobody owns) hold NaN codes, as an unwritten pool may: they are never
    attended, so the outputs stay finite and equal the oracle's."""
    lens = [0, 1, 5, 17, 40, 100]
    w = workloads.to_fp8(workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=128, bs=bs, dtype=BF16,
                                                lens=lens, seed=bs + H, poison=False), seed=bs)
    pool = w.pool.view(w.NB, 2, Hkv, bs, 128)
    owned = set()
    for b, L in enumerate(lens):
        L1 = L + 1
        for j in range(-(-L1 // bs)):
            blk = int(w.block_table[b, j])
            owned.add(blk)
            lo = max(0, L1 - j * bs)
            if lo < bs:
                pool[blk, :, :, lo:, :] = 0x7F
    for blk in range(w.NB):
        if blk not in owned:
            pool[blk] = 0xFF
    run_step(w)
