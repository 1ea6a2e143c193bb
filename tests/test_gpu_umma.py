"""GPU parity of the tcgen05 grouped-query kernel (head_dim 128, 16-bit
caches) against the CPU oracle, on the shapes that reach its own code paths:
several units per CTA (the persistent grid gives each CTA an equal share),
zero-length and bad-table units among a CTA's units, block sizes whose
tiles are fetched as 128-row boxes, sliding windows and split-KV partitions
on and off that box grid, the fused append on every tile position, 16 query
heads per kv head (two head tiles), the split-KV workspace against the
oracle's partial sums, and the full-size batches the benchmark times.  Pools
are poisoned in every slot the step must not read.
"""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tcgen05_batch(Hkv, parts=1, many=False):
    """A batch whose (sequence, kv head[, partition]) units put the launch on
    the tcgen05 kernel: between a third of the SM count and the SM count
    (one unit per CTA), or with many=True at least three times the SM count
    (several units per CTA)."""
    sms, per = _sms(), Hkv * parts
    if many:
        return -(-3 * sms // per)
    b = max(1, (sms // 2) // per)
    assert 3 * b * per >= sms and b * per < sms, "no batch puts this shape on the tcgen05 kernel"
    return b


def _repeat(pattern, n):
    return [pattern[i % len(pattern)] for i in range(n)]


def _batch_on_tcgen05(pattern, *, H, Hkv, bs, window=0, ptok=0):
    """The length pattern repeated (whole, so the table row length stays the
    same) over the smallest batch the library runs on the tcgen05 kernel."""
    probe = workloads.make_generic(B=len(pattern), H=H, Hkv=Hkv, D=128, bs=bs, dtype=BF16, lens=pattern,
                                   seed=0, poison=False)
    for n in range(len(pattern), 8 * _sms()):
        if pa.paged_attention_decode_kernel(hz.shape_of(probe, batch=n), window, ptok) == pa.PA_KERNEL_TCGEN05:
            return _repeat(pattern, n)
    raise AssertionError("no batch puts this shape on the tcgen05 kernel")


def _assert_tcgen05(w, window=0, ptok=0):
    assert pa.paged_attention_decode_kernel(hz.shape_of(w), window, ptok) == pa.PA_KERNEL_TCGEN05


def _ragged(n, seed, hi=700):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, hi, (n,), generator=g).tolist()
    lens[n // 3] = 0            # empty sequences among the units
    lens[n // 2] = 127          # one token short of a tile after the append
    lens[-1] = 128              # a tile and one token
    return lens


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("H,Hkv", [(32, 4), (64, 4)])
def test_many_units_per_cta(dtype, H, Hkv):
    """More units than SMs: every CTA walks through several units, with the
    tile stream running across unit boundaries."""
    B = _tcgen05_batch(Hkv, many=True)
    w = workloads.make_generic(B=B, H=H, Hkv=Hkv, D=128, bs=16, dtype=dtype, lens=_ragged(B, H + Hkv),
                               seed=H, poison=True)
    _assert_tcgen05(w)
    hz.run_step_and_check(w)
    hz.run_fused_step_and_check(w)


@pytest.mark.parametrize("bs", [128, 256])
@pytest.mark.parametrize("H,Hkv", [(8, 1), (16, 2)])
def test_tall_boxes(bs, H, Hkv):
    """Block sizes that are multiples of 128: 128-row boxes, whole tiles per
    copy, a partial last box full of poison."""
    lens = _repeat([0, 1, 127, 128, 129, 255, 256, 1000, 1500], _tcgen05_batch(Hkv))
    w = workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=128, bs=bs, dtype=BF16, lens=lens,
                               seed=bs + H, poison=True)
    _assert_tcgen05(w)
    hz.run_step_and_check(w)
    hz.run_fused_step_and_check(w)


@pytest.mark.parametrize("bs", [16, 256])
@pytest.mark.parametrize("window", [1, 100, 128, 300])
def test_windows_on_the_box_grid(bs, window):
    lens = _repeat([5, 130, 700, 1023, 2000], _tcgen05_batch(4))
    w = workloads.make_generic(B=len(lens), H=32, Hkv=4, D=128, bs=bs, dtype=F16, lens=lens,
                               seed=window + bs, poison=True)
    _assert_tcgen05(w, window=window)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.q)
    pa.paged_attention_decode_window(out, g.q, g.k_flat(), g.v_flat(), g.block_table, g.lens, g.scale,
                                     window, num_kv_heads=w.Hkv, err_word=err, **hz.kw(g))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    flat = w.pool.view(-1)
    ref, e = oracle.attention_decode_window(w.q, flat, flat[w.v_offset:], w.block_table, w.lens, w.scale,
                                            window, num_kv_heads=w.Hkv, **hz.kw(w))
    assert not e.any()
    hz.assert_close(out, ref, F16, f"window {window} bs {bs}")


@pytest.mark.parametrize("bs,ptok", [(256, 256), (256, 512), (256, 48), (16, 128), (128, 384)])
def test_split_on_and_off_the_box_grid(bs, ptok):
    lens = _batch_on_tcgen05([0, 17, 300, 1200, 1777], H=16, Hkv=2, bs=bs, ptok=ptok)
    w = workloads.make_generic(B=len(lens), H=16, Hkv=2, D=128, bs=bs, dtype=BF16, lens=lens,
                               seed=ptok + bs, poison=True)
    _assert_tcgen05(w, ptok=ptok)
    hz.run_step_and_check(w, split_ptok=ptok)


def test_split_partials_match_oracle_partials_gqa():
    """The workspace holds, per partition, the maximum in log2 units and the
    sum and weighted V relative to it."""
    ptok = 256
    parts = -(-((-(-1001 // 16) + 2) * 16) // ptok)       # partitions of the table row
    lens = _repeat([200, 513, 1000], _tcgen05_batch(2, parts))
    w = workloads.make_generic(B=len(lens), H=16, Hkv=2, D=128, bs=16, dtype=BF16, lens=lens, seed=3,
                               poison=True)
    _assert_tcgen05(w, ptok=ptok)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, ws = hz.gpu_split(g, g.lens, ptok, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    P = -(-(w.MB * w.bs) // ptok)
    n = w.B * w.H * P
    raw = ws.cpu()
    m = raw[:4 * n].view(torch.float32).view(w.B, w.H, P).double().numpy()
    l = raw[4 * n:8 * n].view(torch.float32).view(w.B, w.H, P).double().numpy()
    off = (8 * n + 15) // 16 * 16
    acc = raw[off:off + 4 * n * w.D].view(torch.float32).view(w.B, w.H, P, w.D).double().numpy()
    flat = w.pool.view(-1)
    for p in range(P):
        om, ol, oacc, _ = oracle.attention_partial(w.q, flat, flat[w.v_offset:], w.block_table, w.lens,
                                                   w.scale, p * ptok, (p + 1) * ptok, num_kv_heads=w.Hkv,
                                                   **hz.kw(w))
        for b in range(w.B):
            if p * ptok >= int(w.lens[b]):
                continue
            np.testing.assert_allclose(m[b, :, p], om[b] / np.log(2.0), rtol=1e-5, atol=1e-4)
            shift = np.exp2(m[b, :, p] - om[b] / np.log(2.0))
            np.testing.assert_allclose(l[b, :, p] * shift, ol[b], rtol=1e-3, atol=1e-3)
            np.testing.assert_allclose(acc[b, :, p] * shift[:, None], oacc[b], rtol=2e-3, atol=4e-3)


def test_bad_units_among_good_ones():
    """A bad table entry and a length past the table row in the middle of a
    CTA's units: those units are zero and flagged, their neighbours exact."""
    B = _tcgen05_batch(4, many=True)  # several units per CTA
    lens = [300] * B
    w = workloads.make_generic(B=B, H=32, Hkv=4, D=128, bs=16, dtype=BF16, lens=lens, seed=9, poison=True)
    _assert_tcgen05(w)
    w.block_table[7, 5] = -1
    w.block_table[8, 0] = w.NB + 2
    g = w.to("cuda")
    lens_d = g.lens.clone()
    lens_d[11] = w.MB * w.bs + 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = hz.gpu_decode(g, lens_d, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_BLOCK and e & pa.DEVERR_BAD_LEN
    for b in (7, 8, 11):
        assert not out[b].any()
    good = [b for b in range(B) if b not in (7, 8, 11)]
    ref, _ = hz.oracle_decode(w, w.pool, w.lens)
    hz.assert_close(out[good], ref[good], BF16)


def test_large_scores_rescale_in_tensor_memory():
    """Scores that grow along the sequence force the running maximum up by
    far more than 2^8 after the first tile, so the accumulator in tensor
    memory is rescaled."""
    lens = _repeat([1000, 2000, 300], _tcgen05_batch(2))
    w = workloads.make_generic(B=len(lens), H=16, Hkv=2, D=128, bs=16, dtype=F16, lens=lens, seed=4,
                               poison=False)
    _assert_tcgen05(w)
    # K rows grow with their position: later tiles score higher
    pos = torch.arange(w.bs, dtype=torch.float32)
    for b in range(w.B):
        for j in range(-(-int(w.lens[b]) // w.bs)):
            blk = int(w.block_table[b, j])
            w.pool[blk, 0] = (w.pool[blk, 0].float() * (1 + (j * w.bs + pos[None, :, None]) / 60.0)).to(F16)
    workloads.poison_pool(w)
    w.q = (w.q.float() * 3.0).to(F16)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("batch", [16, 64])
def test_workload4_batches_the_bench_times_on_tcgen05(batch):
    """The GQA layer at batch 16 and 64 (full length, block size 16), as the
    benchmark's per-workload entries run it: the tcgen05 kernel, fused append
    + decode in one launch, every output against the oracle."""
    w = workloads.make_workload(4, block_size=16, batch=batch, poison=True)
    _assert_tcgen05(w)
    hz.run_fused_step_and_check(w)


@pytest.mark.parametrize("H,Hkv,lens", [
    (64, 8, [4500]),                                     # 8 units: clusters of 8
    (64, 8, [4500, 1, 129, 0]),                          # 32 units: clusters of 4, some shares empty
    (64, 8, [4500, 1, 129, 0, 700, 2047, 3000, 128]),   # 64 units: clusters of 2
    (16, 1, [4200, 17, 2000]),                          # 16 heads per kv head (two head tiles)
    (32, 4, [1100, 300, 1025]),                          # a short table row: clusters of 2
])
def test_few_units_spread_over_clusters(H, Hkv, lens):
    """Fewer units than SMs: the CTAs of a cluster take equal shares of a
    unit's tiles (shares of short sequences are empty, the appended row falls
    in the last share) and the first CTA merges the shares through
    distributed shared memory."""
    assert len(lens) * Hkv < _sms() // 2, "the batch must have few units"
    w = workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens,
                               seed=H + len(lens), poison=True)
    _assert_tcgen05(w)
    hz.run_step_and_check(w)
    hz.run_fused_step_and_check(w)


def test_bad_block_in_a_later_share():
    """A bad table entry deep in a long sequence (in a share other than the
    merging CTA's) zeroes that unit and raises the flag; the other units of
    the launch stay exact."""
    lens = [4000, 3900, 2500]
    w = workloads.make_generic(B=len(lens), H=32, Hkv=4, D=128, bs=16, dtype=BF16, lens=lens, seed=21,
                               poison=True)
    _assert_tcgen05(w)
    w.block_table[1, 200] = -1          # token 3200: the last shares of sequence 1
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = hz.gpu_decode(g, g.lens, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_BLOCK
    assert not out[1].any()
    ref, _ = hz.oracle_decode(w, w.pool, w.lens)
    hz.assert_close(out[[0, 2]], ref[[0, 2]], BF16)


@pytest.mark.parametrize("window", [1100, 2500])
def test_window_across_cluster_shares(window):
    """Sliding-window decodes long enough to be spread over a cluster: the
    shares start at the window's tile and the rows before the window start
    stay masked."""
    lens = [4096, 3000, 1500]
    w = workloads.make_generic(B=len(lens), H=16, Hkv=2, D=128, bs=16, dtype=F16, lens=lens,
                               seed=window, poison=True)
    _assert_tcgen05(w, window=window)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(g.q)
    pa.paged_attention_decode_window(out, g.q, g.k_flat(), g.v_flat(), g.block_table, g.lens, g.scale,
                                     window, num_kv_heads=w.Hkv, err_word=err, **hz.kw(g))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    flat = w.pool.view(-1)
    ref, e = oracle.attention_decode_window(w.q, flat, flat[w.v_offset:], w.block_table, w.lens, w.scale,
                                            window, num_kv_heads=w.Hkv, **hz.kw(w))
    assert not e.any()
    hz.assert_close(out, ref, F16, f"window {window}")


@pytest.mark.parametrize("B", [1, 2, 5, 9, 12, 19, 24, 40, 57])
def test_batch_sweep_across_dispatch_regimes(B):
    """The GQA layer's shape (64 query heads on 8 kv heads) over a sweep of
    batches that crosses every choice plan_decode makes: one unit per cluster
    of 8, 4 or 2 tcgen05 CTAs, one tcgen05 CTA per unit, the mma.sync kernel,
    and several units per tcgen05 CTA; a long first sequence sets the table
    row length so that clusters apply, and zero-length and short sequences
    sit among the others.  Fused append + decode against the oracle."""
    pattern = [4200, 37, 600, 0, 250, 1500, 129]
    lens = _repeat(pattern, B)
    w = workloads.make_generic(B=B, H=64, Hkv=8, D=128, bs=16, dtype=BF16, lens=lens, seed=100 + B,
                               poison=True)
    assert pa.paged_attention_decode_kernel(hz.shape_of(w), 0, 0) in (pa.PA_KERNEL_TCGEN05, pa.PA_KERNEL_MMA_SYNC)
    hz.run_fused_step_and_check(w)
