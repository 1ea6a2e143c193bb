"""GPU parity of the append + decode step against the CPU oracle, on all five
seeded workloads at their full sizes and in the launch configuration the
benchmark times (append, then decode over L + 1 tokens; split-KV where the
benchmark uses it).  Pools are poisoned (NaN / inf / huge) in every slot the
step must not read, so a read past the valid length or into an unused block
shows up as a non-finite or wrong output.
"""
import numpy as np
import pytest
import torch

import oracle
import pagedattention_decode_paged_gb300 as pa
import workloads
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()


def test_workload1_tiny_fp32():
    w = workloads.make_workload(1, poison=True)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_SIMT
    hz.run_step_and_check(w)


def test_workload2_llama7b_fp16_full_size():
    w = workloads.make_workload(2, poison=True)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_workload3_longtail_bf16(bs):
    w = workloads.make_workload(3, block_size=bs, poison=True)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("bs", [16, 256])
def test_workload4_gqa_tensor_cores(bs):
    w = workloads.make_workload(4, block_size=bs, poison=True)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_TENSOR_GQA
    hz.run_step_and_check(w)


@pytest.mark.parametrize("ptok", [512, 2048])
def test_workload4_gqa_split(ptok):
    w = workloads.make_workload(4, block_size=16, poison=True)
    hz.run_step_and_check(w, split_ptok=ptok)


def test_workload5_shared_beams_single_pass():
    w = workloads.make_workload(5, poison=True)
    hz.run_step_and_check(w)


def test_workload5_shared_beams_split():
    w = workloads.make_workload(5, poison=True)
    hz.run_step_and_check(w, split_ptok=1024)


@pytest.mark.parametrize("ptok", [16, 32, 256, 1024, 4096])
def test_split_partition_sizes_mha(ptok):
    w = workloads.make_workload(2, batch=6, poison=True)
    hz.run_step_and_check(w, split_ptok=ptok)


@pytest.mark.parametrize("ptok", [16, 48, 256])
def test_split_partition_sizes_gqa(ptok):
    w = workloads.make_workload(4, batch=3, max_len=700, poison=True)
    hz.run_step_and_check(w, split_ptok=ptok)


def test_split_partials_match_oracle_partials():
    """The workspace holds m (log2 units), l and acc of each partition."""
    w = workloads.make_workload(2, batch=3, poison=True)
    ptok = 128
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
        om, ol, oacc, _ = oracle.attention_partial(w.q, flat, flat[w.v_offset:], w.block_table,
                                                   w.lens, w.scale, p * ptok, (p + 1) * ptok,
                                                   num_kv_heads=w.Hkv, **hz.kw(w))
        for b in range(w.B):
            if p * ptok >= int(w.lens[b]):
                continue  # partition past the sequence: never written, never read
            # gpu m is in log2 units of the same score: m_gpu = m * log2(e)
            np.testing.assert_allclose(m[b, :, p], om[b] / np.log(2.0), rtol=1e-5, atol=1e-4)
            # l and acc are relative to each side's own m; rescale to compare
            shift = np.exp2(m[b, :, p] - om[b] / np.log(2.0))
            np.testing.assert_allclose(l[b, :, p] * shift, ol[b], rtol=1e-4, atol=1e-4)
            np.testing.assert_allclose(acc[b, :, p] * shift[:, None], oacc[b], rtol=1e-3, atol=2e-3)


def test_shared_blocks_bitwise_equal_to_private_copies():
    w = workloads.make_workload(5, max_len=3000, poison=True)
    u = workloads.unshare(w)
    outs = []
    for x in (w, u):
        g = x.to("cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(hz.gpu_decode(g, g.lens, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    assert torch.equal(outs[0], outs[1])
    assert not torch.equal(outs[0][0], outs[0][1])  # beams differ in their tails


def test_decode_is_deterministic():
    w = workloads.make_workload(4, batch=4, max_len=1000).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = hz.gpu_decode(w, w.lens, err)
    b = hz.gpu_decode(w, w.lens, err)
    s1, _ = hz.gpu_split(w, w.lens, 256, err)
    s2, _ = hz.gpu_split(w, w.lens, 256, err)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(s1, s2)


@pytest.mark.parametrize("index,kwargs", [(1, {}), (4, dict(batch=2, max_len=90))])
def test_multi_step_decode_matches_oracle_every_step(index, kwargs):
    """Repeated append + decode: the multi-turn consistency check of "A strange
    KV Cache bug" (dpshk.com/news/5937191) s6, one token per step."""
    steps = 24
    w = workloads.make_workload(index, poison=True, **kwargs)
    # grow the tables so every step has a block to write into
    need = [-(-(int(L) + steps) // w.bs) for L in w.lens]
    used = set(int(x) for x in w.block_table.flatten() if x >= 0)
    free = [i for i in range(w.NB) if i not in used]
    MB = max(need) + 1
    table = torch.full((w.B, MB), -1, dtype=torch.int32)
    table[:, :w.MB] = w.block_table
    for b in range(w.B):
        have = int((w.block_table[b] >= 0).sum())
        for j in range(have, need[b]):
            table[b, j] = free.pop()
    w.block_table, w.MB = table, MB
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_pool = w.pool.clone()
    gen = torch.Generator().manual_seed(77)
    for step in range(steps):
        kn = torch.randn(w.k_new.shape, generator=gen).to(w.dtype)
        vn = torch.randn(w.v_new.shape, generator=gen).to(w.dtype)
        qn = torch.randn(w.q.shape, generator=gen).to(w.dtype)
        lens = w.lens + step
        g.k_new.copy_(kn)
        g.v_new.copy_(vn)
        g.q.copy_(qn)
        hz.gpu_append(g, lens.cuda(), err)
        out = hz.gpu_decode(g, (lens + 1).cuda(), err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        flat = ref_pool.view(-1)
        oracle.kv_append(kn, vn, flat, flat[w.v_offset:], table, lens, **hz.kw(w))
        w.q = qn
        ref, _ = hz.oracle_decode(w, ref_pool, lens + 1)
        hz.assert_close(out, ref, w.dtype, f"step {step}")
    assert torch.equal(hz.int_view(g.pool.cpu()), hz.int_view(ref_pool))


# ---------------------------------------------------------------------------
# the fused step: paged_attention_decode_append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("index,bs", [(1, None), (2, None), (3, 8), (3, 64), (4, 16), (4, 256), (5, None)])
def test_fused_append_decode_full_size(index, bs):
    w = workloads.make_workload(index, block_size=bs, poison=True)
    hz.run_fused_step_and_check(w)


@pytest.mark.parametrize("index", [2, 4, 5])
def test_fused_equals_separate_calls_bitwise(index):
    w = workloads.make_workload(index, poison=True, **({"max_len": 4000} if index == 5 else {}))
    a, b = w.to("cuda"), w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fused = hz.gpu_fused(a, a.lens, err)
    hz.gpu_append(b, b.lens, err)
    separate = hz.gpu_decode(b, b.lens + 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(fused, separate)
    assert torch.equal(hz.int_view(a.pool), hz.int_view(b.pool))
