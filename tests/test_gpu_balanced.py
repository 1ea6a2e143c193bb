"""GPU parity of paged_attention_decode_balanced -- the decode step on the
persistent, load-balanced grid -- against the CPU oracle: the five workloads
at full size (fused append + decode, and plain decode), every compiled shape
family, sliding windows, skewed length mixes that cut one item across
hundreds of warps, the device-side error handling, and the workspace
contract (its counters are back at zero after every call, so one zero fill
serves any number of calls)."""
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


def check_fused(w, *, window=0):
    """Fused append + decode on the balanced grid vs the oracle's append, then
    (window) decode over the new lengths; the append is bit-exact."""
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, ws = hz.gpu_balanced(g, err, positions=g.lens, window=window)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert not hz.balanced_counters(g, ws).any(), "counters not reset"
    ref_pool, e = hz.oracle_append(w)
    assert not e.any()
    assert torch.equal(hz.int_view(g.pool.cpu()), hz.int_view(ref_pool)), "append not bit-exact"
    if window:
        flat = ref_pool.view(-1)
        ref, e = oracle.attention_decode_window(w.q, flat, flat[w.v_offset:], w.block_table, w.lens + 1,
                                                w.scale, window, num_kv_heads=w.Hkv, **hz.kw(w))
    else:
        ref, e = hz.oracle_decode(w, ref_pool, w.lens + 1)
    assert not e.any()
    return out, hz.assert_close(out, ref, w.dtype, w.name)


def check_plain(w, *, window=0):
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, ws = hz.gpu_balanced(g, err, lens=g.lens, window=window)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert not hz.balanced_counters(g, ws).any(), "counters not reset"
    if window:
        ref, e = oracle.attention_decode_window(w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens,
                                                w.scale, window, num_kv_heads=w.Hkv, **hz.kw(w))
    else:
        ref, e = hz.oracle_decode(w, w.pool, w.lens)
    assert not e.any()
    return out, hz.assert_close(out, ref, w.dtype, w.name)


@pytest.mark.parametrize("index,bs", [(1, None), (2, None), (3, 8), (3, 16), (3, 32), (3, 64),
                                      (4, 16), (4, 256), (5, None)])
def test_balanced_fused_full_size(index, bs):
    w = workloads.make_workload(index, block_size=bs, poison=True)
    check_fused(w)


@pytest.mark.parametrize("index,bs", [(2, None), (3, 16), (4, 16), (5, None)])
def test_balanced_plain_full_size(index, bs):
    w = workloads.make_workload(index, block_size=bs, poison=True)
    check_plain(w)


LENS = [0, 1, 15, 16, 17, 31, 33, 64, 100, 257]
SKEW = [4000, 3, 1, 0, 17, 100, 2, 64, 4095, 1, 1, 700]   # one item over hundreds of warps


@pytest.mark.parametrize("dtype,D", [(F32, 16), (F32, 32), (F32, 64), (F32, 128),
                                     (F16, 32), (F16, 64), (F16, 128), (F16, 256),
                                     (BF16, 32), (BF16, 64), (BF16, 128), (BF16, 256)])
def test_balanced_mha_every_head_dim(dtype, D):
    w = workloads.make_generic(B=len(LENS), H=3, Hkv=3, D=D, bs=16, dtype=dtype, lens=LENS, seed=D)
    check_plain(w)
    check_fused(w)


@pytest.mark.parametrize("bs", [1, 3, 8, 24, 128])
def test_balanced_block_sizes(bs):
    w = workloads.make_generic(B=len(LENS), H=2, Hkv=2, D=128, bs=bs, dtype=BF16, lens=LENS, seed=bs)
    check_fused(w)


@pytest.mark.parametrize("H,Hkv", [(8, 4), (16, 4), (16, 1), (32, 1), (48, 2)])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_balanced_gqa_tensor_path(H, Hkv, dtype):
    w = workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=128, bs=16, dtype=dtype, lens=LENS,
                               seed=H * 7 + Hkv)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_TENSOR_GQA
    check_plain(w)
    check_fused(w)


@pytest.mark.parametrize("D,bs", [(64, 16), (128, 8), (128, 32), (64, 256)])
def test_balanced_gqa_head_dims_and_blocks(D, bs):
    w = workloads.make_generic(B=len(LENS), H=16, Hkv=2, D=D, bs=bs, dtype=BF16, lens=LENS, seed=D + bs)
    check_fused(w)


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(4, 4, BF16, 128, 16), (16, 2, BF16, 128, 16),
                                              (4, 4, F32, 64, 8), (32, 4, F16, 64, 16)])
def test_balanced_skewed_lengths(H, Hkv, dtype, D, bs):
    w = workloads.make_generic(B=len(SKEW), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype, lens=SKEW,
                               seed=H + D)
    check_plain(w)
    check_fused(w)


@pytest.mark.parametrize("H,Hkv,dtype", [(4, 4, F16), (8, 2, BF16)])
def test_balanced_separate_pools(H, Hkv, dtype):
    w = workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=64, bs=16, dtype=dtype, lens=LENS,
                               seed=11, separate_pools=True)
    check_fused(w)


WIN_LENS = [1, 5, 16, 17, 100, 700, 2049]


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(4, 4, F16, 128, 16), (16, 2, BF16, 128, 16),
                                              (8, 2, BF16, 128, 4), (2, 2, F32, 64, 8)])
@pytest.mark.parametrize("window", [1, 13, 100, 5000])
def test_balanced_window(H, Hkv, dtype, D, bs, window):
    w = workloads.make_generic(B=len(WIN_LENS), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype,
                               lens=WIN_LENS, seed=window + H)
    check_plain(w, window=window)
    check_fused(w, window=window)


def test_balanced_matches_single_pass_kernels():
    """Same step through the one-CTA-per-unit kernels: equal up to fp32
    rounding order (both within the oracle tolerance of each other)."""
    for index in (2, 4):
        w = workloads.make_workload(index, batch=8)
        a, b = w.to("cuda"), w.to("cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        bal, _ = hz.gpu_balanced(a, err, positions=a.lens)
        ref = hz.gpu_fused(b, b.lens, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        hz.assert_close(bal, ref.double().cpu().numpy(), w.dtype, f"workload {index}")
        assert torch.equal(hz.int_view(a.pool), hz.int_view(b.pool))


def test_balanced_is_deterministic_and_reuses_its_workspace():
    w = workloads.make_generic(B=len(SKEW), H=16, Hkv=2, D=128, bs=16, dtype=BF16, lens=SKEW, seed=3)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = hz.balanced_ws(g)
    outs = [hz.gpu_balanced(g, err, lens=g.lens, ws=ws)[0].clone() for _ in range(5)]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert not hz.balanced_counters(g, ws).any()


@pytest.mark.parametrize("index,kwargs", [(1, {}), (4, dict(batch=2, max_len=90)),
                                          (3, dict(batch=24))])
def test_balanced_multi_step(index, kwargs):
    """Repeated fused steps on one workspace: the multi-turn consistency check
    of "A strange KV Cache bug" (dpshk.com/news/5937191) s6."""
    steps = 20
    w = workloads.make_workload(index, poison=True, **kwargs)
    need = [-(-(int(L) + steps) // w.bs) for L in w.lens]
    used = set(int(x) for x in w.block_table.flatten() if x >= 0)
    free = [i for i in range(w.NB) if i not in used]
    if len(free) < sum(need) - int((w.block_table >= 0).sum()):
        pytest.skip("pool too small for the extra steps")
    MB = max(max(need) + 1, w.MB)
    table = torch.full((w.B, MB), -1, dtype=torch.int32)
    table[:, :w.MB] = w.block_table
    for b in range(w.B):
        have = int((w.block_table[b] >= 0).sum())
        for j in range(have, need[b]):
            table[b, j] = free.pop()
    w.block_table, w.MB = table, MB
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = hz.balanced_ws(g)
    ref_pool = w.pool.clone()
    gen = torch.Generator().manual_seed(78)
    for step in range(steps):
        kn = torch.randn(w.k_new.shape, generator=gen).to(w.dtype)
        vn = torch.randn(w.v_new.shape, generator=gen).to(w.dtype)
        qn = torch.randn(w.q.shape, generator=gen).to(w.dtype)
        lens = w.lens + step
        g.k_new.copy_(kn)
        g.v_new.copy_(vn)
        g.q.copy_(qn)
        out, _ = hz.gpu_balanced(g, err, positions=lens.cuda(), ws=ws)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        flat = ref_pool.view(-1)
        oracle.kv_append(kn, vn, flat, flat[w.v_offset:], table, lens, **hz.kw(w))
        w.q = qn
        ref, _ = hz.oracle_decode(w, ref_pool, lens + 1)
        hz.assert_close(out, ref, w.dtype, f"step {step}")
    assert torch.equal(hz.int_view(g.pool.cpu()), hz.int_view(ref_pool))
    assert not hz.balanced_counters(g, ws).any()


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_balanced_bad_entries_and_lengths(H, Hkv):
    lens = [900, 900, 900, 900, 40]
    w = workloads.make_generic(B=5, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens, seed=31)
    w.block_table[1, 40] = -1            # hole deep inside the valid range
    w.block_table[2, 0] = w.NB + 3       # first block past the pool
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_lens = torch.tensor([900, 900, 900, w.MB * w.bs + 5, 40], dtype=torch.int32, device="cuda")
    out, ws = hz.gpu_balanced(g, err, lens=bad_lens)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_BLOCK and e & pa.DEVERR_BAD_LEN
    assert not out[1].any() and not out[2].any() and not out[3].any()
    assert not hz.balanced_counters(g, ws).any()
    ref, _ = hz.oracle_decode(w, w.pool, torch.tensor(lens, dtype=torch.int32))
    hz.assert_close(out[[0, 4]], ref[[0, 4]], BF16)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_balanced_fused_errors(H, Hkv):
    lens = [40, 40, 40, 47]
    w = workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens, seed=41)
    g = w.to("cuda")
    before = g.pool.clone()
    pos = torch.tensor([40, w.MB * w.bs, -1, 47], dtype=torch.int32, device="cuda")
    g.block_table[3, 2] = w.NB + 1          # target of sequence 3's append (47 // 16 = 2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, ws = hz.gpu_balanced(g, err, positions=pos)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_POS and e & pa.DEVERR_BAD_BLOCK
    assert not out[1].any() and not out[2].any() and not out[3].any()
    changed = (hz.int_view(g.pool) != hz.int_view(before)).reshape(w.NB, -1).any(1)
    assert set(torch.nonzero(changed).flatten().tolist()) == {int(w.block_table[0, 2])}
    assert not hz.balanced_counters(g, ws).any()
    ref_pool, _ = hz.oracle_append(w)
    ref, _ = hz.oracle_decode(w, ref_pool, w.lens + 1)
    hz.assert_close(out[0:1], ref[0:1], BF16)


def test_balanced_workspace_too_small_and_batch_too_large():
    w = workloads.make_generic(B=3, H=4, Hkv=4, D=64, bs=16, dtype=F16, lens=[5, 6, 7], seed=2)
    g = w.to("cuda")
    ws = hz.balanced_ws(g)
    small = ws[:ws.numel() - 16 * 16]   # short by at least one record's worth
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as ei:
        hz.gpu_balanced(g, err, lens=g.lens, ws=small)
    assert ei.value.status == pa.PA_ERR_WORKSPACE
    # a batch whose schedule tables do not fit in shared memory is rejected
    # on the host, and leaves no error behind in the CUDA runtime
    huge = hz.shape_of(w, batch=60000)
    assert pa.paged_attention_balanced_workspace(huge) == 0
    assert torch.cuda.is_available() and torch.zeros(1, device="cuda").item() == 0


def test_balanced_step_captured_in_cuda_graph():
    w = workloads.make_workload(3, batch=64, poison=True)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = hz.balanced_ws(g)
    out = torch.empty_like(g.q)
    pool0 = g.pool.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        hz.gpu_balanced(g, err, positions=g.lens, ws=ws, out=out)   # warm-up (plans, limits)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g.pool.copy_(pool0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        hz.gpu_balanced(g, err, positions=g.lens, ws=ws, out=out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert not hz.balanced_counters(g, ws).any()
    ref_pool, _ = hz.oracle_append(w)
    assert torch.equal(hz.int_view(g.pool.cpu()), hz.int_view(ref_pool))
    ref, _ = hz.oracle_decode(w, ref_pool, w.lens + 1)
    hz.assert_close(out, ref, w.dtype, "graph replay")
