"""GPU parity of the paths around the decode step: the multi-token (prefill)
write, sliding-window decode, and the step captured in a CUDA graph."""
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


# ---------------------------------------------------------------------------
# prefill write: paged_kv_append_tokens
# ---------------------------------------------------------------------------

def _prefill_case(dtype, bs, D=64, Hkv=2, seed=0):
    counts = torch.tensor([0, 1, 15, 16, 17, 70], dtype=torch.int32)
    starts = torch.tensor([5, 0, 3, 16, 31, 2], dtype=torch.int32)
    B, T = len(counts), int(counts.max()) + 3
    g = torch.Generator().manual_seed(seed)
    kn = torch.randn(B, T, Hkv, D, generator=g).to(dtype)
    vn = torch.randn(B, T, Hkv, D, generator=g).to(dtype)
    for b in range(B):          # padding rows: must never reach the cache
        kn[b, counts[b]:] = float("nan")
        vn[b, counts[b]:] = float("nan")
    nblk = [-(-(int(s) + int(c)) // bs) for s, c in zip(starts, counts)]
    MB = max(nblk) + 1
    NB = sum(nblk) + 5
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    table = torch.full((B, MB), -1, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[cur:cur + n]
        cur += n
    pool = torch.randn(NB, 2, Hkv, bs, D, generator=g).to(dtype)
    return dict(kn=kn, vn=vn, counts=counts, starts=starts, table=table, pool=pool, NB=NB, bs=bs,
                Hkv=Hkv, D=D, stride=2 * Hkv * bs * D)


@pytest.mark.parametrize("dtype,bs", [(F32, 16), (F16, 1), (BF16, 3), (BF16, 16), (F16, 64)])
def test_prefill_write_bit_exact(dtype, bs):
    c = _prefill_case(dtype, bs, seed=bs)
    ref = c["pool"].clone()
    flat = ref.view(-1)
    kw = dict(block_size=bs, block_stride=c["stride"], num_blocks=c["NB"])
    e = oracle.kv_append_tokens(c["kn"], c["vn"], flat, flat[c["Hkv"] * bs * c["D"]:], c["table"],
                                c["starts"], c["counts"], **kw)
    assert not e.any()
    pool = c["pool"].cuda()
    gflat = pool.view(-1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.paged_kv_append_tokens(c["kn"].cuda(), c["vn"].cuda(), gflat, gflat[c["Hkv"] * bs * c["D"]:],
                              c["table"].cuda(), c["starts"].cuda(), c["counts"].cuda(),
                              err_word=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(hz.int_view(pool.cpu()), hz.int_view(ref))


def test_prefill_write_flags():
    c = _prefill_case(BF16, 16, seed=3)
    c["counts"][0] = c["kn"].shape[1] + 1          # more tokens than the padded batch holds
    c["starts"][1] = c["table"].shape[1] * 16       # past the table row
    c["table"][5, 2] = c["NB"] + 4                  # one target block past the pool
    ref = c["pool"].clone()
    flat = ref.view(-1)
    kw = dict(block_size=16, block_stride=c["stride"], num_blocks=c["NB"])
    e = oracle.kv_append_tokens(c["kn"], c["vn"], flat, flat[c["Hkv"] * 16 * c["D"]:], c["table"],
                                c["starts"], c["counts"], **kw)
    assert e[0] == oracle.SEQ_BAD_LEN and e[1] == oracle.SEQ_BAD_POS and e[5] == oracle.SEQ_BAD_BLOCK
    pool = c["pool"].cuda()
    gflat = pool.view(-1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.paged_kv_append_tokens(c["kn"].cuda(), c["vn"].cuda(), gflat, gflat[c["Hkv"] * 16 * c["D"]:],
                              c["table"].cuda(), c["starts"].cuda(), c["counts"].cuda(),
                              err_word=err, **kw)
    torch.cuda.synchronize()
    got = int(err.item())
    assert got & pa.DEVERR_BAD_LEN and got & pa.DEVERR_BAD_POS and got & pa.DEVERR_BAD_BLOCK
    assert torch.equal(hz.int_view(pool.cpu()), hz.int_view(ref))


@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 2)])
def test_prefill_then_decode(H, Hkv):
    """Write whole prompts into an empty paged cache, then decode over them."""
    lens = [1, 40, 333, 90]
    B, D, bs = len(lens), 128, 16
    T = max(lens)
    g = torch.Generator().manual_seed(H)
    kn = torch.randn(B, T, Hkv, D, generator=g).to(BF16)
    vn = torch.randn(B, T, Hkv, D, generator=g).to(BF16)
    w = workloads.make_generic(B=B, H=H, Hkv=Hkv, D=D, bs=bs, dtype=BF16, lens=lens, seed=H,
                               poison=True)
    g_ = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts = torch.tensor(lens, dtype=torch.int32)
    pa.paged_kv_append_tokens(kn.cuda(), vn.cuda(), g_.k_flat(), g_.v_flat(), g_.block_table,
                              torch.zeros(B, dtype=torch.int32, device="cuda"), counts.cuda(),
                              err_word=err, **hz.kw(w))
    out = hz.gpu_decode(g_, counts.cuda(), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = np.zeros((B, H, D))
    for b in range(B):
        for h in range(H):
            ref[b, h] = oracle.attention_contiguous(w.q[b, h].double().numpy(),
                                                    kn[b, :lens[b], h // (H // Hkv)].double().numpy(),
                                                    vn[b, :lens[b], h // (H // Hkv)].double().numpy(),
                                                    w.scale)
    hz.assert_close(out, ref, BF16)


# ---------------------------------------------------------------------------
# sliding-window decode
# ---------------------------------------------------------------------------

WIN_LENS = [1, 5, 16, 17, 100, 700, 2049]


def _poison_before_window(w, window, grain):
    """Poison every block that ends at or before the first row a kernel may
    fetch (the window start rounded down to `grain`)."""
    bad = float("nan")
    for b in range(w.B):
        L = int(w.lens[b])
        first = (max(0, L - window) // grain) * grain
        for j in range(first // w.bs):
            w.pool[int(w.block_table[b, j])] = bad


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(4, 4, F16, 128, 16), (2, 2, F32, 64, 8),
                                              (16, 2, BF16, 128, 16), (8, 1, F16, 64, 32),
                                              (8, 2, BF16, 128, 4)])
@pytest.mark.parametrize("window", [1, 13, 16, 100, 5000])
def test_window_decode(H, Hkv, dtype, D, bs, window):
    w = workloads.make_generic(B=len(WIN_LENS), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype,
                               lens=WIN_LENS, seed=window + H)
    _poison_before_window(w, window, 16)
    ref, e = oracle.attention_decode_window(w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens,
                                            w.scale, window, num_kv_heads=Hkv, **hz.kw(w))
    assert not e.any()
    g = w.to("cuda")
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.paged_attention_decode_window(out, g.q, g.k_flat(), g.v_flat(), g.block_table, g.lens,
                                     w.scale, window, num_kv_heads=Hkv, err_word=err, **hz.kw(w))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hz.assert_close(out, ref, dtype, f"window {window}")


def test_window_equals_full_decode_when_wide():
    w = workloads.make_workload(4, batch=3, max_len=700).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    full = hz.gpu_decode(w, w.lens, err)
    out = torch.empty_like(w.q)
    pa.paged_attention_decode_window(out, w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens,
                                     w.scale, 1 << 20, num_kv_heads=w.Hkv, err_word=err, **hz.kw(w))
    torch.cuda.synchronize()
    assert torch.equal(full, out)


# ---------------------------------------------------------------------------
# the step in a CUDA graph
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("index,mode", [(2, "fused"), (4, "fused"), (2, "unfused"), (5, "split")])
def test_step_captured_in_cuda_graph(index, mode):
    """Capture one step (append + decode, positions += 1) and replay it for
    several tokens; the pool and the last output match the oracle."""
    steps = 6
    kwargs = {"batch": 4} if index in (2, 4) else {"max_len": 3000}
    w = workloads.make_workload(index, poison=True, **kwargs)
    # room for `steps` more tokens per sequence
    used = set(int(x) for x in w.block_table.flatten() if x >= 0)
    free = [i for i in range(w.NB) if i not in used]
    need = [-(-(int(L) + steps) // w.bs) for L in w.lens]
    MB = max(max(need) + 1, w.MB)
    table = torch.full((w.B, MB), -1, dtype=torch.int32)
    table[:, :w.MB] = w.block_table
    for b in range(w.B):
        have = int((w.block_table[b] >= 0).sum())
        for j in range(have, need[b]):
            table[b, j] = free.pop()
    w.block_table, w.MB = table, MB
    g = w.to("cuda")
    pos = g.lens.clone()
    lens_after = pos + 1
    out = torch.empty_like(g.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pa.workspace_for(g.q, g.block_table, 1024, num_kv_heads=g.Hkv, **hz.kw(g)) \
        if mode == "split" else None

    def step():
        if mode == "fused":
            pa.paged_attention_decode_append(out, g.q, g.k_new, g.v_new, g.k_flat(), g.v_flat(),
                                             g.block_table, pos, g.scale, num_kv_heads=g.Hkv,
                                             err_word=err, **hz.kw(g))
        else:
            pa.paged_kv_append(g.k_new, g.v_new, g.k_flat(), g.v_flat(), g.block_table, pos,
                               err_word=err, **hz.kw(g))
            torch.add(pos, 1, out=lens_after)
            if mode == "unfused":
                pa.paged_attention_decode(out, g.q, g.k_flat(), g.v_flat(), g.block_table,
                                          lens_after, g.scale, num_kv_heads=g.Hkv, err_word=err,
                                          **hz.kw(g))
            else:
                pa.paged_attention_decode_partial(g.q, g.k_flat(), g.v_flat(), g.block_table,
                                                  lens_after, g.scale, 1024, ws,
                                                  num_kv_heads=g.Hkv, err_word=err, **hz.kw(g))
                pa.paged_attention_decode_reduce(out, ws, lens_after, 1024, num_kv_heads=g.Hkv,
                                                 max_blocks_per_seq=g.MB, err_word=err, **hz.kw(g))
        pos.add_(1)

    # warm up outside the capture (lazy module loading, function attributes)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    pos.copy_(g.lens)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    ref_pool = w.pool.clone()
    gen = torch.Generator().manual_seed(5)
    for s in range(steps):
        kn = torch.randn(w.k_new.shape, generator=gen).to(w.dtype)
        vn = torch.randn(w.v_new.shape, generator=gen).to(w.dtype)
        g.k_new.copy_(kn)
        g.v_new.copy_(vn)
        graph.replay()
        flat = ref_pool.view(-1)
        oracle.kv_append(kn, vn, flat, flat[w.v_offset:], table, w.lens + s, **hz.kw(w))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(hz.int_view(g.pool.cpu()), hz.int_view(ref_pool))
    ref, _ = hz.oracle_decode(w, ref_pool, w.lens + steps)
    hz.assert_close(out, ref, w.dtype, f"graph {mode}")
