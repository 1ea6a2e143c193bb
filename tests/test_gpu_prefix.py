"""GPU parity of paged_attention_decode_shared_prefix -- split-KV decode that
reads blocks shared by a group of sequences once per group -- against the
CPU oracle: the shared-beams workload at full size, groups of several sizes
(MHA and grouped-query heads) next to ungrouped sequences, partitions that
straddle the end of the shared prefix, and the device-side check of the
declared sharing."""
import pytest
import torch

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


def gpu_prefix(g, lens, ptok, err, group_first, shared_tokens):
    ws = pa.workspace_for(g.q, g.block_table, ptok, num_kv_heads=g.Hkv, **hz.kw(g))
    ws.fill_(0xFF)   # NaN pattern: a slot the reduce reads without a write shows up
    out = torch.empty_like(g.q)
    pa.paged_attention_decode_shared_prefix(out, g.q, g.k_flat(), g.v_flat(), g.block_table, lens,
                                            g.scale, ptok, ws, group_first=group_first,
                                            shared_tokens=shared_tokens, num_kv_heads=g.Hkv,
                                            err_word=err, **hz.kw(g))
    return out


def check(w, ptok, group_first, shared_tokens, *, append=True):
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if append:
        hz.gpu_append(g, g.lens, err)
        lens = g.lens + 1
    else:
        lens = g.lens
    out = gpu_prefix(g, lens, ptok, err, group_first, shared_tokens)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    if append:
        ref_pool, e = hz.oracle_append(w)
        assert not e.any()
        ref, e = hz.oracle_decode(w, ref_pool, w.lens + 1)
    else:
        ref, e = hz.oracle_decode(w, w.pool, w.lens)
    assert not e.any()
    return out, hz.assert_close(out, ref, w.dtype, w.name)


@pytest.mark.parametrize("ptok", [512, 1024, 2048])
def test_shared_beams_full_size(ptok):
    w = workloads.make_workload(5, poison=True)
    shared = w.meta["shared_blocks"] * w.bs
    check(w, ptok, [0, w.B], [shared])


@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(4, 4, BF16, 128, 16), (16, 2, F16, 128, 16),
                                              (8, 8, BF16, 64, 32), (16, 4, BF16, 128, 8),
                                              (4, 2, F16, 64, 256)])
@pytest.mark.parametrize("ptok", [16, 64, 256])
def test_groups_next_to_ungrouped_sequences(H, Hkv, dtype, D, bs, ptok):
    g = H // Hkv
    big = max(1, min(4, 16 // g))
    sizes = [big, 1, 2, 1]
    w = workloads.make_prefix_groups(group_sizes=sizes, shared_blocks=[600 // bs + 1, 0, 300 // bs, 2],
                                     tails=[3, 17, 40, 9, 0, 33, 5, 71][:sum(sizes)], H=H, Hkv=Hkv, D=D,
                                     bs=bs, dtype=dtype, seed=H + D + bs)
    check(w, ptok, w.meta["group_first"], w.meta["shared_tokens"])


def test_equals_the_plain_split_pair():
    w = workloads.make_prefix_groups(group_sizes=[4, 3], shared_blocks=[40, 25], tails=[5, 9, 100, 0, 31, 64, 2],
                                     H=32, Hkv=32, D=128, bs=16, dtype=BF16, seed=3)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = gpu_prefix(g, g.lens, 128, err, w.meta["group_first"], w.meta["shared_tokens"])
    b, _ = hz.gpu_split(g, g.lens, 128, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hz.assert_close(a, b.double().cpu().numpy(), BF16)


def test_declared_sharing_is_checked():
    """A member whose table leaves the shared blocks, or whose length does not
    cover the declared prefix, turns its group's outputs to zeros with
    PA_DEVERR_BAD_PREFIX; other groups are unaffected."""
    w = workloads.make_prefix_groups(group_sizes=[3, 2], shared_blocks=[20, 20], tails=[5, 9, 7, 3, 4],
                                     H=4, Hkv=4, D=128, bs=16, dtype=BF16, seed=4, poison=False)
    g = w.to("cuda")
    # group 0: member 1 names a different (valid) block inside the prefix
    g.block_table[1, 3] = g.block_table[3, 3]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_prefix(g, g.lens, 64, err, w.meta["group_first"], w.meta["shared_tokens"])
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_PREFIX
    assert not out[0:3].any()
    ref, _ = hz.oracle_decode(w, w.pool, w.lens)
    hz.assert_close(out[3:5], ref[3:5], BF16)
    # group 1 declares more shared tokens than member 4 holds
    g2 = w.to("cuda")
    err.zero_()
    lens = g2.lens.clone()
    lens[4] = 100
    out = gpu_prefix(g2, lens, 64, err, w.meta["group_first"], w.meta["shared_tokens"])
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BAD_PREFIX
    assert not out[3:5].any()
    hz.assert_close(out[0:3], ref[0:3], BF16)


def test_rejects_what_it_cannot_run():
    w = workloads.make_prefix_groups(group_sizes=[5], shared_blocks=[4], tails=[1, 2, 3, 4, 5],
                                     H=8, Hkv=2, D=128, bs=16, dtype=BF16, seed=5)
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as ei:   # 5 members x 4 heads > 16 columns
        gpu_prefix(g, g.lens, 64, err, [0, 5], [64])
    assert ei.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PagedAttnError) as ei:   # not ascending
        gpu_prefix(g, g.lens, 64, err, [0, 3, 2], [64, 0])
    assert ei.value.status == pa.PA_ERR_INVALID_ARG
