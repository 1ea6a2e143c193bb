"""GPU edge cases: shapes off the five workloads (every compiled head_dim and
dtype, GQA group sizes, block sizes, separate K/V pools), empty and
single-token sequences, and the device-side error handling (bad table
entries, lengths past the table row, bad append positions), which must
report through err_word and never trap."""
import numpy as np
import pytest
import torch

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


LENS = [0, 1, 15, 16, 17, 31, 33, 64, 100, 257]   # pre-append lengths: ragged tails


@pytest.mark.parametrize("dtype,D", [(F32, 16), (F32, 32), (F32, 64), (F32, 128),
                                     (F16, 32), (F16, 64), (F16, 128), (F16, 256),
                                     (BF16, 32), (BF16, 64), (BF16, 128), (BF16, 256)])
def test_mha_every_head_dim(dtype, D):
    w = workloads.make_generic(B=len(LENS), H=3, Hkv=3, D=D, bs=16, dtype=dtype, lens=LENS,
                               seed=D)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("bs", [1, 3, 8, 24, 32, 128])
def test_mha_block_sizes(bs):
    w = workloads.make_generic(B=len(LENS), H=2, Hkv=2, D=128, bs=bs, dtype=BF16, lens=LENS, seed=bs)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("H,Hkv", [(8, 4), (16, 4), (16, 1), (32, 1), (48, 2)])
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_gqa_group_sizes_tensor_path(H, Hkv, dtype):
    w = workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=128, bs=16, dtype=dtype, lens=LENS,
                               seed=H * 7 + Hkv)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_TENSOR_GQA
    hz.run_step_and_check(w)


@pytest.mark.parametrize("D,bs", [(64, 16), (128, 8), (128, 32), (64, 256)])
def test_gqa_head_dims_and_blocks(D, bs):
    w = workloads.make_generic(B=len(LENS), H=16, Hkv=2, D=D, bs=bs, dtype=BF16, lens=LENS,
                               seed=D + bs)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_TENSOR_GQA
    hz.run_step_and_check(w)
    hz.run_step_and_check(w, split_ptok=32)


@pytest.mark.parametrize("dtype,D,bs", [(F32, 64, 16), (BF16, 256, 16), (BF16, 128, 4)])
def test_gqa_on_the_simt_path(dtype, D, bs):
    w = workloads.make_generic(B=len(LENS), H=8, Hkv=2, D=D, bs=bs, dtype=dtype, lens=LENS, seed=3)
    assert pa.paged_attention_decode_path(hz.shape_of(w)) == pa.PA_PATH_SIMT
    hz.run_step_and_check(w)


@pytest.mark.parametrize("H,Hkv,dtype", [(4, 4, F16), (8, 2, BF16), (4, 4, F32)])
def test_separate_k_and_v_pools(H, Hkv, dtype):
    w = workloads.make_generic(B=len(LENS), H=H, Hkv=Hkv, D=64, bs=16, dtype=dtype, lens=LENS,
                               seed=11, separate_pools=True)
    hz.run_step_and_check(w)
    hz.run_step_and_check(w, split_ptok=16)


def _decode_only(w, lens, *, split=None, err_word=True):
    g = w.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda") if err_word else None
    lens_d = torch.as_tensor(lens, dtype=torch.int32).cuda()
    if split is None:
        out = hz.gpu_decode(g, lens_d, err)
    else:
        out, _ = hz.gpu_split(g, lens_d, split, err)
    torch.cuda.synchronize()
    return out, (int(err.item()) if err_word else None)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
@pytest.mark.parametrize("split", [None, 16])
def test_zero_length_sequences_give_zeros(H, Hkv, split):
    w = workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=[0, 20, 0, 5],
                               seed=5)
    out, err = _decode_only(w, [0, 20, 0, 5], split=split)
    assert err == 0
    assert not out[0].any() and not out[2].any()
    ref, _ = hz.oracle_decode(w, w.pool, torch.tensor([0, 20, 0, 5], dtype=torch.int32))
    hz.assert_close(out, ref, BF16)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
@pytest.mark.parametrize("split", [None, 32])
def test_bad_table_entries_are_reported_and_zeroed(H, Hkv, split):
    lens = [40, 40, 40, 40]
    w = workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens, seed=9)
    w.block_table[1, 1] = -1             # hole inside the valid range
    w.block_table[2, 2] = w.NB           # id past the pool
    w.block_table[0, 3:] = -1            # past ceil(40/16) = 3: never read
    out, err = _decode_only(w, lens, split=split)
    assert err & pa.DEVERR_BAD_BLOCK
    assert not out[1].any() and not out[2].any()
    ref, e = hz.oracle_decode(w, w.pool, torch.tensor(lens, dtype=torch.int32))
    assert list(e) == [0, 2, 2, 0]
    hz.assert_close(out[[0, 3]], ref[[0, 3]], BF16)


@pytest.mark.parametrize("split", [None, 16])
def test_length_past_table_row_is_reported(split):
    w = workloads.make_generic(B=3, H=4, Hkv=4, D=64, bs=16, dtype=F16, lens=[10, 10, 10], seed=1)
    too_long = w.MB * w.bs + 1
    out, err = _decode_only(w, [10, too_long, -3], split=split)
    assert err & pa.DEVERR_BAD_LEN
    assert not out[1].any() and not out[2].any()
    ref, _ = hz.oracle_decode(w, w.pool, torch.tensor([10, 0, 0], dtype=torch.int32))
    hz.assert_close(out[0:1], ref[0:1], F16)


def test_null_err_word_is_allowed():
    w = workloads.make_generic(B=2, H=4, Hkv=4, D=64, bs=16, dtype=F16, lens=[10, 10], seed=2)
    w.block_table[0, 0] = -5
    out, _ = _decode_only(w, [10, 10], err_word=False)
    assert not out[0].any() and out[1].abs().sum() > 0


def test_append_reports_bad_position_and_block():
    w = workloads.make_generic(B=4, H=4, Hkv=2, D=64, bs=16, dtype=BF16, lens=[3, 3, 3, 3], seed=4)
    g = w.to("cuda")
    before = g.pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.tensor([3, w.MB * w.bs, -1, 3], dtype=torch.int32, device="cuda")
    g.block_table[3, 0] = w.NB + 10
    hz.gpu_append(g, pos, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_POS and e & pa.DEVERR_BAD_BLOCK
    changed = (hz.int_view(g.pool) != hz.int_view(before)).reshape(w.NB, -1).any(1)
    touched = set(torch.nonzero(changed).flatten().tolist())
    assert touched == {int(w.block_table[0, 0])}   # only sequence 0 wrote


def test_output_guard_canaries_untouched():
    w = workloads.make_generic(B=5, H=8, Hkv=2, D=128, bs=16, dtype=BF16, lens=[7, 0, 70, 16, 1],
                               seed=6)
    g = w.to("cuda")
    n = w.B * w.H * w.D
    buf = torch.full((n + 2048,), 7.25, dtype=BF16, device="cuda")
    out = buf[1024:1024 + n].view(w.B, w.H, w.D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hz.gpu_decode(g, g.lens, err, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 7.25) and torch.all(buf[1024 + n:] == 7.25)
    ref, _ = hz.oracle_decode(w, w.pool, w.lens)
    hz.assert_close(out, ref, BF16)


def test_empty_batch_is_a_no_op():
    w = workloads.make_generic(B=2, H=4, Hkv=4, D=64, bs=16, dtype=F16, lens=[3, 3], seed=8)
    g = w.to("cuda")
    empty_q = g.q[:0]
    out = torch.empty_like(empty_q)
    pa.paged_attention_decode(out, empty_q, g.k_flat(), g.v_flat(), g.block_table[:0], g.lens[:0],
                              0.1, num_kv_heads=4, **hz.kw(g))
    torch.cuda.synchronize()


def test_huge_scores_stay_finite():
    """Scores of +-1e4 after scaling: the running max keeps exp2 in range."""
    w = workloads.make_generic(B=3, H=4, Hkv=4, D=64, bs=16, dtype=BF16, lens=[50, 200, 3],
                               seed=12, poison=True)
    w.q *= 100.0
    hz.run_step_and_check(w)


# Few sequences with long contexts: the single-pass decode spreads each
# (sequence, head) unit over a thread-block cluster and merges the CTAs'
# partial softmax states through distributed shared memory.
CLUSTER_LENS = [0, 1500, 37, 700, 1]


@pytest.mark.parametrize("H,Hkv,dtype", [(4, 4, F16), (2, 2, F32), (16, 2, BF16), (8, 1, F16)])
def test_cluster_split_single_pass(H, Hkv, dtype):
    w = workloads.make_generic(B=len(CLUSTER_LENS), H=H, Hkv=Hkv, D=128 if dtype != F32 else 64,
                               bs=16, dtype=dtype, lens=CLUSTER_LENS, seed=21 + H)
    hz.run_step_and_check(w)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_cluster_split_bad_entries_and_lengths(H, Hkv):
    lens = [900, 900, 900, 900]
    w = workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens, seed=31)
    w.block_table[1, 40] = -1            # hole deep inside the valid range
    w.block_table[2, 0] = w.NB + 3       # first block past the pool
    out, err = _decode_only(w, [900, 900, 900, w.MB * w.bs + 5])
    assert err & pa.DEVERR_BAD_BLOCK and err & pa.DEVERR_BAD_LEN
    assert not out[1].any() and not out[2].any() and not out[3].any()
    ref, _ = hz.oracle_decode(w, w.pool, torch.tensor(lens, dtype=torch.int32))
    hz.assert_close(out[0:1], ref[0:1], BF16)



@pytest.mark.parametrize("H,Hkv,dtype,D,bs", [(3, 3, F32, 64, 16), (4, 4, F16, 128, 8),
                                              (16, 2, BF16, 128, 16), (8, 2, BF16, 64, 32),
                                              (8, 2, F32, 64, 4), (4, 4, BF16, 256, 3)])
@pytest.mark.parametrize("lens", [LENS, CLUSTER_LENS])
def test_fused_append_decode_shapes(H, Hkv, dtype, D, bs, lens):
    w = workloads.make_generic(B=len(lens), H=H, Hkv=Hkv, D=D, bs=bs, dtype=dtype, lens=lens,
                               seed=H + D + bs)
    hz.run_fused_step_and_check(w)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (16, 2)])
def test_fused_append_decode_errors(H, Hkv):
    lens = [40, 40, 40, 47]
    w = workloads.make_generic(B=4, H=H, Hkv=Hkv, D=128, bs=16, dtype=BF16, lens=lens, seed=41)
    g = w.to("cuda")
    before = g.pool.clone()
    pos = torch.tensor([40, w.MB * w.bs, -1, 47], dtype=torch.int32, device="cuda")
    g.block_table[3, 2] = w.NB + 1          # target of sequence 3's append (47 // 16 = 2)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = hz.gpu_fused(g, pos, err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & pa.DEVERR_BAD_POS and e & pa.DEVERR_BAD_BLOCK
    assert not out[1].any() and not out[2].any() and not out[3].any()
    changed = (hz.int_view(g.pool) != hz.int_view(before)).reshape(w.NB, -1).any(1)
    assert set(torch.nonzero(changed).flatten().tolist()) == {int(w.block_table[0, 2])}
    ref_pool, _ = hz.oracle_append(w)
    ref, _ = hz.oracle_decode(w, ref_pool, w.lens + 1)
    hz.assert_close(out[0:1], ref[0:1], BF16)


@pytest.mark.parametrize("H,Hkv,dtype", [(8, 8, F16), (16, 2, BF16)])
def test_pool_alignment_128_expected_16_required(H, Hkv, dtype):
    """Device pools start on a 128-byte boundary ("KV Block design" s3.7);
    a pool moved to a 16- but not 128-byte aligned address (allowed, slower)
    gives bit-identical results, and a pool off the 16-byte rule is refused
    before anything runs."""
    w = workloads.make_generic(B=3, H=H, Hkv=Hkv, D=128, bs=16, dtype=dtype, lens=[70, 5, 300],
                               seed=51, poison=True)
    g = w.to("cuda")
    assert g.pool.data_ptr() % 128 == 0
    out = hz.gpu_decode(g, g.lens, torch.zeros(1, dtype=torch.int32, device="cuda"))
    es = g.pool.element_size()
    n = g.pool.numel()
    buf = torch.empty(n + 64 // es, dtype=dtype, device="cuda")
    off = 16 // es                                      # 16 bytes past a 512-byte boundary
    shifted = buf[off:off + n]
    shifted.copy_(g.pool.view(-1))
    assert shifted.data_ptr() % 128 == 16
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(g.q)
    pa.paged_attention_decode(out2, g.q, shifted, shifted[w.v_offset:], g.block_table, g.lens, g.scale,
                              num_kv_heads=Hkv, err_word=err, **hz.kw(g))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(hz.int_view(out), hz.int_view(out2))
    ref, _ = hz.oracle_decode(w, w.pool, w.lens)
    hz.assert_close(out2, ref, dtype)
    bad = buf[off + 1:off + 1 + n - 8]                  # 2 bytes off: breaks the 16-byte rule
    with pytest.raises(pa.PagedAttnError) as e:
        pa.paged_attention_decode(out2, g.q, bad, bad[w.v_offset:], g.block_table, g.lens, g.scale,
                                  num_kv_heads=Hkv, **hz.kw(g))
    assert e.value.status == pa.PA_ERR_MISALIGNED
