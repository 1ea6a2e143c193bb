"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test pins one part of oracle/pa_oracle.c to something other than
itself: a worked example or byte count printed on the pages (fixtures under
tests/golden/), a library routine (numpy's binary16 decoder, torch's bfloat16
decoder, torch's scaled_dot_product_attention in float64), a closed form, an
invariant of paging (relabelling physical blocks changes nothing), or brute
force on tiny inputs.  test_planted_mistakes_are_caught compiles copies of the
oracle with plausible bugs planted and checks that this battery fails each.
"""
import json
import math
import os
import subprocess
import sys
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# test-side helpers (independent of the oracle)
# ---------------------------------------------------------------------------

def scatter_to_pool(K, V, bs, NB, rng, dtype=np.float32, layout="colocated"):
    """Lay contiguous K/V [B][Hkv][L][D] into a paged pool.

    Returns (k_pool flat, v_pool flat, table [B][MB], block_stride).  Unused
    slots are NaN so that reading one poisons the result.
    """
    B, Hkv, L, D = K.shape
    nblk = -(-L // bs)
    MB = nblk + 1
    perm = rng.permutation(NB)
    table = np.full((B, MB), -1, dtype=np.int32)
    for b in range(B):
        table[b, :nblk] = perm[b * nblk:(b + 1) * nblk]
    if layout == "colocated":
        pool = np.full((NB, 2, Hkv, bs, D), np.nan, dtype=dtype)
        kp, vp = pool[:, 0], pool[:, 1]
        stride = 2 * Hkv * bs * D
    else:
        kp = np.full((NB, Hkv, bs, D), np.nan, dtype=dtype)
        vp = np.full((NB, Hkv, bs, D), np.nan, dtype=dtype)
        stride = Hkv * bs * D
    for b in range(B):
        for t in range(L):
            blk, slot = table[b, t // bs], t % bs
            kp[blk, :, slot, :] = K[b, :, t, :]
            vp[blk, :, slot, :] = V[b, :, t, :]
    if layout == "colocated":
        flat = pool.reshape(-1)
        return flat, flat[Hkv * bs * D:], table, stride
    return kp.reshape(-1), vp.reshape(-1), table, stride


def sdpa_reference(q, K, V, lens, scale):
    """torch SDPA in float64 on contiguous K/V, GQA heads mapped h -> h // g."""
    B, H, D = q.shape
    Hkv = K.shape[1]
    g = H // Hkv
    out = np.zeros((B, H, D))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        qb = torch.from_numpy(q[b]).double()[:, None, :]                  # [H][1][D]
        kb = torch.from_numpy(K[b, :, :L]).double().repeat_interleave(g, 0)  # [H][L][D]
        vb = torch.from_numpy(V[b, :, :L]).double().repeat_interleave(g, 0)
        o = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


def numpy_softmax_reference(q, K, V, lens, scale):
    """Explicit full softmax with numpy (no max subtraction; tiny inputs)."""
    B, H, D = q.shape
    g = H // K.shape[1]
    out = np.zeros((B, H, D))
    for b in range(B):
        L = int(lens[b])
        for h in range(H):
            if L == 0:
                continue
            s = (K[b, h // g, :L] @ q[b, h]) * scale
            e = np.exp(s)
            out[b, h] = (e[:, None] * V[b, h // g, :L]).sum(0) / e.sum()
    return out


def tiny_case(rng, B=3, H=4, Hkv=2, D=16, Lmax=40, bs=8, dtype=np.float32, lens=None):
    if lens is None:
        lens = rng.integers(1, Lmax + 1, size=B)
    lens = np.asarray(lens, dtype=np.int32)
    L = int(lens.max())
    K = rng.standard_normal((B, Hkv, L, D)).astype(dtype)
    V = rng.standard_normal((B, Hkv, L, D)).astype(dtype)
    q = rng.standard_normal((B, H, D)).astype(dtype)
    nblk = -(-L // bs)
    NB = B * nblk + 5
    kp, vp, table, stride = scatter_to_pool(K, V, bs, NB, rng, dtype=dtype)
    return dict(q=q, K=K, V=V, lens=lens, kp=kp, vp=vp, table=table, stride=stride,
                NB=NB, bs=bs, Hkv=Hkv, D=D)


def run_decode(c, scale, **kw):
    return oracle.attention_decode(c["q"], c["kp"], c["vp"], c["table"], c["lens"], scale,
                                   num_kv_heads=c["Hkv"], block_size=c["bs"],
                                   block_stride=c["stride"], num_blocks=c["NB"], **kw)


# ---------------------------------------------------------------------------
# worked examples and byte counts printed on the pages
# ---------------------------------------------------------------------------

def test_blocks_needed_worked_example():
    g = _golden("blockmanager_example.json")
    got = [oracle.blocks_needed(L, g["block_size"]) for L in g["lengths"]]
    assert got == g["expected_blocks"]
    assert sum(g["lengths"]) == g["total_tokens"]
    assert got[1] == len(g["request2_block_ids"])


def test_blocks_needed_edges():
    assert oracle.blocks_needed(0, 16) == 0
    assert oracle.blocks_needed(1, 16) == 1
    assert oracle.blocks_needed(16, 16) == 1
    assert oracle.blocks_needed(17, 16) == 2
    # the 450..520-token window of the block-size section: 29..33 blocks of
    # 16 and 8..9 blocks of 64 (the page's "28-33" and "7-8" are misprints
    # of these ceilings)
    assert oracle.blocks_needed(450, 16) == 29 and oracle.blocks_needed(520, 16) == 33
    assert oracle.blocks_needed(450, 64) == 8 and oracle.blocks_needed(520, 64) == 9


def test_kv_byte_counts_from_pages():
    g = _golden("byte_counts.json")
    t = g["per_token"]
    assert oracle.kv_bytes(1, t["heads"], 1, t["head_dim"], t["dtype_bytes"]) == t["bytes"]
    blk = g["per_block_all_layers"]
    assert blk["layers"] * oracle.kv_bytes(1, blk["heads"], blk["block_size"], blk["head_dim"],
                                           blk["dtype_bytes"]) == blk["bytes"]
    c = g["contiguous_prealloc_7b"]
    assert c["layers"] * oracle.kv_bytes(c["batch"], c["heads"], c["max_seq_len"], c["head_dim"],
                                         c["dtype_bytes"]) == c["bytes"]


def test_kv_bytes_counts_the_gathered_elements():
    """The formula equals the bytes actually gathered for K and V."""
    rng = np.random.default_rng(5)
    c = tiny_case(rng, B=3, H=2, Hkv=2, D=8, lens=[5, 17, 9], bs=4)
    gathered = 0
    for b in range(3):
        for hk in range(2):
            Kc, Vc = oracle.gather(c["kp"], c["vp"], c["table"][b], hk, int(c["lens"][b]),
                                   block_size=4, head_dim=8, num_kv_heads=2,
                                   block_stride=c["stride"])
            gathered += (Kc.size + Vc.size) * 4
    per_seq = sum(oracle.kv_bytes(1, 2, int(L), 8, 4) for L in c["lens"])
    assert per_seq == gathered


# ---------------------------------------------------------------------------
# element decoding against library decoders
# ---------------------------------------------------------------------------

def test_f16_decoder_matches_numpy_on_every_code():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = oracle.to_double(codes.view(np.float16))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_matches_torch_on_every_code():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    ref = codes.double().numpy()
    got = oracle.to_double(codes.contiguous())
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f32_decoder_is_exact():
    x = np.random.default_rng(1).standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.to_double(x), x.astype(np.float64))


# ---------------------------------------------------------------------------
# brute force against library attention on tiny inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 1)])
@pytest.mark.parametrize("bs", [1, 3, 8, 16])
def test_decode_matches_sdpa_float64(H, Hkv, bs):
    rng = np.random.default_rng(100 + 10 * H + Hkv + bs)
    c = tiny_case(rng, B=4, H=H, Hkv=Hkv, D=16, Lmax=40, bs=bs)
    scale = 1.0 / math.sqrt(16)
    out, err = run_decode(c, scale)
    assert not err.any()
    ref = sdpa_reference(c["q"].astype(np.float64), c["K"].astype(np.float64),
                         c["V"].astype(np.float64), c["lens"], scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    ref2 = numpy_softmax_reference(c["q"].astype(np.float64), c["K"].astype(np.float64),
                                   c["V"].astype(np.float64), c["lens"], scale)
    np.testing.assert_allclose(out, ref2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_16bit_inputs_match_sdpa(dtype):
    rng = np.random.default_rng(7)
    c = tiny_case(rng, B=3, H=4, Hkv=2, D=16, Lmax=33, bs=8)
    tdt = workloads.DTYPES[dtype]
    # round the inputs to the 16-bit type, decode them with torch (not the oracle)
    for key in ("q", "K", "V"):
        c[key] = torch.from_numpy(c[key]).to(tdt)
    qd, Kd, Vd = (c[k].double().numpy() for k in ("q", "K", "V"))
    kp, vp, table, stride = scatter_to_pool(Kd, Vd, 8, c["NB"], rng, dtype=np.float64)
    pool16 = torch.from_numpy(np.ascontiguousarray(kp.reshape(c["NB"], 2, 2, 8, 16))).to(tdt)
    flat = pool16.reshape(-1)
    scale = 0.25
    out, err = oracle.attention_decode(c["q"].contiguous(), flat, flat[2 * 8 * 16:], table,
                                       c["lens"], scale, num_kv_heads=2, block_size=8,
                                       block_stride=stride, num_blocks=c["NB"])
    assert not err.any()
    ref = sdpa_reference(qd, Kd, Vd, c["lens"], scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_single_token_returns_v0_exactly():
    rng = np.random.default_rng(11)
    c = tiny_case(rng, B=2, H=2, Hkv=2, D=16, lens=[1, 1], bs=4)
    out, _ = run_decode(c, 0.3)
    for b in range(2):
        for h in range(2):
            assert np.array_equal(out[b, h], c["V"][b, h, 0].astype(np.float64))


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(12)
    c = tiny_case(rng, B=2, H=2, Hkv=2, D=16, lens=[7, 30], bs=8)
    c["q"][:] = 0
    out, _ = run_decode(c, 1.0)
    for b in range(2):
        L = int(c["lens"][b])
        for h in range(2):
            np.testing.assert_allclose(out[b, h], c["V"][b, h, :L].astype(np.float64).mean(0),
                                       rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(13)
    c = tiny_case(rng, B=1, H=1, Hkv=1, D=8, lens=[19], bs=4)
    K = np.repeat(c["K"][:, :, :1], 19, axis=2)
    kp, vp, table, stride = scatter_to_pool(K, c["V"], 4, c["NB"], rng)
    c.update(kp=kp, vp=vp, table=table, stride=stride)
    out, _ = run_decode(c, 0.7)
    np.testing.assert_allclose(out[0, 0], c["V"][0, 0].astype(np.float64).mean(0), atol=1e-13)


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(14)
    c = tiny_case(rng, B=2, H=2, Hkv=1, D=8, lens=[3, 25], bs=4)
    V = np.full_like(c["V"], 0.625)
    kp, vp, table, stride = scatter_to_pool(c["K"], V, 4, c["NB"], rng)
    c.update(kp=kp, vp=vp, table=table, stride=stride)
    out, _ = run_decode(c, 0.5)
    np.testing.assert_allclose(out, 0.625, rtol=0, atol=1e-14)


def test_score_shift_invariance():
    """Adding u to every key adds scale*q.u to every score: output unchanged."""
    rng = np.random.default_rng(15)
    B, H, Hkv, D, bs = 2, 2, 2, 8, 4
    lens = np.array([9, 21], dtype=np.int32)
    # quarter-integer data keeps K and K + u exact in float32
    K = (rng.integers(-8, 8, size=(B, Hkv, 21, D)) / 4).astype(np.float32)
    V = rng.standard_normal((B, Hkv, 21, D)).astype(np.float32)
    q = rng.standard_normal((B, H, D)).astype(np.float32)
    u = np.float32(0.5)
    NB = 20
    kp, vp, table, stride = scatter_to_pool(K, V, bs, NB, np.random.default_rng(0))
    kp2, vp2, table2, _ = scatter_to_pool(K + u, V, bs, NB, np.random.default_rng(0))
    kw = dict(num_kv_heads=Hkv, block_size=bs, block_stride=stride, num_blocks=NB)
    o1, _ = oracle.attention_decode(q, kp, vp, table, lens, 0.5, **kw)
    o2, _ = oracle.attention_decode(q, kp2, vp2, table2, lens, 0.5, **kw)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_zero_length_gives_zero():
    rng = np.random.default_rng(16)
    c = tiny_case(rng, B=3, H=2, Hkv=2, D=8, lens=[0, 5, 0], bs=4)
    out, err = run_decode(c, 1.0)
    assert not err.any()
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[1]))


# ---------------------------------------------------------------------------
# paging is a pure relabelling
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["colocated", "separate"])
def test_relabelling_and_block_size_do_not_change_anything(layout):
    rng = np.random.default_rng(21)
    B, H, Hkv, D = 3, 4, 2, 16
    lens = np.array([37, 64, 5], dtype=np.int32)
    K = rng.standard_normal((B, Hkv, 64, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, 64, D)).astype(np.float32)
    q = rng.standard_normal((B, H, D)).astype(np.float32)
    scale = 0.25
    # unpaged: the oracle's own contiguous attention on the contiguous rows
    ref = np.zeros((B, H, D))
    for b in range(B):
        for h in range(H):
            L = int(lens[b])
            ref[b, h] = oracle.attention_contiguous(q[b, h].astype(np.float64), K[b, h // 2, :L],
                                                    V[b, h // 2, :L], scale)
    for bs in (8, 16, 32, 64, 5):
        for seed in (1, 2):
            NB = B * (-(-64 // bs)) + 7
            kp, vp, table, stride = scatter_to_pool(K, V, bs, NB, np.random.default_rng(seed),
                                                    layout=layout)
            out, err = oracle.attention_decode(q, kp, vp, table, lens, scale, num_kv_heads=Hkv,
                                               block_size=bs, block_stride=stride, num_blocks=NB)
            assert not err.any()
            assert np.array_equal(out, ref), (bs, seed)


def test_poisoned_padding_and_unused_blocks_change_nothing():
    """Valid length, never allocated length ("A strange KV Cache bug" s2.4)."""
    w = workloads.make_workload(1, poison=False)
    w_p = workloads.make_workload(1, poison=True)
    lens = w.lens
    kw = dict(num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride, num_blocks=w.NB)
    o1, e1 = oracle.attention_decode(w.q, w.k_flat(), w.v_flat(), w.block_table, lens, w.scale, **kw)
    o2, e2 = oracle.attention_decode(w_p.q, w_p.k_flat(), w_p.v_flat(), w_p.block_table, lens,
                                     w.scale, **kw)
    assert not e1.any() and not e2.any()
    assert np.all(np.isfinite(o2))
    assert np.array_equal(o1, o2)
    # and the poison is really there: reading one slot too many breaks it
    o3, _ = oracle.attention_decode(w_p.q, w_p.k_flat(), w_p.v_flat(), w_p.block_table, lens + 1,
                                    w.scale, **kw)
    assert not np.all(np.isfinite(o3))


def test_shared_blocks_equal_private_copies():
    w = workloads.make_workload(5, max_len=700)
    assert w.meta["shared_blocks"] > 0
    u = workloads.unshare(w)
    kw = dict(num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride)
    o1, _ = oracle.attention_decode(w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens, w.scale,
                                    num_blocks=w.NB, **kw)
    o2, _ = oracle.attention_decode(u.q, u.k_flat(), u.v_flat(), u.block_table, u.lens, u.scale,
                                    num_blocks=u.NB, **kw)
    assert np.array_equal(o1, o2)
    # beams share the prefix but differ in their tails
    assert not np.array_equal(o1[0], o1[1])


# ---------------------------------------------------------------------------
# split-KV partial sums and their merge
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ptok", [8, 24, 64, 1000])
def test_partials_merge_to_full_attention(ptok):
    w = workloads.make_workload(1)
    kw = dict(num_kv_heads=w.Hkv, block_size=w.bs, block_stride=w.block_stride, num_blocks=w.NB)
    full, _ = oracle.attention_decode(w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens, w.scale, **kw)
    Lmax = int(w.lens.max())
    parts = []
    for t0 in range(0, Lmax, ptok):
        parts.append(oracle.attention_partial(w.q, w.k_flat(), w.v_flat(), w.block_table, w.lens,
                                              w.scale, t0, t0 + ptok, **kw))
    for b in range(w.B):
        for h in range(w.H):
            m = np.array([p[0][b, h] for p in parts])
            l = np.array([p[1][b, h] for p in parts])
            acc = np.stack([p[2][b, h] for p in parts])
            np.testing.assert_allclose(oracle.merge_partials(m, l, acc), full[b, h],
                                       rtol=0, atol=1e-12)


def test_partial_of_single_token_and_empty_range():
    rng = np.random.default_rng(31)
    c = tiny_case(rng, B=1, H=1, Hkv=1, D=8, lens=[10], bs=4)
    kw = dict(num_kv_heads=1, block_size=4, block_stride=c["stride"], num_blocks=c["NB"])
    m, l, acc, _ = oracle.attention_partial(c["q"], c["kp"], c["vp"], c["table"], c["lens"],
                                            0.5, 3, 4, **kw)
    x = 0.5 * float(c["q"][0, 0].astype(np.float64) @ c["K"][0, 0, 3].astype(np.float64))
    assert m[0, 0] == pytest.approx(x, abs=1e-14)
    assert l[0, 0] == 1.0
    assert np.array_equal(acc[0, 0], c["V"][0, 0, 3].astype(np.float64))
    m, l, acc, _ = oracle.attention_partial(c["q"], c["kp"], c["vp"], c["table"], c["lens"],
                                            0.5, 10, 20, **kw)
    assert m[0, 0] == -np.inf and l[0, 0] == 0 and not acc.any()


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_append_token_by_token_rebuilds_the_contiguous_cache(dtype):
    """Appending tokens 0..L-1 one by one lays them out in logical order."""
    tdt = workloads.DTYPES[dtype]
    B, Hkv, D, bs, L = 3, 2, 8, 4, 11
    g = torch.Generator().manual_seed(3)
    K = torch.randn(B, Hkv, L, D, generator=g).to(tdt)
    V = torch.randn(B, Hkv, L, D, generator=g).to(tdt)
    nblk = -(-L // bs)
    NB = B * nblk + 4
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    table = torch.full((B, nblk + 1), -1, dtype=torch.int32)
    for b in range(B):
        table[b, :nblk] = perm[b * nblk:(b + 1) * nblk]
    pool = torch.full((NB, 2, Hkv, bs, D), float("nan"), dtype=tdt)
    flat = pool.view(-1)
    vflat = flat[Hkv * bs * D:]
    stride = 2 * Hkv * bs * D
    untouched = pool.clone()
    for t in range(L):
        err = oracle.kv_append(K[:, :, t].contiguous(), V[:, :, t].contiguous(), flat, vflat,
                               table, torch.full((B,), t, dtype=torch.int32), block_size=bs,
                               block_stride=stride, num_blocks=NB)
        assert not err.any()
    for b in range(B):
        for t in range(L):
            blk, slot = int(table[b, t // bs]), t % bs
            assert torch.equal(pool[blk, 0, :, slot].view(torch.int16) if dtype != "f32"
                               else pool[blk, 0, :, slot].view(torch.int32),
                               K[b, :, t].view(torch.int16) if dtype != "f32"
                               else K[b, :, t].view(torch.int32))
            assert torch.equal(pool[blk, 1, :, slot].float(), V[b, :, t].float())
    # slots past L in the last blocks and unused blocks are untouched
    written = torch.zeros_like(pool, dtype=torch.bool)
    for b in range(B):
        for t in range(L):
            written[int(table[b, t // bs]), :, :, t % bs] = True
    same = (pool.float().isnan() & untouched.float().isnan()) | (pool.float() == untouched.float())
    assert bool(same[~written].all())
    # gathering the appended cache gives back the contiguous rows
    for b in range(B):
        for hk in range(Hkv):
            Kc, Vc = oracle.gather(flat, vflat, table[b], hk, L, block_size=bs, head_dim=D,
                                   num_kv_heads=Hkv, block_stride=stride)
            assert np.array_equal(Kc, K[b, hk].double().numpy())
            assert np.array_equal(Vc, V[b, hk].double().numpy())


def test_append_rejects_bad_position_and_unallocated_block():
    B, Hkv, D, bs = 3, 1, 4, 4
    pool = torch.zeros(8, 2, Hkv, bs, D)
    flat = pool.view(-1)
    table = torch.tensor([[0, 1], [2, -1], [3, 9]], dtype=torch.int32)
    kn = torch.ones(B, Hkv, D)
    err = oracle.kv_append(kn, kn, flat, flat[Hkv * bs * D:], table,
                           torch.tensor([8, 4, 5], dtype=torch.int32), block_size=bs,
                           block_stride=2 * Hkv * bs * D, num_blocks=8)
    assert err[0] == oracle.SEQ_BAD_POS        # 8 >= 2 blocks * 4 slots
    assert err[1] == oracle.SEQ_BAD_BLOCK      # logical block 1 is -1
    assert err[2] == oracle.SEQ_BAD_BLOCK      # block 9 is outside a pool of 8
    assert not pool.any()


# ---------------------------------------------------------------------------
# validation
# ---------------------------------------------------------------------------

def test_validation_flags_bad_tables_and_lengths():
    rng = np.random.default_rng(41)
    c = tiny_case(rng, B=4, H=2, Hkv=2, D=8, lens=[9, 9, 9, 9], bs=4)
    c["table"][1, 1] = -1                       # hole inside the valid range
    c["table"][2, 2] = c["NB"]                  # id past the pool
    c["lens"][3] = c["table"].shape[1] * 4 + 1  # longer than the table row
    c["table"][0, 3:] = -1                      # past ceil(9/4)=3: ignored
    out, err = run_decode(c, 1.0)
    assert err[0] == 0 and np.all(np.isfinite(out[0]))
    assert err[1] == oracle.SEQ_BAD_BLOCK and not out[1].any()
    assert err[2] == oracle.SEQ_BAD_BLOCK and not out[2].any()
    assert err[3] == oracle.SEQ_BAD_LEN and not out[3].any()


# ---------------------------------------------------------------------------
# multi-token append (prefill write) and sliding-window decode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_token_append_equals_token_by_token(dtype):
    """A padded batch written at once equals its valid tokens written one by
    one; padding rows (t >= counts[b]) never reach the pool ("A strange KV
    Cache bug", s2.3-2.4)."""
    tdt = workloads.DTYPES[dtype]
    B, T, Hkv, D, bs = 4, 9, 2, 8, 4
    g = torch.Generator().manual_seed(17)
    counts = torch.tensor([9, 0, 5, 3], dtype=torch.int32)
    starts = torch.tensor([0, 7, 6, 13], dtype=torch.int32)
    kn = torch.randn(B, T, Hkv, D, generator=g).to(tdt)
    vn = torch.randn(B, T, Hkv, D, generator=g).to(tdt)
    for b in range(B):
        kn[b, counts[b]:] = float("nan")
        vn[b, counts[b]:] = float("nan")
    MB = 5
    NB = B * MB + 2
    perm = torch.randperm(NB, generator=g).to(torch.int32)
    table = perm[:B * MB].view(B, MB).contiguous()
    stride = 2 * Hkv * bs * D
    pool_a = torch.zeros(NB, 2, Hkv, bs, D, dtype=tdt)
    pool_b = pool_a.clone()
    fa, fb = pool_a.view(-1), pool_b.view(-1)
    kw = dict(block_size=bs, block_stride=stride, num_blocks=NB)
    err = oracle.kv_append_tokens(kn, vn, fa, fa[Hkv * bs * D:], table, starts, counts, **kw)
    assert not err.any()
    for b in range(B):
        for t in range(int(counts[b])):
            one = torch.zeros(B, dtype=torch.int32)
            mask = torch.zeros(B, dtype=torch.bool)
            mask[b] = True
            # append only sequence b's token t: other rows get a position past the table
            pos = torch.where(mask, starts + t, torch.full((B,), MB * bs, dtype=torch.int32))
            e = oracle.kv_append(kn[:, t].contiguous(), vn[:, t].contiguous(), fb,
                                 fb[Hkv * bs * D:], table, pos, **kw)
            assert e[b] == 0
    assert torch.equal(pool_a.view(torch.int16 if dtype != "f32" else torch.int32),
                       pool_b.view(torch.int16 if dtype != "f32" else torch.int32))
    assert not pool_a.float().isnan().any()


def test_multi_token_append_flags():
    B, T, Hkv, D, bs, MB = 4, 4, 1, 4, 4, 2
    pool = torch.zeros(10, 2, Hkv, bs, D)
    flat = pool.view(-1)
    table = torch.tensor([[0, 1], [2, 3], [4, -1], [6, 7]], dtype=torch.int32)
    kn = torch.ones(B, T, Hkv, D)
    err = oracle.kv_append_tokens(kn, kn, flat, flat[Hkv * bs * D:], table,
                                  torch.tensor([0, 6, 2, 0], dtype=torch.int32),
                                  torch.tensor([5, 3, 4, 2], dtype=torch.int32),
                                  block_size=bs, block_stride=2 * Hkv * bs * D, num_blocks=10)
    assert err[0] == oracle.SEQ_BAD_LEN        # 5 tokens in a batch of 4
    assert err[1] == oracle.SEQ_BAD_POS        # 6 + 3 > 2 blocks * 4 slots
    assert err[2] == oracle.SEQ_BAD_BLOCK      # tokens 4, 5 land in the unallocated block
    assert err[3] == 0
    assert pool[4, :, :, 2:].all() and not pool[2:4].any()


def test_window_decode_pins():
    rng = np.random.default_rng(51)
    B, H, Hkv, D, bs = 3, 4, 2, 16, 4
    lens = np.array([1, 23, 40], dtype=np.int32)
    K = rng.standard_normal((B, Hkv, 40, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, 40, D)).astype(np.float32)
    q = rng.standard_normal((B, H, D)).astype(np.float32)
    NB = B * 10 + 3
    kp, vp, table, stride = scatter_to_pool(K, V, bs, NB, rng)
    kw = dict(num_kv_heads=Hkv, block_size=bs, block_stride=stride, num_blocks=NB)
    full, _ = oracle.attention_decode(q, kp, vp, table, lens, 0.3, **kw)
    for W in (40, 1000):
        o, e = oracle.attention_decode_window(q, kp, vp, table, lens, 0.3, W, **kw)
        assert not e.any() and np.array_equal(o, full)
    o, _ = oracle.attention_decode_window(q, kp, vp, table, lens, 0.3, 1, **kw)
    for b in range(B):
        for h in range(H):
            assert np.array_equal(o[b, h], V[b, h // 2, lens[b] - 1].astype(np.float64))
    for W in (3, 7, 16):
        o, _ = oracle.attention_decode_window(q, kp, vp, table, lens, 0.3, W, **kw)
        ref = np.zeros_like(o)
        for b in range(B):
            L = int(lens[b])
            lo = max(0, L - W)
            for h in range(H):
                ref[b, h] = oracle.attention_contiguous(q[b, h].astype(np.float64),
                                                        K[b, h // 2, lo:L], V[b, h // 2, lo:L], 0.3)
        assert np.array_equal(o, ref), W
        sd = sdpa_reference(q.astype(np.float64),
                            np.stack([np.pad(K[b, :, max(0, lens[b] - W):lens[b]],
                                             ((0, 0), (0, 40 - min(W, lens[b])), (0, 0)))
                                      for b in range(B)]).astype(np.float64),
                            np.stack([np.pad(V[b, :, max(0, lens[b] - W):lens[b]],
                                             ((0, 0), (0, 40 - min(W, lens[b])), (0, 0)))
                                      for b in range(B)]).astype(np.float64),
                            np.minimum(lens, W), 0.3)
        np.testing.assert_allclose(o, sd, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# int8 cache blocks with per-(block, kv head) scales
# ---------------------------------------------------------------------------

def _np_quantize(x, s):
    """Independent restatement of the code rule: IEEE binary32 quotient,
    numpy's round-half-to-even, clamp to [-127, 127], NaN to 0."""
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        r = np.rint(np.asarray(x, dtype=np.float32) / np.float32(s))
    r = np.where(np.isnan(r), 0.0, np.clip(r, -127.0, 127.0))
    return r.astype(np.int8)


def test_quantize_i8_pins():
    # worked by hand: ties go to the even integer, out-of-range values clamp
    cases = [(2.5, 1.0, 2), (3.5, 1.0, 4), (-2.5, 1.0, -2), (-3.5, 1.0, -4), (0.5, 1.0, 0),
             (1.5, 1.0, 2), (0.75, 0.5, 2), (0.25, 0.5, 0), (127.5, 1.0, 127), (-127.5, 1.0, -127),
             (1e6, 1.0, 127), (-1e6, 1.0, -127), (float("inf"), 1.0, 127),
             (float("-inf"), 1.0, -127), (float("nan"), 1.0, 0), (0.3, 0.1, 3), (-0.0, 2.0, 0)]
    for x, sc, c in cases:
        assert int(oracle.quantize_i8([x], sc)[0]) == c, (x, sc, c)
    rng = np.random.default_rng(5)
    x = (rng.normal(0.0, 3.0, 20000)).astype(np.float32)
    sc = np.float32(0.037)
    codes = oracle.quantize_i8(x, sc)
    assert np.array_equal(codes, _np_quantize(x, sc))
    inside = np.abs(x) <= 127 * sc
    err = np.abs(x[inside].astype(np.float64) - codes[inside].astype(np.float64) * float(sc))
    assert err.max() <= float(sc) / 2 * (1 + 1e-6)


def _i8_case(seed, B=3, H=4, Hkv=2, D=16, bs=4, lens=(0, 5, 11)):
    rng = np.random.default_rng(seed)
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + 3
    MB = max(nblk) + 1
    perm = rng.permutation(NB)
    table = np.full((B, MB), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        table[b, :nblk[b]] = perm[k:k + nblk[b]]
        k += nblk[b]
    pool = rng.integers(-127, 128, size=(NB, 2, Hkv, bs, D)).astype(np.int8)
    scales = rng.uniform(0.01, 0.1, size=(NB, 2, Hkv)).astype(np.float32)
    q = rng.normal(size=(B, H, D)).astype(np.float32)
    return dict(B=B, H=H, Hkv=Hkv, D=D, bs=bs, NB=NB, MB=MB, lens=np.array(lens, dtype=np.int32),
                table=table, pool=pool, scales=scales, q=q, stride=2 * Hkv * bs * D)


def test_i8_decode_brute_force():
    """Tiny case against per-token Python loops over the dequantised values."""
    c = _i8_case(11)
    flat = c["pool"].reshape(-1)
    out, err = oracle.attention_decode_i8(c["q"], flat, flat[c["Hkv"] * c["bs"] * c["D"]:],
                                          c["scales"], c["table"], c["lens"], 0.3,
                                          num_kv_heads=c["Hkv"], block_size=c["bs"],
                                          block_stride=c["stride"], num_blocks=c["NB"])
    assert not err.any()
    g = c["H"] // c["Hkv"]
    for b in range(c["B"]):
        for h in range(c["H"]):
            hk = h // g
            L = int(c["lens"][b])
            if L == 0:
                assert not out[b, h].any()
                continue
            K = np.empty((L, c["D"]))
            V = np.empty((L, c["D"]))
            for t in range(L):
                blk = c["table"][b, t // c["bs"]]
                K[t] = c["pool"][blk, 0, hk, t % c["bs"]].astype(np.float64) * float(c["scales"][blk, 0, hk])
                V[t] = c["pool"][blk, 1, hk, t % c["bs"]].astype(np.float64) * float(c["scales"][blk, 1, hk])
            x = 0.3 * (K @ c["q"][b, h].astype(np.float64))
            w = np.exp(x - x.max())
            np.testing.assert_allclose(out[b, h], (w[:, None] * V).sum(0) / w.sum(), rtol=0, atol=1e-12)


def test_i8_decode_equals_float_decode_on_exact_values():
    """Codes times power-of-two scales are exact in binary32: the int8 oracle
    and the float oracle (pinned to torch's attention above) see the same
    values, so they agree to rounding."""
    c = _i8_case(12, B=2, H=8, Hkv=2, D=32, bs=8, lens=(40, 17))
    c["scales"] = (2.0 ** np.random.default_rng(3).integers(-8, -2, size=c["scales"].shape)).astype(np.float32)
    deq = c["pool"].astype(np.float32) * c["scales"][:, :, :, None, None]
    fflat = np.ascontiguousarray(deq).reshape(-1)
    iflat = c["pool"].reshape(-1)
    off = c["Hkv"] * c["bs"] * c["D"]
    kw = dict(num_kv_heads=c["Hkv"], block_size=c["bs"], block_stride=c["stride"], num_blocks=c["NB"])
    ref, e1 = oracle.attention_decode(c["q"], fflat, fflat[off:], c["table"], c["lens"], 0.2, **kw)
    got, e2 = oracle.attention_decode_i8(c["q"], iflat, iflat[off:], c["scales"], c["table"], c["lens"],
                                         0.2, **kw)
    assert not e1.any() and not e2.any()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_i8_append_writes_the_codes_of_its_block_scale():
    c = _i8_case(13, B=3, H=4, Hkv=2, D=16, bs=4, lens=(3, 8, 9))
    NB, Hkv, D, bs = c["NB"], c["Hkv"], c["D"], c["bs"]
    # give every sequence a block for position len
    used = set(int(x) for x in c["table"].ravel() if x >= 0)
    free = [i for i in range(NB) if i not in used]
    for b in range(c["B"]):
        for j in range(-(-(int(c["lens"][b]) + 1) // bs)):
            if c["table"][b, j] < 0:
                c["table"][b, j] = free.pop()
    gen = torch.Generator().manual_seed(4)
    kn = torch.randn((c["B"], Hkv, D), generator=gen).to(torch.bfloat16)
    vn = torch.randn((c["B"], Hkv, D), generator=gen).to(torch.bfloat16)
    pool = c["pool"].copy()
    flat = pool.reshape(-1)
    err = oracle.kv_append_i8(kn, vn, flat, flat[Hkv * bs * D:], c["scales"], c["table"], c["lens"],
                              block_size=bs, block_stride=c["stride"], num_blocks=NB)
    assert not err.any()
    want = c["pool"].copy()
    for b in range(c["B"]):
        pos = int(c["lens"][b])
        blk = c["table"][b, pos // bs]
        for hk in range(Hkv):
            want[blk, 0, hk, pos % bs] = _np_quantize(kn[b, hk].float().numpy(), c["scales"][blk, 0, hk])
            want[blk, 1, hk, pos % bs] = _np_quantize(vn[b, hk].float().numpy(), c["scales"][blk, 1, hk])
    assert np.array_equal(pool, want)
    # a position past the row and a hole in the table are skipped and flagged
    pos = c["lens"].copy()
    pos[0] = c["MB"] * bs
    tab = c["table"].copy()
    tab[1, int(c["lens"][1]) // bs] = -1
    pool2 = c["pool"].copy()
    f2 = pool2.reshape(-1)
    err = oracle.kv_append_i8(kn, vn, f2, f2[Hkv * bs * D:], c["scales"], tab, pos,
                              block_size=bs, block_stride=c["stride"], num_blocks=NB)
    assert list(err) == [oracle.SEQ_BAD_POS, oracle.SEQ_BAD_BLOCK, 0]
    changed = np.nonzero((pool2 != c["pool"]).reshape(NB, -1).any(1))[0]
    assert list(changed) == [int(c["table"][2, int(c["lens"][2]) // bs])]


# ---------------------------------------------------------------------------
# fp8 (E4M3) cache: the format pinned to torch's float8_e4m3fn (a library
# routine) and to values worked by hand, the decode to brute force
# ---------------------------------------------------------------------------

def _torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_value_of_every_code_matches_torch():
    ref = _torch_e4m3_values()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert list(np.nonzero(np.isnan(got))[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    # by hand: the largest finite, the smallest normal and subnormal, one
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x80) == 0.0


def test_e4m3_encode_pins():
    vals = _torch_e4m3_values()
    # every finite code round-trips (both zeros included)
    for c in range(256):
        if not np.isnan(vals[c]):
            assert oracle.e4m3_encode(np.float32(vals[c])) == c, c
    # midpoints between neighbours go to the even code; one ulp off decides
    pos = [(c, vals[c]) for c in range(0x7F)]
    for (c0, v0), (c1, v1) in zip(pos, pos[1:]):
        mid = np.float32((v0 + v1) / 2)
        assert float(mid) == (v0 + v1) / 2
        assert oracle.e4m3_encode(mid) == (c0 if c0 % 2 == 0 else c1), (c0, c1)
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(np.inf))) == c1
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(0))) == c0
        assert oracle.e4m3_encode(-mid) == 0x80 | oracle.e4m3_encode(mid)
    # worked by hand: subnormal ties, saturation beyond 448, NaN
    cases = [(2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (5 * 2.0 ** -10, 0x02), (1.0625, 0x38),
             (1.1875, 0x3A), (449.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (1e30, 0x7E),
             (float("inf"), 0x7E), (-500.0, 0xFE), (float("-inf"), 0xFE), (float("nan"), 0x7F)]
    for x, c in cases:
        assert oracle.e4m3_encode(x) == c, (x, c)
    # inside the finite range it is torch's rounding
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.uniform(-463.0, 463.0, 50000), rng.normal(0.0, 0.05, 50000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.quantize_fp8(x, 1.0), ref)


def test_quantize_fp8_divides_in_binary32():
    # the quotient is taken in binary32 before rounding to E4M3
    rng = np.random.default_rng(10)
    x = rng.normal(0.0, 3.0, 20000).astype(np.float32)
    sc = np.float32(0.0137)
    q = (x / sc).astype(np.float32)
    ref = torch.from_numpy(np.clip(q, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.quantize_fp8(x, sc), ref)


def _fp8_case(seed, B=3, H=4, Hkv=2, D=16, bs=4, lens=(0, 5, 11)):
    c = _i8_case(seed, B=B, H=H, Hkv=Hkv, D=D, bs=bs, lens=lens)
    rng = np.random.default_rng(seed + 100)
    codes = rng.integers(0, 256, size=c["pool"].shape).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C   # no NaN codes in the cache
    c["pool"] = codes
    return c


def _fp8_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_fp8_decode_brute_force():
    """Tiny case against per-token Python loops over the dequantised values
    (codes read by torch's float8_e4m3fn)."""
    c = _fp8_case(21)
    flat = c["pool"].reshape(-1)
    out, err = oracle.attention_decode_fp8(c["q"], flat, flat[c["Hkv"] * c["bs"] * c["D"]:],
                                           c["scales"], c["table"], c["lens"], 0.05,
                                           num_kv_heads=c["Hkv"], block_size=c["bs"],
                                           block_stride=c["stride"], num_blocks=c["NB"])
    assert not err.any()
    deq = _fp8_values(c["pool"])
    g = c["H"] // c["Hkv"]
    for b in range(c["B"]):
        for h in range(c["H"]):
            hk = h // g
            L = int(c["lens"][b])
            if L == 0:
                assert not out[b, h].any()
                continue
            K = np.empty((L, c["D"]))
            V = np.empty((L, c["D"]))
            for t in range(L):
                blk = c["table"][b, t // c["bs"]]
                K[t] = deq[blk, 0, hk, t % c["bs"]] * float(c["scales"][blk, 0, hk])
                V[t] = deq[blk, 1, hk, t % c["bs"]] * float(c["scales"][blk, 1, hk])
            x = 0.05 * (K @ c["q"][b, h].astype(np.float64))
            w = np.exp(x - x.max())
            np.testing.assert_allclose(out[b, h], (w[:, None] * V).sum(0) / w.sum(), rtol=0, atol=1e-12)


def test_fp8_append_writes_the_codes_of_its_block_scale():
    c = _fp8_case(23, B=3, H=4, Hkv=2, D=16, bs=4, lens=(3, 8, 9))
    NB, Hkv, D, bs = c["NB"], c["Hkv"], c["D"], c["bs"]
    used = set(int(x) for x in c["table"].ravel() if x >= 0)
    free = [i for i in range(NB) if i not in used]
    for b in range(c["B"]):
        for j in range(-(-(int(c["lens"][b]) + 1) // bs)):
            if c["table"][b, j] < 0:
                c["table"][b, j] = free.pop()
    gen = torch.Generator().manual_seed(24)
    kn = torch.randn((c["B"], Hkv, D), generator=gen).to(torch.float16)
    vn = torch.randn((c["B"], Hkv, D), generator=gen).to(torch.float16)
    pool = c["pool"].copy()
    flat = pool.reshape(-1)
    err = oracle.kv_append_fp8(kn, vn, flat, flat[Hkv * bs * D:], c["scales"], c["table"], c["lens"],
                               block_size=bs, block_stride=c["stride"], num_blocks=NB)
    assert not err.any()
    want = c["pool"].copy()

    def codes(x, s):
        q = (x.float().numpy() / np.float32(s)).astype(np.float32)
        return torch.from_numpy(np.clip(q, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    for b in range(c["B"]):
        pos = int(c["lens"][b])
        blk = c["table"][b, pos // bs]
        for hk in range(Hkv):
            want[blk, 0, hk, pos % bs] = codes(kn[b, hk], c["scales"][blk, 0, hk])
            want[blk, 1, hk, pos % bs] = codes(vn[b, hk], c["scales"][blk, 1, hk])
    assert np.array_equal(pool, want)
    # a position past the row and a hole in the table are skipped and flagged
    pos = c["lens"].copy()
    pos[0] = c["MB"] * bs
    tab = c["table"].copy()
    tab[1, int(c["lens"][1]) // bs] = -1
    pool2 = c["pool"].copy()
    f2 = pool2.reshape(-1)
    err = oracle.kv_append_fp8(kn, vn, f2, f2[Hkv * bs * D:], c["scales"], tab, pos,
                               block_size=bs, block_stride=c["stride"], num_blocks=NB)
    assert list(err) == [oracle.SEQ_BAD_POS, oracle.SEQ_BAD_BLOCK, 0]


# ---------------------------------------------------------------------------
# the battery catches plausible mistakes planted in a copy of the oracle
# ---------------------------------------------------------------------------

MUTANTS = {
    "scale dropped": ("x[t] = scale * dot;", "x[t] = dot;"),
    "exponent sign flipped": ("double w = exp(x[t] - m);", "double w = exp(m - x[t]);"),
    "no normalisation": ("        o[d] /= wsum;\n    free(x);", "    free(x);"),
    "K used as V": ("o[d] += w * Vc[t * D + d];", "o[d] += w * Kc[t * D + d];"),
    "slot and head swapped": ("(int64_t)hk * bs * D + slot * D;", "(int64_t)hk * D + slot * Hkv * D;"),
    "block from slot": ("int64_t blk = table_row[t / bs];", "int64_t blk = table_row[t % bs];"),
    "query head uses kv head": ("qd[d] = pao_element(q, ((int64_t)b * H + h) * D + d, dtype);",
                                "qd[d] = pao_element(q, ((int64_t)b * H + hk) * D + d, dtype);"),
    "f16 exponent bias": ("expo - 25", "expo - 24"),
    "window one token too long": ("int64_t first = len > window ? len - window : 0;",
                                  "int64_t first = len > window ? len - window - 1 : 0;"),
    "prefill writes padding": ("for (int64_t t = 0; t < n; ++t) {\n                int64_t pos = start + t;",
                               "for (int64_t t = 0; t < T && start + t < (int64_t)MB * bs; ++t) {\n                int64_t pos = start + t;"),
    "one padding slot read": ("int64_t len = seq_lens[b];\n        if (seq_err[b]) {",
                              "int64_t len = seq_lens[b] + (seq_lens[b] % bs != 0);\n        if (seq_err[b]) {"),
    "int8 codes truncated": ("float r = rintf(q);", "float r = truncf(q);"),
    "int8 ties away from zero": ("float r = rintf(q);", "float r = roundf(q);"),
    "int8 not clamped": ("    if (r > 127.0f)\n        r = 127.0f;\n", ""),
    "int8 K read with the V scale": ("double sk = kv_scales[(blk * 2 + 0) * Hkv + hk];",
                                     "double sk = kv_scales[(blk * 2 + 1) * Hkv + hk];"),
    "int8 scale of the logical block": ("double sv = kv_scales[(blk * 2 + 1) * Hkv + hk];",
                                        "double sv = kv_scales[((t / bs) * 2 + 1) * Hkv + hk];"),
    "int8 append with the V scale": ("float sk = kv_scales[(blk * 2 + 0) * Hkv + hk];",
                                     "float sk = kv_scales[(blk * 2 + 1) * Hkv + hk];"),
    "fp8 exponent bias off by one": ("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 9);"),
    "fp8 subnormals as normals": ("v = ldexp((double)m, -9);", "v = ldexp((double)(8 + m), -10);"),
    "fp8 ties away from zero": ("r = nearbyint(a / ldexp(1.0, E - 3));", "r = round(a / ldexp(1.0, E - 3));"),
    "fp8 truncated": ("r = nearbyint(a / ldexp(1.0, -9));", "r = floor(a / ldexp(1.0, -9));"),
    "fp8 no saturation": ("    if (a >= 448.0)\n        return sign | 0x7E;\n", ""),
    "fp8 carry into the exponent lost": ("        r = 8.0;\n        E += 1;", "        r = 15.0;"),
    "fp8 V read with the K scale": ("            Vc[t * D + d] = pao_e4m3_value(v_pool[base + d]) * sv;",
                                    "            Vc[t * D + d] = pao_e4m3_value(v_pool[base + d]) * sk;"),
}


def _battery(lib) -> bool:
    """True if every check passes against the library `lib`."""
    saved = oracle._handle
    oracle._handle = lib
    try:
        tests = [lambda: test_decode_matches_sdpa_float64(4, 2, 3),
                 lambda: test_decode_matches_sdpa_float64(8, 1, 16),
                 lambda: test_decode_16bit_inputs_match_sdpa("f16"),
                 test_single_token_returns_v0_exactly,
                 test_constant_values_give_that_constant,
                 test_window_decode_pins,
                 lambda: test_multi_token_append_equals_token_by_token("f32"),
                 test_quantize_i8_pins,
                 test_i8_decode_brute_force,
                 test_i8_append_writes_the_codes_of_its_block_scale,
                 test_e4m3_value_of_every_code_matches_torch,
                 test_e4m3_encode_pins,
                 test_fp8_decode_brute_force,
                 test_fp8_append_writes_the_codes_of_its_block_scale]
        for t in tests:
            try:
                t()
            except AssertionError:
                return False
        return True
    finally:
        oracle._handle = saved


def _load_like_real(path):
    real = oracle._lib()
    lib = ctypes.CDLL(str(path))
    for fn in ("pao_blocks_needed", "pao_kv_bytes", "pao_convert", "pao_gather",
               "pao_attention_contiguous", "pao_attention_decode", "pao_attention_partial",
               "pao_merge_partials", "pao_kv_append", "pao_kv_append_tokens",
               "pao_attention_decode_window", "pao_quantize_i8", "pao_quantize_i8_array",
               "pao_kv_append_i8", "pao_gather_i8", "pao_attention_decode_i8",
               "pao_e4m3_value", "pao_e4m3_encode", "pao_quantize_fp8", "pao_quantize_fp8_array",
               "pao_kv_append_fp8", "pao_gather_fp8", "pao_attention_decode_fp8"):
        getattr(lib, fn).restype = getattr(real, fn).restype
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
    return lib


def _battery_in_child(so_path) -> int:
    """Run the battery against a mutant in a child process (a mutant may crash).

    Exit status 0 means every check passed, i.e. the mistake went unnoticed.
    """
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r);"
            "import tests.test_oracle as t;"
            "sys.exit(0 if t._battery(t._load_like_real(%r)) else 1)"
            % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
               os.path.dirname(os.path.abspath(__file__)), str(so_path)))
    return subprocess.run([sys.executable, "-c", code], capture_output=True).returncode


def test_planted_mistakes_are_caught(tmp_path):
    src = open(oracle._SRC).read()
    assert _battery(oracle._lib())
    assert _battery_in_child(oracle._LIB) == 0   # control: the real oracle passes in a child
    for i, (name, (old, new)) in enumerate(MUTANTS.items()):
        assert old in src, name
        path = tmp_path / f"mutant{i}.c"
        path.write_text(src.replace(old, new, 1))
        so = tmp_path / f"mutant{i}.so"
        subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"],
                       check=True)
        assert _battery_in_child(so) != 0, f"planted mistake not caught: {name}"
