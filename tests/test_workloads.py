"""CPU checks of the seeded input generators that the parity tests rely on:
the shared-prefix groups really share what they declare and nothing else,
every table row has room for the step's append, the shared-beam workload has
the block structure of its reading (937 shared blocks, a copied boundary
block, 88 private blocks per beam after the append), and the quantised
counterparts keep the table, lengths and queries of the workload."""
import torch

import workloads


def _rows(w):
    return [[int(x) for x in w.block_table[b] if int(x) >= 0] for b in range(w.B)]


def test_prefix_groups_share_exactly_what_they_declare():
    sizes, shared, tails = [3, 1, 2], [5, 0, 2], [4, 0, 9, 16, 1, 31]
    w = workloads.make_prefix_groups(group_sizes=sizes, shared_blocks=shared, tails=tails, H=4, Hkv=2, D=16,
                                     bs=8, dtype=torch.float16, seed=1, poison=False)
    first = w.meta["group_first"]
    assert first == [0, 3, 4, 6]
    assert w.meta["shared_tokens"] == [s * w.bs for s in shared]
    rows = _rows(w)
    owner = {}
    for gi, n in enumerate(sizes):
        members = range(first[gi], first[gi + 1])
        common = rows[first[gi]][:shared[gi]]
        for b in members:
            L = int(w.lens[b])
            assert L == shared[gi] * w.bs + tails[b]
            assert len(rows[b]) == -(-(L + 1) // w.bs)          # room for the step's append
            assert rows[b][:shared[gi]] == common
            for j, blk in enumerate(rows[b]):
                key = ("shared", gi) if j < shared[gi] else ("own", b)
                assert owner.setdefault(blk, key) == key          # no block outside its owner
    assert all(0 <= blk < w.NB for r in rows for blk in r)


def test_shared_beams_workload_block_structure():
    w = workloads.make_workload(5)
    bs, S = w.bs, w.meta["shared_blocks"]
    assert (w.B, bs, S) == (4, 32, 937)
    rows = _rows(w)
    assert all(r[:S] == rows[0][:S] for r in rows)
    # the block holding the end of the 30000-token prompt is a copy per beam
    assert len({r[S] for r in rows}) == w.B
    private = [set(r[S:]) for r in rows]
    assert all(len(p) == 88 for p in private)
    assert len(set().union(*private)) == 4 * 88
    assert len(set().union(*map(set, rows))) == 937 + 4 * 88


def test_quantised_counterparts_keep_table_lengths_and_queries():
    w = workloads.make_generic(B=3, H=4, Hkv=2, D=64, bs=16, dtype=torch.bfloat16, lens=[5, 40, 0], seed=2,
                               poison=False)
    for conv, dt in ((workloads.to_int8, torch.int8), (workloads.to_fp8, torch.uint8)):
        c = conv(w)
        assert c.pool.dtype == dt and c.pool.shape == (w.NB, 2, w.Hkv, w.bs, w.D)
        assert torch.equal(c.block_table, w.block_table) and torch.equal(c.lens, w.lens)
        assert torch.equal(c.q, w.q) and torch.equal(c.k_new, w.k_new) and torch.equal(c.v_new, w.v_new)
        assert c.scales.shape == (w.NB, 2, w.Hkv) and bool((c.scales > 0).all())
        assert c.block_stride == 2 * w.Hkv * w.bs * w.D
    f = workloads.to_fp8(w)
    assert not bool(((f.pool & 0x7F) == 0x7F).any())           # no NaN codes drawn
