"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays out a paged KV cache the way a
block allocator would (a seeded permutation of physical block ids, a table row
per sequence, -1 for unallocated entries).  It holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle may consume its output.

The five workloads mirror the structure of the pages' examples:

1. tiny MHA fp32 case with lengths [32, 128, 64, 96] and block_size 16, the
   4-request example of "KV Cache and BlockManager" (dpshk.com/news/5906718)
   section 2;
2. a Llama-7B-like layer (32 heads, head_dim 128, fp16, block_size 16) with
   request lengths in 450..520, the length window of that page's section 3;
3. a long-tail serving mix: log-normal lengths with median 87 (the short-query
   traffic of the same section), sigma 1.0, clipped to [4, 4096], swept over
   block sizes 8/16/32/64;
4. a GQA 70B-like layer (64 query heads, 8 KV heads, bf16, length 2048) at
   block sizes 16 and 256 (the 256-token block of "KV Cache paging in LLM
   inference", intelliparadigm.com, section 2.1);
5. 4 beams of 32768 tokens sharing a 30000-token prefix through shared
   physical blocks (reference-counted sharing of the vLLM course, ch. 3 "KV
   Block design", section 3.4), block_size 32.

Lengths given here are the cache contents BEFORE the step's append; the step
appends one token at position L and then attends over L + 1 tokens.

Random recipe: torch generator seeded with 1000 + workload index; lengths
first, then the physical-id permutation, then the pool, q, k_new, v_new, all
N(0, 1) drawn in float32 and cast to the cache dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    B: int                      # sequences
    H: int                      # query heads
    Hkv: int                    # kv heads
    D: int                      # head_dim
    bs: int                     # block_size (tokens per block)
    NB: int                     # physical blocks in the pool
    MB: int                     # max_blocks_per_seq (block_table row length)
    dtype: torch.dtype
    lens: torch.Tensor          # int32 [B], cache length before the append
    block_table: torch.Tensor   # int32 [B][MB], -1 where unallocated
    pool: torch.Tensor          # [NB][2][Hkv][bs][D]: K and V co-located per block
    q: torch.Tensor             # [B][H][D]
    k_new: torch.Tensor         # [B][Hkv][D]
    v_new: torch.Tensor         # [B][Hkv][D]
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def block_stride(self) -> int:
        """Elements between consecutive physical blocks of one pool."""
        return 2 * self.Hkv * self.bs * self.D

    @property
    def v_offset(self) -> int:
        """Elements from the K half of a block to its V half."""
        return self.Hkv * self.bs * self.D

    def k_flat(self) -> torch.Tensor:
        return self.pool.view(-1)

    def v_flat(self) -> torch.Tensor:
        return self.pool.view(-1)[self.v_offset:]

    def to(self, device) -> "Workload":
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                 for k, v in self.__dict__.items()}
        return Workload(**moved)

    def clone(self) -> "Workload":
        copied = {k: (v.clone() if isinstance(v, torch.Tensor) else v)
                  for k, v in self.__dict__.items()}
        return Workload(**copied)


def _randn(shape, gen, dtype, device):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(dtype)


def _alloc_tables(nblk_per_seq, NB, MB, gen):
    """Distinct physical ids from a seeded permutation, handed out in order."""
    need = int(sum(nblk_per_seq))
    if need > NB:
        raise ValueError(f"pool of {NB} blocks cannot hold {need}")
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    table = torch.full((len(nblk_per_seq), MB), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(nblk_per_seq):
        table[b, :n] = perm[cursor:cursor + n]
        cursor += n
    return table


def _ceil_div(a, b):
    return -(-a // b)


def poison_pool(w: Workload, after_append: bool = False) -> None:
    """Fill every slot the step never reads with NaN/inf/huge values.

    Slots at positions >= L (>= L + 1 when after_append) in each sequence's
    last block, and every block no table row references, are poisoned.  The
    valid-length rule ("A strange KV Cache bug", dpshk.com/news/5937191,
    section 2.4) says none of them may influence the output.
    """
    bad = [float("nan"), float("inf"), -float("inf"), 3.0e38 if w.dtype != torch.float16 else 6.0e4]
    pool = w.pool
    used = torch.zeros(w.NB, dtype=torch.bool)
    flat_tab = w.block_table.cpu()
    for b in range(w.B):
        L = int(w.lens[b]) + (1 if after_append else 0)
        n_alloc = int((flat_tab[b] >= 0).sum())
        for j in range(n_alloc):
            blk = int(flat_tab[b, j])
            used[blk] = True
            lo = max(0, L - j * w.bs)
            if lo < w.bs:
                val = bad[(b + j) % len(bad)]
                pool[blk, :, :, lo:, :] = val
    unused = (~used).nonzero().flatten()
    for i, blk in enumerate(unused.tolist()):
        pool[blk] = bad[i % len(bad)]


def make_workload(index: int, *, block_size: int | None = None, device="cpu",
                  seed: int | None = None, poison: bool = False,
                  batch: int | None = None, max_len: int | None = None) -> Workload:
    """Build workload `index` (1..5) on `device`.

    block_size overrides the default block size where the workload sweeps it
    (3: 8/16/32/64, 4: 16/256).  batch and max_len shrink a workload for fast
    parity runs while keeping its structure.
    """
    seed = 1000 + index if seed is None else seed
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    dev_gen = gen if str(device) == "cpu" else torch.Generator(device=device)
    if dev_gen is not gen:
        dev_gen.manual_seed(seed + 7919)

    meta = {"index": index, "seed": seed}
    if index == 1:
        B, H, Hkv, D, bs, dtype = 4, 4, 4, 64, block_size or 16, torch.float32
        lens = torch.tensor([32, 128, 64, 96], dtype=torch.int32)
        NB = 64 * 16 // bs
        name = "tiny-mha-f32"
    elif index == 2:
        B, H, Hkv, D, bs, dtype = batch or 64, 32, 32, 128, block_size or 16, torch.float16
        lens = torch.randint(450, 521, (B,), generator=gen, dtype=torch.int32)
        NB = 4096 * 16 // bs
        name = "llama7b-mha-f16"
    elif index == 3:
        B, H, Hkv, D, bs, dtype = batch or 256, 32, 32, 128, block_size or 16, torch.bfloat16
        z = torch.randn(B, generator=gen, dtype=torch.float64)
        lens = torch.clamp(torch.round(torch.exp(math.log(87.0) + 1.0 * z)), 4, 4096).to(torch.int32)
        NB = None
        name = "longtail-mha-bf16"
        meta["sigma"] = 1.0
    elif index == 4:
        B, H, Hkv, D, bs, dtype = batch or 32, 64, 8, 128, block_size or 16, torch.bfloat16
        lens = torch.full((B,), 2048, dtype=torch.int32)
        NB = None
        name = "gqa70b-bf16"
    elif index == 5:
        return _make_shared_beams(gen, dev_gen, device, poison, seed,
                                  block_size or 32, max_len)
    else:
        raise ValueError(f"unknown workload {index}")

    if max_len is not None:
        lens = torch.clamp(lens, max=max_len)
    nblk = [_ceil_div(int(L) + 1, bs) for L in lens]
    MB = max(nblk) + 2
    if NB is None:
        NB = int(math.ceil(1.1 * sum(nblk))) + 16
    NB = max(NB, sum(nblk))
    table = _alloc_tables(nblk, NB, MB, gen)
    pool = _randn((NB, 2, Hkv, bs, D), dev_gen, dtype, device)
    q = _randn((B, H, D), dev_gen, dtype, device)
    k_new = _randn((B, Hkv, D), dev_gen, dtype, device)
    v_new = _randn((B, Hkv, D), dev_gen, dtype, device)
    w = Workload(name, B, H, Hkv, D, bs, NB, MB, dtype, lens, table.to(device), pool,
                 q, k_new, v_new, 1.0 / math.sqrt(D), meta)
    w.lens = w.lens.to(device)
    if poison:
        poison_pool(w)
    return w


def _make_shared_beams(gen, dev_gen, device, poison, seed, bs, max_len):
    """4 beams of 32768 tokens; the first 30000 tokens are shared.

    The 30000-token prefix fills 937 whole blocks of 32 (29984 tokens) that
    every beam's table references (reference count 4); the prefix's last 16
    tokens sit in a partly filled block that each beam holds its own copy of
    (copy on write), followed by each beam's private tail.
    """
    B, H, Hkv, D, dtype = 4, 32, 32, 128, torch.bfloat16
    L = 32768 if max_len is None else max_len
    prefix = 30000 if max_len is None else (L * 30000) // 32768
    n_shared = prefix // bs                      # whole blocks of the prefix
    nblk = _ceil_div(L + 1, bs)                  # blocks per beam after the append
    n_private = nblk - n_shared
    NB = 2048 if max_len is None else max(64, n_shared + B * n_private + 8)
    MB = nblk + 2
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    table = torch.full((B, MB), -1, dtype=torch.int32)
    for b in range(B):
        table[b, :n_shared] = perm[:n_shared]
        start = n_shared + b * n_private
        table[b, n_shared:nblk] = perm[start:start + n_private]
    pool = _randn((NB, 2, Hkv, bs, D), dev_gen, dtype, device)
    # the partly shared block: copy the prefix rows of beam 0 into the others
    rows = prefix - n_shared * bs
    if rows > 0:
        src = int(table[0, n_shared])
        for b in range(1, B):
            dst = int(table[b, n_shared])
            pool[dst, :, :, :rows, :] = pool[src, :, :, :rows, :]
    q = _randn((B, H, D), dev_gen, dtype, device)
    k_new = _randn((B, Hkv, D), dev_gen, dtype, device)
    v_new = _randn((B, Hkv, D), dev_gen, dtype, device)
    lens = torch.full((B,), L, dtype=torch.int32)
    meta = {"index": 5, "seed": seed, "prefix": prefix, "shared_blocks": n_shared,
            "private_blocks_per_beam": n_private,
            "unique_blocks": n_shared + B * n_private}
    w = Workload("shared-beams-bf16", B, H, Hkv, D, bs, NB, MB, dtype, lens.to(device),
                 table.to(device), pool, q, k_new, v_new, 1.0 / math.sqrt(D), meta)
    if poison:
        poison_pool(w)
    return w


def unshare(w: Workload) -> Workload:
    """Same logical data with every table row pointing at private copies.

    Used to check that reading shared physical blocks gives exactly what
    private copies give.
    """
    rows = []
    blocks = []
    tab = w.block_table.cpu()
    nxt = 0
    for b in range(w.B):
        n = int((tab[b] >= 0).sum())
        row = torch.full((w.MB,), -1, dtype=torch.int32)
        for j in range(n):
            blocks.append(int(tab[b, j]))
            row[j] = nxt
            nxt += 1
        rows.append(row)
    src = torch.tensor(blocks, dtype=torch.long, device=w.pool.device)
    pool = w.pool.index_select(0, src).contiguous()
    out = w.clone()
    out.pool = pool
    out.NB = pool.shape[0]
    out.block_table = torch.stack(rows).to(w.block_table.device)
    return out


def make_generic(*, B, H, Hkv, D, bs, dtype, lens, seed=0, device="cpu", poison=True,
                 extra_blocks=3, separate_pools=False, name="generic") -> Workload:
    """Any shape: lens (pre-append) per sequence, shuffled distinct block ids.

    With separate_pools the K and V halves of each block are placed in two
    different regions of one buffer (block_stride = Hkv*bs*D), exercising the
    non-co-located layout.
    """
    gen = torch.Generator().manual_seed(seed)
    lens = torch.as_tensor(lens, dtype=torch.int32)
    nblk = [_ceil_div(int(L) + 1, bs) for L in lens]
    MB = max(nblk) + 2
    NB = sum(nblk) + extra_blocks
    table = _alloc_tables(nblk, NB, MB, gen)
    pool = _randn((NB, 2, Hkv, bs, D), gen, dtype, "cpu")
    q = _randn((B, H, D), gen, dtype, "cpu")
    k_new = _randn((B, Hkv, D), gen, dtype, "cpu")
    v_new = _randn((B, Hkv, D), gen, dtype, "cpu")
    w = Workload(name, B, H, Hkv, D, bs, NB, MB, dtype, lens, table, pool, q, k_new, v_new,
                 1.0 / math.sqrt(D), {"seed": seed, "separate_pools": separate_pools})
    if poison:
        poison_pool(w)
    if separate_pools:
        w = SeparatePoolWorkload(**w.__dict__)
    return w.to(device) if str(device) != "cpu" else w


@dataclass
class SeparatePoolWorkload(Workload):
    """Same data as a co-located pool, stored as [2][NB][Hkv][bs][D]: all K
    blocks first, then all V blocks."""

    @property
    def block_stride(self) -> int:
        return self.Hkv * self.bs * self.D

    @property
    def v_offset(self) -> int:
        return self.NB * self.Hkv * self.bs * self.D

    def __post_init__(self):
        if not self.meta.get("k_blocks_first"):
            self.pool = self.pool.transpose(0, 1).contiguous()
            self.meta = dict(self.meta, k_blocks_first=True)

    def to(self, device):
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                 for k, v in self.__dict__.items()}
        return SeparatePoolWorkload(**moved)

    def clone(self):
        copied = {k: (v.clone() if isinstance(v, torch.Tensor) else v)
                  for k, v in self.__dict__.items()}
        return SeparatePoolWorkload(**copied)


def with_long_sequence(w: Workload, length: int, *, seed: int = 7, device="cpu") -> Workload:
    """The same shape as `w` with its last sequence replaced by one of
    `length` tokens (pre-append): a serving batch where one long-context
    request runs beside many ordinary ones.  Fresh seeded data, shuffled
    block ids, unpoisoned."""
    lens = [int(x) for x in w.lens.cpu()]
    lens[-1] = int(length)
    return make_generic(B=w.B, H=w.H, Hkv=w.Hkv, D=w.D, bs=w.bs, dtype=w.dtype, lens=lens,
                        seed=seed, device=device, poison=False,
                        name=f"{w.name}+1x{length}")


@dataclass
class Int8Workload:
    """A quantised cache in the layout of `Workload`: pool [NB][2][Hkv][bs][D]
    of one-byte codes (int8, or uint8 E4M3 codes for an fp8 cache), scales
    [NB][2][Hkv] fp32 (K, V per block and kv head), q and the new rows in
    `dtype`."""
    name: str
    B: int
    H: int
    Hkv: int
    D: int
    bs: int
    NB: int
    MB: int
    dtype: torch.dtype
    lens: torch.Tensor
    block_table: torch.Tensor
    pool: torch.Tensor
    scales: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    scale: float
    meta: dict

    @property
    def block_stride(self) -> int:
        return 2 * self.Hkv * self.bs * self.D

    @property
    def v_offset(self) -> int:
        return self.Hkv * self.bs * self.D

    def k_flat(self) -> torch.Tensor:
        return self.pool.view(-1)

    def v_flat(self) -> torch.Tensor:
        return self.pool.view(-1)[self.v_offset:]

    def to(self, device) -> "Int8Workload":
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                 for k, v in self.__dict__.items()}
        return Int8Workload(**moved)


def to_int8(w: Workload, *, seed: int = 17, scale_range=(0.004, 0.012), device="cpu") -> Int8Workload:
    """The int8 counterpart of workload `w` (same shape, table, lengths, q
    and new rows): seeded uniform codes in [-127, 127] and per-(block, K|V,
    kv head) scales drawn uniformly from scale_range, so the values the
    codes stand for have a spread comparable to N(0, 1) data.  The codes and
    scales are drawn on `device` (a CUDA generator gives other numbers than
    the CPU one for the same seed) and every tensor lands there."""
    gen = torch.Generator(device=device).manual_seed(seed)
    pool = torch.randint(-127, 128, (w.NB, 2, w.Hkv, w.bs, w.D), generator=gen, dtype=torch.int8,
                         device=device)
    lo, hi = scale_range
    scales = (torch.rand((w.NB, 2, w.Hkv), generator=gen, dtype=torch.float32, device=device)
              * (hi - lo) + lo)
    mv = lambda t: t.to(device) if isinstance(t, torch.Tensor) else t
    return Int8Workload(w.name + "-int8", w.B, w.H, w.Hkv, w.D, w.bs, w.NB, w.MB, w.dtype,
                        mv(w.lens), mv(w.block_table), pool, scales, mv(w.q), mv(w.k_new),
                        mv(w.v_new), w.scale, dict(w.meta, int8_seed=seed))


def to_fp8(w: Workload, *, seed: int = 19, scale_range=(0.002, 0.006), device="cpu") -> Int8Workload:
    """The fp8 (E4M3) counterpart of workload `w` (same shape, table,
    lengths, q and new rows): seeded uniform bytes over the finite E4M3 codes
    (the two NaN codes are redrawn as zero) and per-(block, K|V, kv head)
    scales drawn uniformly from scale_range, so that the values the codes
    stand for stay within a few units.  The pool is uint8.  Drawn on
    `device`, as to_int8."""
    gen = torch.Generator(device=device).manual_seed(seed)
    pool = torch.randint(0, 256, (w.NB, 2, w.Hkv, w.bs, w.D), generator=gen, dtype=torch.uint8,
                         device=device)
    pool[(pool & 0x7F) == 0x7F] = 0
    lo, hi = scale_range
    scales = (torch.rand((w.NB, 2, w.Hkv), generator=gen, dtype=torch.float32, device=device)
              * (hi - lo) + lo)
    mv = lambda t: t.to(device) if isinstance(t, torch.Tensor) else t
    return Int8Workload(w.name + "-fp8", w.B, w.H, w.Hkv, w.D, w.bs, w.NB, w.MB, w.dtype,
                        mv(w.lens), mv(w.block_table), pool, scales, mv(w.q), mv(w.k_new),
                        mv(w.v_new), w.scale, dict(w.meta, fp8_seed=seed))


def make_prefix_groups(*, group_sizes, shared_blocks, tails, H, Hkv, D, bs, dtype, seed=0,
                       poison=True, device="cpu") -> Workload:
    """Sequences forked from common prompts: group i has group_sizes[i]
    members whose tables share the same shared_blocks[i] physical blocks
    (reference count = group size), then each member's private blocks for
    its own tails[b] tokens.  meta["group_first"] / meta["shared_tokens"]
    describe the groups (group_first has one entry more than the groups)."""
    gen = torch.Generator().manual_seed(seed)
    B = sum(group_sizes)
    assert len(tails) == B and len(shared_blocks) == len(group_sizes)
    lens, first, shared = [], [0], []
    for gi, n in enumerate(group_sizes):
        for m in range(n):
            lens.append(shared_blocks[gi] * bs + tails[first[-1] + m])
        shared.append(shared_blocks[gi] * bs)
        first.append(first[-1] + n)
    nblk = [_ceil_div(L + 1, bs) for L in lens]
    MB = max(nblk) + 2
    NB = sum(shared_blocks) + sum(nblk[b] - shared_blocks[gi] for gi in range(len(group_sizes))
                                  for b in range(first[gi], first[gi + 1])) + 4
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    table = torch.full((B, MB), -1, dtype=torch.int32)
    k = 0
    for gi in range(len(group_sizes)):
        common = perm[k:k + shared_blocks[gi]]
        k += shared_blocks[gi]
        for b in range(first[gi], first[gi + 1]):
            table[b, :shared_blocks[gi]] = common
            own = nblk[b] - shared_blocks[gi]
            table[b, shared_blocks[gi]:nblk[b]] = perm[k:k + own]
            k += own
    pool = _randn((NB, 2, Hkv, bs, D), gen, dtype, "cpu")
    q = _randn((B, H, D), gen, dtype, "cpu")
    k_new = _randn((B, Hkv, D), gen, dtype, "cpu")
    v_new = _randn((B, Hkv, D), gen, dtype, "cpu")
    w = Workload("prefix-groups", B, H, Hkv, D, bs, NB, MB, dtype,
                 torch.tensor(lens, dtype=torch.int32), table, pool, q, k_new, v_new,
                 1.0 / math.sqrt(D), {"seed": seed, "group_first": first, "shared_tokens": shared})
    if poison:
        poison_pool(w)
    return w.to(device) if str(device) != "cpu" else w
