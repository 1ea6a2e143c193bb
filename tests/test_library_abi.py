"""CPU checks of the C ABI: the library builds, loads and exports every
function include/pagedattn.h declares, and host-side validation rejects bad
arguments before anything is enqueued.  Only calls that fail validation are
made here (they return before touching the CUDA runtime), so no GPU is
needed."""
import ctypes
import os
import re
import subprocess

import pytest

import pagedattention_decode_paged_gb300 as pa
from pagedattention_decode_paged_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("paged_kv_append", "paged_attention_decode", "paged_attention_decode_partial",
              "paged_attention_decode_reduce", "paged_attention_partial_workspace",
              "pa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", str(pa.LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(pa.EXPORTED) <= exported


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "pagedattn.h"\nint main(void){ pa_shape s; (void)s; return 0; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{ROOT}/include", "-c", str(src),
                    "-o", str(tmp_path / "t.o")], check=True)


def test_version_and_status_strings(lib):
    assert pa.version() == 10000
    for s in range(6):
        assert pa.status_string(s)
    assert pa.status_string(0) == "ok"
    assert "unknown" in pa.status_string(99)


def base_shape(**over):
    d = dict(batch=2, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
             max_blocks_per_seq=8, num_blocks=64, block_stride=2 * 2 * 16 * 128, dtype=pa.PA_BF16)
    d.update(over)
    return pa.make_shape(**d)


def test_path_selection(lib):
    assert pa.paged_attention_decode_path(base_shape()) == pa.PA_PATH_TENSOR_GQA
    assert pa.paged_attention_decode_path(base_shape(num_kv_heads=8, block_stride=2 * 8 * 16 * 128)) \
        == pa.PA_PATH_SIMT                                             # MHA
    assert pa.paged_attention_decode_path(base_shape(dtype=pa.PA_F32)) == pa.PA_PATH_SIMT
    assert pa.paged_attention_decode_path(base_shape(block_size=4, block_stride=2 * 2 * 4 * 128)) \
        == pa.PA_PATH_SIMT                                             # block too small for TMA boxes
    assert pa.paged_attention_decode_path(base_shape(head_dim=256, block_stride=2 * 2 * 16 * 256)) \
        == pa.PA_PATH_SIMT
    assert pa.paged_attention_decode_path(base_shape(num_heads=7)) == pa.PA_PATH_INVALID
    assert pa.paged_attention_decode_path(base_shape(head_dim=96, block_stride=2 * 2 * 16 * 96)) \
        == pa.PA_PATH_INVALID


def test_workspace_size(lib):
    s = base_shape()
    n = pa.paged_attention_partial_workspace(s, 32)
    P = (8 * 16 + 31) // 32
    BH = 2 * 8
    assert n == ((8 * BH * P + 15) // 16) * 16 + 4 * BH * P * 128
    assert pa.paged_attention_partial_workspace(s, 0) == 0
    assert pa.paged_attention_partial_workspace(s, 24) == 0          # not a multiple of 16


FAKE = 1 << 20          # a 16-byte aligned address that is never dereferenced on the host


def call_decode(lib, shape, out=FAKE, q=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, sl=FAKE, scale=0.1):
    return lib.paged_attention_decode(ctypes.byref(shape) if shape is not None else None,
                                      out, q, kp, vp, bt, sl, scale, None, None)


def test_decode_rejects_bad_arguments(lib):
    assert call_decode(lib, None) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(num_heads=7)) == pa.PA_ERR_INVALID_ARG   # H % Hkv
    assert call_decode(lib, base_shape(dtype=7)) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(block_stride=10)) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(head_dim=96, block_stride=2 * 2 * 16 * 96)) \
        == pa.PA_ERR_UNSUPPORTED
    assert call_decode(lib, base_shape(), q=None) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(), out=None) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(), kp=FAKE + 8) == pa.PA_ERR_MISALIGNED
    assert call_decode(lib, base_shape(), out=FAKE + 2) == pa.PA_ERR_MISALIGNED
    assert call_decode(lib, base_shape(), scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    assert call_decode(lib, base_shape(block_stride=2 * 2 * 16 * 128 + 1)) == pa.PA_ERR_MISALIGNED
    assert call_decode(lib, base_shape(max_blocks_per_seq=1 << 28, block_size=16)) == pa.PA_ERR_INVALID_ARG
    # an empty batch is valid and enqueues nothing
    assert call_decode(lib, base_shape(batch=0), q=None, out=None) == pa.PA_OK


def test_append_rejects_bad_arguments(lib):
    s = base_shape()
    f = lib.paged_kv_append
    assert f(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == pa.PA_ERR_MISALIGNED
    assert f(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None) == pa.PA_ERR_INVALID_ARG


def test_fused_append_decode_rejects_bad_arguments(lib):
    f = lib.paged_attention_decode_append
    s = base_shape()
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    assert f(None, *ok, 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), None, *ok[1:], 0.1, None, None) == pa.PA_ERR_INVALID_ARG      # out
    assert f(ctypes.byref(s), FAKE, FAKE, None, *ok[3:], 0.1, None, None) == pa.PA_ERR_INVALID_ARG  # k_new
    assert f(ctypes.byref(s), *ok[:7], None, 0.1, None, None) == pa.PA_ERR_INVALID_ARG     # positions
    assert f(ctypes.byref(s), FAKE, FAKE, FAKE + 4, *ok[3:], 0.1, None, None) == pa.PA_ERR_MISALIGNED
    assert f(ctypes.byref(s), *ok, float("inf"), None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(base_shape(batch=0)), *ok, 0.1, None, None) == pa.PA_OK


def test_split_rejects_bad_arguments(lib):
    s = base_shape()
    need = pa.paged_attention_partial_workspace(s, 32)
    part = lib.paged_attention_decode_partial
    red = lib.paged_attention_decode_reduce
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, 0.1)
    assert part(ctypes.byref(s), *args, 24, FAKE, need, None, None) == pa.PA_ERR_INVALID_ARG
    assert part(ctypes.byref(s), *args, 32, FAKE, need - 1, None, None) == pa.PA_ERR_WORKSPACE
    assert part(ctypes.byref(s), *args, 32, None, need, None, None) == pa.PA_ERR_INVALID_ARG
    assert part(ctypes.byref(s), *args, 32, FAKE + 8, need, None, None) == pa.PA_ERR_MISALIGNED
    assert red(ctypes.byref(s), FAKE, FAKE, need - 1, FAKE, 32, None, None) == pa.PA_ERR_WORKSPACE
    assert red(ctypes.byref(s), FAKE, FAKE, need, FAKE, 0, None, None) == pa.PA_ERR_INVALID_ARG
    assert red(ctypes.byref(s), None, FAKE, need, FAKE, 32, None, None) == pa.PA_ERR_INVALID_ARG


def test_balanced_rejects_bad_arguments(lib):
    f = lib.paged_attention_decode_balanced
    s = base_shape()
    # (out, q, k_pool, v_pool, block_table, seq_lens, positions, k_new, v_new)
    plain = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None)
    fused = (FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE)
    tail = (0.1, 0, FAKE, 1 << 30, None, None)
    assert f(None, *plain, *tail) == pa.PA_ERR_INVALID_ARG
    both = plain[:6] + (FAKE,) + plain[7:]
    neither = plain[:5] + (None,) + plain[6:]
    assert f(ctypes.byref(s), *both, *tail) == pa.PA_ERR_INVALID_ARG      # seq_lens and positions
    assert f(ctypes.byref(s), *neither, *tail) == pa.PA_ERR_INVALID_ARG   # neither
    assert f(ctypes.byref(s), *fused[:7], None, FAKE, *tail) == pa.PA_ERR_INVALID_ARG  # k_new
    assert f(ctypes.byref(s), *plain, 0.1, -1, FAKE, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), *plain, float("nan"), 0, FAKE, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), *plain, 0.1, 0, None, 1 << 30, None, None) == pa.PA_ERR_INVALID_ARG
    assert f(ctypes.byref(s), *plain, 0.1, 0, FAKE + 8, 1 << 30, None, None) == pa.PA_ERR_MISALIGNED
    assert f(ctypes.byref(s), FAKE + 2, *plain[1:], *tail) == pa.PA_ERR_MISALIGNED
    assert f(ctypes.byref(base_shape(head_dim=96, block_stride=2 * 2 * 16 * 96)), *plain, *tail) \
        == pa.PA_ERR_UNSUPPORTED
    assert f(ctypes.byref(base_shape(batch=0)), *plain, *tail) == pa.PA_OK
    # sizes are queried on the device: no device here, so no size
    assert pa.paged_attention_balanced_workspace(base_shape(batch=0)) == 0


def test_int8_rejects_bad_arguments(lib):
    s8 = base_shape(block_stride=2 * 2 * 16 * 128)   # bytes: one per element
    dec = lib.paged_attention_decode_int8
    app = lib.paged_kv_append_int8
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)   # out, q, k_pool, v_pool, scales, table, lens
    assert dec(None, *ok, 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    assert dec(ctypes.byref(base_shape(head_dim=32, block_stride=2 * 2 * 16 * 32)), *ok, 0.1, None, None) \
        == pa.PA_ERR_UNSUPPORTED
    assert dec(ctypes.byref(base_shape(block_stride=2 * 2 * 16 * 128 + 8)), *ok, 0.1, None, None) \
        == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), *ok[:4], None, *ok[5:], 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    assert dec(ctypes.byref(s8), *ok[:4], FAKE + 2, *ok[5:], 0.1, None, None) == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), FAKE, FAKE, FAKE + 8, *ok[3:], 0.1, None, None) == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), *ok, float("inf"), None, None) == pa.PA_ERR_INVALID_ARG
    assert dec(ctypes.byref(base_shape(batch=0)), *ok, 0.1, None, None) == pa.PA_OK
    ok_a = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)  # k_new, v_new, k_pool, v_pool, scales, table, pos
    assert app(ctypes.byref(s8), *ok_a[:4], None, *ok_a[5:], None, None) == pa.PA_ERR_INVALID_ARG
    assert app(ctypes.byref(s8), *ok_a[:2], FAKE + 4, *ok_a[3:], None, None) == pa.PA_ERR_MISALIGNED
    assert app(ctypes.byref(base_shape(head_dim=96, block_stride=2 * 2 * 16 * 96)), *ok_a, None, None) \
        == pa.PA_ERR_UNSUPPORTED


def test_fp8_rejects_bad_arguments(lib):
    s8 = base_shape(block_stride=2 * 2 * 16 * 128)   # bytes: one per element
    dec = lib.paged_attention_decode_fp8
    app = lib.paged_kv_append_fp8
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)   # out, q, k_pool, v_pool, scales, table, lens
    assert dec(None, *ok, 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    # head_dim 64, 128 and 256 only
    for D in (32, 96, 512):
        assert dec(ctypes.byref(base_shape(head_dim=D, block_stride=2 * 2 * 16 * D)), *ok, 0.1, None, None) \
            == pa.PA_ERR_UNSUPPORTED
        assert app(ctypes.byref(base_shape(head_dim=D, block_stride=2 * 2 * 16 * D)), *ok, None, None) \
            == pa.PA_ERR_UNSUPPORTED
    assert dec(ctypes.byref(base_shape(block_stride=2 * 2 * 16 * 128 + 8)), *ok, 0.1, None, None) \
        == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), *ok[:4], None, *ok[5:], 0.1, None, None) == pa.PA_ERR_INVALID_ARG
    assert dec(ctypes.byref(s8), *ok[:4], FAKE + 2, *ok[5:], 0.1, None, None) == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), FAKE, FAKE, FAKE + 8, *ok[3:], 0.1, None, None) == pa.PA_ERR_MISALIGNED
    assert dec(ctypes.byref(s8), *ok, float("nan"), None, None) == pa.PA_ERR_INVALID_ARG
    assert dec(ctypes.byref(base_shape(batch=0)), *ok, 0.1, None, None) == pa.PA_OK
    ok_a = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)  # k_new, v_new, k_pool, v_pool, scales, table, pos
    assert app(ctypes.byref(s8), *ok_a[:4], None, *ok_a[5:], None, None) == pa.PA_ERR_INVALID_ARG
    assert app(ctypes.byref(s8), *ok_a[:2], FAKE + 4, *ok_a[3:], None, None) == pa.PA_ERR_MISALIGNED
    # fp32 queries and rows are accepted (the shape check passes; no device here)
    assert app(ctypes.byref(base_shape(batch=0, dtype=pa.PA_F32, block_stride=2 * 2 * 16 * 128)), *ok_a,
               None, None) == pa.PA_OK


def test_shared_prefix_rejects_bad_arguments(lib):
    f = lib.paged_attention_decode_shared_prefix
    s = base_shape()
    need = pa.paged_attention_partial_workspace(s, 32)
    first = (ctypes.c_int32 * 3)(0, 1, 2)
    shared = (ctypes.c_int32 * 2)(32, 0)
    io = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)   # out, q, k_pool, v_pool, table, lens

    def call(shape=s, n=2, fst=first, sh=shared, ptok=32, ws=FAKE, nbytes=need):
        return f(ctypes.byref(shape), *io, n, ctypes.cast(fst, ctypes.c_void_p) if fst is not None else None,
                 ctypes.cast(sh, ctypes.c_void_p) if sh is not None else None, 0.1, ptok, ws, nbytes, None, None)

    assert call(ptok=24) == pa.PA_ERR_INVALID_ARG
    assert call(n=17) == pa.PA_ERR_INVALID_ARG
    assert call(fst=None) == pa.PA_ERR_INVALID_ARG
    assert call(shape=base_shape(dtype=pa.PA_F32, block_stride=2 * 2 * 16 * 128)) == pa.PA_ERR_UNSUPPORTED
    assert call(nbytes=need - 1) == pa.PA_ERR_WORKSPACE
    assert call(fst=(ctypes.c_int32 * 3)(0, 2, 1)) == pa.PA_ERR_INVALID_ARG       # not ascending
    assert call(fst=(ctypes.c_int32 * 3)(0, 1, 3)) == pa.PA_ERR_INVALID_ARG       # past the batch
    assert call(sh=(ctypes.c_int32 * 2)(-16, 0)) == pa.PA_ERR_INVALID_ARG
    wide = base_shape(batch=3, num_heads=16, num_kv_heads=2)   # 2 members x 8 heads = 16: fine; 3 x 8 not
    assert call(shape=wide, n=1, fst=(ctypes.c_int32 * 2)(0, 3), sh=(ctypes.c_int32 * 1)(64),
                nbytes=1 << 30) == pa.PA_ERR_UNSUPPORTED
    assert call(shape=base_shape(batch=0)) == pa.PA_OK


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_shared_prefix_codes_reject_bad_arguments(lib, fmt):
    f = getattr(lib, f"paged_attention_decode_shared_prefix_{fmt}")
    s = base_shape()   # block_stride counts bytes: one per element
    need = pa.paged_attention_partial_workspace(s, 32)
    first = (ctypes.c_int32 * 3)(0, 1, 2)
    shared = (ctypes.c_int32 * 2)(32, 0)

    def call(shape=s, n=2, fst=first, sh=shared, ptok=32, ws=FAKE, nbytes=need, kp=FAKE, scales=FAKE,
             scale=0.1):
        return f(ctypes.byref(shape), FAKE, FAKE, kp, FAKE, scales, FAKE, FAKE, n,
                 ctypes.cast(fst, ctypes.c_void_p) if fst is not None else None,
                 ctypes.cast(sh, ctypes.c_void_p) if sh is not None else None, scale, ptok, ws, nbytes,
                 None, None)

    assert call(ptok=24) == pa.PA_ERR_INVALID_ARG
    assert call(n=17) == pa.PA_ERR_INVALID_ARG
    assert call(fst=None) == pa.PA_ERR_INVALID_ARG
    assert call(scale=float("inf")) == pa.PA_ERR_INVALID_ARG
    assert call(scales=None) == pa.PA_ERR_INVALID_ARG
    assert call(scales=FAKE + 2) == pa.PA_ERR_MISALIGNED
    assert call(kp=FAKE + 8) == pa.PA_ERR_MISALIGNED
    assert call(shape=base_shape(block_stride=2 * 2 * 16 * 128 + 8)) == pa.PA_ERR_MISALIGNED
    assert call(shape=base_shape(head_dim=256, block_stride=2 * 2 * 16 * 256)) == pa.PA_ERR_UNSUPPORTED
    f32 = base_shape(dtype=pa.PA_F32)
    if fmt == "int8":   # fp32 queries over int8 have no tensor-core kernel
        assert call(shape=f32) == pa.PA_ERR_UNSUPPORTED
    else:               # fp8 takes them: the call gets as far as the workspace check
        assert call(shape=f32, nbytes=need - 1) == pa.PA_ERR_WORKSPACE
    assert call(nbytes=need - 1) == pa.PA_ERR_WORKSPACE
    assert call(fst=(ctypes.c_int32 * 3)(0, 2, 1)) == pa.PA_ERR_INVALID_ARG       # not ascending
    wide = base_shape(batch=3, num_heads=16, num_kv_heads=2)   # 3 members x 8 heads > 16 columns
    assert call(shape=wide, n=1, fst=(ctypes.c_int32 * 2)(0, 3), sh=(ctypes.c_int32 * 1)(64),
                nbytes=1 << 30) == pa.PA_ERR_UNSUPPORTED
    assert call(shape=base_shape(batch=0)) == pa.PA_OK


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
def test_shared_prefix_codes_wrappers_marshal_their_arguments(lib, fmt):
    """The Python wrappers pass every argument through ctypes (a mismatch with
    the declared argument types raises before the call); the library then
    rejects the partition size on the host, before any CUDA call (the
    default stream is passed as 0, so torch needs no device either)."""
    import torch
    fn = getattr(pa, f"paged_attention_decode_shared_prefix_{fmt}")
    B, H, Hkv, D, bs, NB, MB = 2, 4, 2, 128, 16, 8, 4
    q = torch.zeros((B, H, D), dtype=torch.bfloat16)
    pool = torch.zeros((NB, 2, Hkv, bs, D), dtype=torch.int8 if fmt == "int8" else torch.uint8)
    flat = pool.view(-1)
    scales = torch.ones((NB, 2, Hkv), dtype=torch.float32)
    table = torch.zeros((B, MB), dtype=torch.int32)
    lens = torch.ones(B, dtype=torch.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(pa.PagedAttnError) as ei:
        fn(torch.empty_like(q), q, flat, flat[Hkv * bs * D:], scales, table, lens, 0.1, 24, ws,
           group_first=[0, 2], shared_tokens=[32], num_kv_heads=Hkv, block_size=bs, num_blocks=NB,
           block_stride=2 * Hkv * bs * D, stream=0)
    assert ei.value.status == pa.PA_ERR_INVALID_ARG
    call = fn(torch.empty_like(q), q, flat, flat[Hkv * bs * D:], scales, table, lens, 0.1, 24, ws,
              group_first=[0, 2], shared_tokens=[32], num_kv_heads=Hkv, block_size=bs, num_blocks=NB,
              block_stride=2 * Hkv * bs * D, stream=0, prepare=True)
    with pytest.raises(pa.PagedAttnError):
        call()


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(pa, "LIB_PATH", tmp_path / "missing.so")
    monkeypatch.setattr(pa, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        pa.load()


PAGE_TAGS = ("[BM]", "[KB]", "[BUG]", "[PG]")


def declaration_comments():
    """For each function the header declares, the comment block nearest above
    its declaration (declarations that follow one another without a comment
    of their own share the block above the first; comments that trail a line,
    such as those of enum members, do not count)."""
    text = open(HEADER).read()
    out, last = {}, ""
    for m in re.finditer(r"^/\*.*?\*/|^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.S | re.M):
        if m.group(0).startswith("/*"):
            last = " ".join(re.sub(r"\n\s*\*(?!/)", " ", m.group(0)).split())   # one line of words
        elif m.group(1) and m.group(1) != "defined":
            out[m.group(1)] = last
    return out


def test_every_declaration_cites_its_passage_or_says_it_has_none():
    """Each entry point names the passage of the pages that defines what it
    computes, or states that the pages have no counterpart for it."""
    comments = declaration_comments()
    assert set(comments) == set(declared_functions())
    for name, comment in comments.items():
        assert any(t in comment for t in PAGE_TAGS) or "no counterpart" in comment, name
    # the split-KV pair rests on the per-block aggregation of [PG] s2.2
    for name in ("paged_attention_partial_workspace", "paged_attention_decode_partial",
                 "paged_attention_decode_reduce"):
        assert "[PG] s2.2" in comments[name], name


def _layouts():
    """Every workload layout the tests and the benchmark use, with its int8
    and fp8 counterparts (the strides do not depend on the lengths, so short
    sequences keep the pools small)."""
    import workloads
    for index, bs in [(1, None), (2, None), (3, 8), (3, 16), (3, 32), (3, 64), (4, 16), (4, 256),
                      (5, None)]:
        w = workloads.make_workload(index, block_size=bs, batch=4 if index in (2, 3, 4) else None,
                                    max_len=64)
        yield f"workload {index} bs {w.bs}", w
        if w.D in (64, 128, 256):
            yield f"workload {index} bs {w.bs} int8", workloads.to_int8(w)
            yield f"workload {index} bs {w.bs} fp8", workloads.to_fp8(w)


def test_workload_blocks_start_on_128_byte_boundaries():
    """"KV Block design" s3.7 wants every block to start on a 128-byte
    boundary.  With a pool base on a 128-byte boundary (the caching allocator
    of the GPU hands out 512-byte aligned blocks; test_gpu_edges checks the
    device pools), that holds for every block, both halves and every kv head
    when the block stride, the K-to-V offset and the (block, kv head) chunk
    are multiples of 128 bytes."""
    for what, w in _layouts():
        es = w.pool.element_size()
        assert w.pool.is_contiguous(), what
        assert (w.block_stride * es) % 128 == 0, what
        assert (w.v_offset * es) % 128 == 0, what
        assert (w.bs * w.D * es) % 128 == 0, what
        # the chunk start of every (block, K|V, kv head) relative to the base
        starts = [(blk * w.block_stride + half * w.v_offset + hk * w.bs * w.D) * es
                  for blk in (0, 1, w.NB - 1) for half in (0, 1) for hk in range(w.Hkv)]
        assert all(s % 128 == 0 for s in starts), what


def test_kernel_query_rejects_bad_arguments(lib):
    """paged_attention_decode_kernel validates like the launches it
    describes (no device is needed for a rejection)."""
    s = base_shape()
    assert pa.paged_attention_decode_kernel(base_shape(num_heads=7)) == pa.PA_KERNEL_INVALID
    assert pa.paged_attention_decode_kernel(s, -1, 0) == pa.PA_KERNEL_INVALID       # window
    assert pa.paged_attention_decode_kernel(s, 0, 24) == pa.PA_KERNEL_INVALID       # partition size
    assert pa.paged_attention_decode_kernel(s, 0, -16) == pa.PA_KERNEL_INVALID
    # a CUDA-core shape never reaches a tensor-core kernel
    assert pa.paged_attention_decode_kernel(base_shape(dtype=pa.PA_F32)) == pa.PA_KERNEL_SIMT
