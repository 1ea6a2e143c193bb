"""Python binding of libpagedattn.so (include/pagedattn.h), via ctypes.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of the library.  Tensors are torch CUDA tensors; their data pointers
and torch's current CUDA stream are handed to the C ABI unchanged.  If the
library has not been built, importing works but every call raises -- there is
no CPU fallback.

Names follow the C ABI: paged_kv_append, paged_attention_decode,
paged_attention_decode_append (both in one launch), paged_kv_append_tokens
(prefill write), paged_attention_decode_window (sliding window),
paged_attention_partial_workspace, paged_attention_decode_partial,
paged_attention_decode_reduce, paged_attention_decode_path,
paged_attention_decode_kernel (which kernel runs a shape on this device),
paged_attention_balanced_workspace, paged_attention_decode_balanced
(persistent load-balanced schedule), paged_kv_append_int8,
paged_attention_decode_int8 (int8 cache with per-block scales),
paged_kv_append_fp8, paged_attention_decode_fp8 (fp8 E4M3 cache with
per-block scales).
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import torch

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_lib" / "libpagedattn.so"

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_MISALIGNED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(6)
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
PA_PATH_INVALID, PA_PATH_SIMT, PA_PATH_TENSOR_GQA = 0, 1, 2
PA_KERNEL_INVALID, PA_KERNEL_SIMT, PA_KERNEL_MMA_SYNC, PA_KERNEL_TCGEN05 = 0, 1, 2, 3
DEVERR_BAD_LEN, DEVERR_BAD_BLOCK, DEVERR_BAD_POS, DEVERR_TIMEOUT, DEVERR_BAD_PREFIX = 1, 2, 4, 8, 16

EXPORTED = ("pa_status_string", "pa_version", "paged_kv_append", "paged_attention_decode",
            "paged_attention_decode_append", "paged_attention_decode_split_static",
            "paged_kv_append_tokens", "paged_attention_decode_window",
            "paged_attention_decode_path", "paged_attention_decode_kernel",
            "paged_attention_partial_workspace",
            "paged_attention_decode_partial", "paged_attention_decode_reduce",
            "paged_attention_balanced_workspace", "paged_attention_decode_balanced",
            "paged_kv_append_int8", "paged_attention_decode_int8",
            "paged_kv_append_fp8", "paged_attention_decode_fp8",
            "paged_attention_decode_shared_prefix", "paged_attention_decode_shared_prefix_int8",
            "paged_attention_decode_shared_prefix_fp8")


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class Shape(ctypes.Structure):
    """Mirror of pa_shape."""
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("block_stride", ctypes.c_int64),
                ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(str(LIB_PATH))
            vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
            sp = ctypes.POINTER(Shape)
            lib.pa_status_string.restype = ctypes.c_char_p
            lib.pa_status_string.argtypes = [ctypes.c_int]
            lib.pa_version.restype = i32
            lib.pa_version.argtypes = []
            lib.paged_kv_append.restype = ctypes.c_int
            lib.paged_kv_append.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.paged_attention_decode.restype = ctypes.c_int
            lib.paged_attention_decode.argtypes = [sp, vp, vp, vp, vp, vp, vp, f32, vp, vp]
            lib.paged_attention_decode_append.restype = ctypes.c_int
            lib.paged_attention_decode_append.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, f32,
                                                          vp, vp]
            lib.paged_kv_append_tokens.restype = ctypes.c_int
            lib.paged_kv_append_tokens.argtypes = [sp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp]
            lib.paged_attention_decode_window.restype = ctypes.c_int
            lib.paged_attention_decode_window.argtypes = [sp, vp, vp, vp, vp, vp, vp, f32, i32, vp,
                                                          vp]
            lib.paged_attention_decode_path.restype = ctypes.c_int
            lib.paged_attention_decode_path.argtypes = [sp]
            lib.paged_attention_decode_kernel.restype = ctypes.c_int
            lib.paged_attention_decode_kernel.argtypes = [sp, i32, i32]
            lib.paged_attention_partial_workspace.restype = sz
            lib.paged_attention_partial_workspace.argtypes = [sp, i32]
            lib.paged_attention_decode_partial.restype = ctypes.c_int
            lib.paged_attention_decode_partial.argtypes = [sp, vp, vp, vp, vp, vp, f32, i32, vp, sz,
                                                           vp, vp]
            lib.paged_attention_decode_reduce.restype = ctypes.c_int
            lib.paged_attention_decode_reduce.argtypes = [sp, vp, vp, sz, vp, i32, vp, vp]
            lib.paged_attention_decode_shared_prefix.restype = ctypes.c_int
            lib.paged_attention_decode_shared_prefix.argtypes = [sp, vp, vp, vp, vp, vp, vp, i32, vp, vp,
                                                                 f32, i32, vp, sz, vp, vp]
            for name in ("paged_attention_decode_shared_prefix_int8", "paged_attention_decode_shared_prefix_fp8"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, f32, i32, vp, sz, vp, vp]
            lib.paged_kv_append_int8.restype = ctypes.c_int
            lib.paged_kv_append_int8.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.paged_attention_decode_int8.restype = ctypes.c_int
            lib.paged_attention_decode_int8.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp]
            lib.paged_kv_append_fp8.restype = ctypes.c_int
            lib.paged_kv_append_fp8.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.paged_attention_decode_fp8.restype = ctypes.c_int
            lib.paged_attention_decode_fp8.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp]
            lib.paged_attention_balanced_workspace.restype = sz
            lib.paged_attention_balanced_workspace.argtypes = [sp]
            lib.paged_attention_decode_balanced.restype = ctypes.c_int
            lib.paged_attention_decode_balanced.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                            f32, i32, vp, sz, vp, vp]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def version() -> int:
    return int(load().pa_version())


def dtype_code(dtype: torch.dtype) -> int:
    try:
        return {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}[dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {dtype}") from None


def make_shape(*, batch, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
               num_blocks, block_stride, dtype) -> Shape:
    return Shape(int(batch), int(num_heads), int(num_kv_heads), int(head_dim), int(block_size),
                 int(max_blocks_per_seq), int(num_blocks), int(block_stride),
                 dtype if isinstance(dtype, int) else dtype_code(dtype))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, what)


class Prepared:
    """A C-ABI call with its arguments marshalled once.

    Calling it re-issues the same call (same buffers, shape, scale and
    stream), costing a few microseconds of host time instead of the full
    marshalling; the tensors it was built from must stay alive and keep their
    storage.  Every wrapper below returns one when given prepare=True.
    """

    __slots__ = ("_fn", "_args", "_what", "_keep")

    def __init__(self, fn, args, what, keep):
        self._fn, self._args, self._what, self._keep = fn, args, what, keep

    def __call__(self) -> None:
        status = self._fn(*self._args)
        if status != PA_OK:
            raise PagedAttnError(status, self._what)


def _issue(fn, args, what, prepare, keep=()):
    if prepare:
        return Prepared(fn, args, what, keep)
    _check(fn(*args), what)
    return None


def decode_shape(q, block_table, *, num_kv_heads, block_size, num_blocks, block_stride) -> Shape:
    B, H, D = q.shape
    return make_shape(batch=B, num_heads=H, num_kv_heads=num_kv_heads, head_dim=D,
                      block_size=block_size, max_blocks_per_seq=block_table.shape[1],
                      num_blocks=num_blocks, block_stride=block_stride, dtype=q.dtype)


def paged_kv_append(k_new, v_new, k_pool, v_pool, block_table, positions, *, block_size,
                    num_blocks, block_stride, err_word=None, stream=None, prepare=False):
    """Write k_new/v_new [B][Hkv][D] at positions[b] through block_table."""
    B, Hkv, D = k_new.shape
    shape = make_shape(batch=B, num_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=block_size,
                       max_blocks_per_seq=block_table.shape[1], num_blocks=num_blocks,
                       block_stride=block_stride, dtype=k_new.dtype)
    args = (
            ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
            _ptr(block_table), _ptr(positions), _ptr(err_word), _stream(stream))
    return _issue(load().paged_kv_append, args, "paged_kv_append", prepare,
                  (shape,))


def paged_attention_decode(out, q, k_pool, v_pool, block_table, seq_lens, scale, *, num_kv_heads,
                           block_size, num_blocks, block_stride, err_word=None,
                           stream=None, prepare=False):
    """out[B][H][D] = attention of q over the valid tokens of each sequence."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    args = (
            ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
            _ptr(block_table), _ptr(seq_lens), float(scale), _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode, args, "paged_attention_decode", prepare,
                  (shape,))


def paged_attention_decode_append(out, q, k_new, v_new, k_pool, v_pool, block_table, positions,
                                  scale, *, num_kv_heads, block_size, num_blocks, block_stride,
                                  err_word=None, stream=None, prepare=False):
    """Append k_new/v_new at positions[b], then attend over positions[b] + 1 tokens."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    args = (
            ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
            _ptr(v_pool), _ptr(block_table), _ptr(positions), float(scale), _ptr(err_word),
            _stream(stream))
    return _issue(load().paged_attention_decode_append, args, "paged_attention_decode_append", prepare,
                  (shape,))


def paged_kv_append_tokens(k_new, v_new, k_pool, v_pool, block_table, positions, counts, *,
                           block_size, num_blocks, block_stride, err_word=None,
                           stream=None, prepare=False):
    """Prefill write: counts[b] rows of the padded batch k_new/v_new [B][T][Hkv][D]
    go to positions[b] + t."""
    B, T, Hkv, D = k_new.shape
    shape = make_shape(batch=B, num_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=block_size,
                       max_blocks_per_seq=block_table.shape[1], num_blocks=num_blocks,
                       block_stride=block_stride, dtype=k_new.dtype)
    args = (
            ctypes.byref(shape), _ptr(k_new), _ptr(v_new), int(T), _ptr(k_pool), _ptr(v_pool),
            _ptr(block_table), _ptr(positions), _ptr(counts), _ptr(err_word), _stream(stream))
    return _issue(load().paged_kv_append_tokens, args, "paged_kv_append_tokens", prepare,
                  (shape,))


def paged_attention_decode_window(out, q, k_pool, v_pool, block_table, seq_lens, scale, window,
                                  *, num_kv_heads, block_size, num_blocks, block_stride,
                                  err_word=None, stream=None, prepare=False):
    """Decode attention over the last `window` valid tokens of each sequence."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    args = (
            ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
            _ptr(block_table), _ptr(seq_lens), float(scale), int(window), _ptr(err_word),
            _stream(stream))
    return _issue(load().paged_attention_decode_window, args, "paged_attention_decode_window", prepare,
                  (shape,))


def paged_attention_decode_path(shape: Shape) -> int:
    return int(load().paged_attention_decode_path(ctypes.byref(shape)))


def paged_attention_decode_kernel(shape: Shape, window: int = 0, partition_tokens: int = 0) -> int:
    """PA_KERNEL_* the decode of `shape` runs on the current device (single
    pass, sliding window, or the split-KV partial pass when partition_tokens
    is positive)."""
    return load().paged_attention_decode_kernel(ctypes.byref(shape), window, partition_tokens)


def paged_attention_partial_workspace(shape: Shape, partition_tokens: int) -> int:
    return int(load().paged_attention_partial_workspace(ctypes.byref(shape), int(partition_tokens)))


def paged_attention_decode_partial(q, k_pool, v_pool, block_table, seq_lens, scale,
                                   partition_tokens, workspace, *, num_kv_heads, block_size,
                                   num_blocks, block_stride, err_word=None, stream=None, prepare=False):
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    nbytes = workspace.numel() * workspace.element_size()
    args = (
            ctypes.byref(shape), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
            _ptr(seq_lens), float(scale), int(partition_tokens), _ptr(workspace), nbytes,
            _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode_partial, args, "paged_attention_decode_partial", prepare,
                  (shape,))


def paged_attention_decode_reduce(out, workspace, seq_lens, partition_tokens, *, num_kv_heads,
                                  block_size, num_blocks, block_stride, max_blocks_per_seq,
                                  err_word=None, stream=None, prepare=False):
    B, H, D = out.shape
    shape = make_shape(batch=B, num_heads=H, num_kv_heads=num_kv_heads, head_dim=D,
                       block_size=block_size, max_blocks_per_seq=max_blocks_per_seq,
                       num_blocks=num_blocks, block_stride=block_stride, dtype=out.dtype)
    nbytes = workspace.numel() * workspace.element_size()
    args = (
            ctypes.byref(shape), _ptr(out), _ptr(workspace), nbytes, _ptr(seq_lens),
            int(partition_tokens), _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode_reduce, args, "paged_attention_decode_reduce", prepare,
                  (shape,))


def workspace_for(q, block_table, partition_tokens, *, num_kv_heads, block_size, num_blocks,
                  block_stride) -> torch.Tensor:
    """Allocate (through torch) a workspace big enough for the split-KV pair."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    n = paged_attention_partial_workspace(shape, partition_tokens)
    if n == 0:
        raise PagedAttnError(PA_ERR_INVALID_ARG, "paged_attention_partial_workspace")
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=q.device)


def paged_attention_balanced_workspace(shape: Shape) -> int:
    return int(load().paged_attention_balanced_workspace(ctypes.byref(shape)))


def balanced_workspace_for(q, block_table, *, num_kv_heads, block_size, num_blocks,
                           block_stride) -> torch.Tensor:
    """Allocate (through torch) a zero-filled workspace for
    paged_attention_decode_balanced on q's device."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    with torch.cuda.device(q.device):
        n = paged_attention_balanced_workspace(shape)
    if n == 0:
        raise PagedAttnError(PA_ERR_UNSUPPORTED, "paged_attention_balanced_workspace")
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=q.device)


def paged_attention_decode_balanced(out, q, k_pool, v_pool, block_table, scale, workspace, *,
                                    seq_lens=None, positions=None, k_new=None, v_new=None,
                                    window=0, num_kv_heads, block_size, num_blocks, block_stride,
                                    err_word=None, stream=None, prepare=False):
    """One decode step on the load-balanced persistent grid: plain decode
    (seq_lens) or fused append + decode (positions, k_new, v_new), over the
    last `window` tokens when window > 0."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    nbytes = workspace.numel() * workspace.element_size()
    args = (
            ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
            _ptr(seq_lens), _ptr(positions), _ptr(k_new), _ptr(v_new), float(scale), int(window),
            _ptr(workspace), nbytes, _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode_balanced, args, "paged_attention_decode_balanced",
                  prepare, (shape,))


def paged_kv_append_int8(k_new, v_new, k_pool, v_pool, kv_scales, block_table, positions, *,
                         block_size, num_blocks, block_stride, err_word=None, stream=None,
                         prepare=False):
    """Quantising append of k_new/v_new [B][Hkv][D] into int8 pools (codes of
    the target block's scales)."""
    B, Hkv, D = k_new.shape
    shape = make_shape(batch=B, num_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=block_size,
                       max_blocks_per_seq=block_table.shape[1], num_blocks=num_blocks,
                       block_stride=block_stride, dtype=k_new.dtype)
    args = (ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
            _ptr(kv_scales), _ptr(block_table), _ptr(positions), _ptr(err_word), _stream(stream))
    return _issue(load().paged_kv_append_int8, args, "paged_kv_append_int8", prepare, (shape,))


def paged_attention_decode_int8(out, q, k_pool, v_pool, kv_scales, block_table, seq_lens, scale, *,
                                num_kv_heads, block_size, num_blocks, block_stride, err_word=None,
                                stream=None, prepare=False):
    """Decode attention over an int8 cache with per-(block, kv head) scales."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    args = (ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_scales),
            _ptr(block_table), _ptr(seq_lens), float(scale), _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode_int8, args, "paged_attention_decode_int8", prepare,
                  (shape,))


def paged_kv_append_fp8(k_new, v_new, k_pool, v_pool, kv_scales, block_table, positions, *,
                        block_size, num_blocks, block_stride, err_word=None, stream=None,
                        prepare=False):
    """Quantising append of k_new/v_new [B][Hkv][D] into fp8 (E4M3) pools
    (codes of the target block's scales)."""
    B, Hkv, D = k_new.shape
    shape = make_shape(batch=B, num_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=block_size,
                       max_blocks_per_seq=block_table.shape[1], num_blocks=num_blocks,
                       block_stride=block_stride, dtype=k_new.dtype)
    args = (ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
            _ptr(kv_scales), _ptr(block_table), _ptr(positions), _ptr(err_word), _stream(stream))
    return _issue(load().paged_kv_append_fp8, args, "paged_kv_append_fp8", prepare, (shape,))


def paged_attention_decode_fp8(out, q, k_pool, v_pool, kv_scales, block_table, seq_lens, scale, *,
                               num_kv_heads, block_size, num_blocks, block_stride, err_word=None,
                               stream=None, prepare=False):
    """Decode attention over an fp8 (E4M3) cache with per-(block, kv head)
    scales."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    args = (ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_scales),
            _ptr(block_table), _ptr(seq_lens), float(scale), _ptr(err_word), _stream(stream))
    return _issue(load().paged_attention_decode_fp8, args, "paged_attention_decode_fp8", prepare,
                  (shape,))


def paged_attention_decode_shared_prefix(out, q, k_pool, v_pool, block_table, seq_lens, scale,
                                         partition_tokens, workspace, *, group_first, shared_tokens,
                                         num_kv_heads, block_size, num_blocks, block_stride,
                                         err_word=None, stream=None, prepare=False):
    """Split-KV decode where each group of sequences [group_first[i],
    group_first[i+1]) shares the blocks of its first shared_tokens[i] tokens:
    those partitions are read once per group (host lists)."""
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    n = len(shared_tokens)
    first = (ctypes.c_int32 * (n + 1))(*[int(x) for x in group_first])
    shared = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in shared_tokens])
    nbytes = workspace.numel() * workspace.element_size()
    args = (ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
            _ptr(seq_lens), n, ctypes.cast(first, ctypes.c_void_p), ctypes.cast(shared, ctypes.c_void_p),
            float(scale), int(partition_tokens), _ptr(workspace), nbytes, _ptr(err_word),
            _stream(stream))
    return _issue(load().paged_attention_decode_shared_prefix, args,
                  "paged_attention_decode_shared_prefix", prepare, (shape, first, shared))


def _shared_prefix_codes(name, out, q, k_pool, v_pool, kv_scales, block_table, seq_lens, scale,
                         partition_tokens, workspace, group_first, shared_tokens, num_kv_heads,
                         block_size, num_blocks, block_stride, err_word, stream, prepare):
    shape = decode_shape(q, block_table, num_kv_heads=num_kv_heads, block_size=block_size,
                         num_blocks=num_blocks, block_stride=block_stride)
    n = len(shared_tokens)
    first = (ctypes.c_int32 * (n + 1))(*[int(x) for x in group_first])
    shared = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in shared_tokens])
    nbytes = workspace.numel() * workspace.element_size()
    args = (ctypes.byref(shape), _ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_scales),
            _ptr(block_table), _ptr(seq_lens), n, ctypes.cast(first, ctypes.c_void_p),
            ctypes.cast(shared, ctypes.c_void_p), float(scale), int(partition_tokens), _ptr(workspace),
            nbytes, _ptr(err_word), _stream(stream))
    return _issue(getattr(load(), name), args, name, prepare, (shape, first, shared))


def paged_attention_decode_shared_prefix_int8(out, q, k_pool, v_pool, kv_scales, block_table, seq_lens,
                                              scale, partition_tokens, workspace, *, group_first,
                                              shared_tokens, num_kv_heads, block_size, num_blocks,
                                              block_stride, err_word=None, stream=None, prepare=False):
    """paged_attention_decode_shared_prefix over an int8 cache with
    per-(block, kv head) scales (host group lists)."""
    return _shared_prefix_codes("paged_attention_decode_shared_prefix_int8", out, q, k_pool, v_pool,
                                kv_scales, block_table, seq_lens, scale, partition_tokens, workspace,
                                group_first, shared_tokens, num_kv_heads, block_size, num_blocks,
                                block_stride, err_word, stream, prepare)


def paged_attention_decode_shared_prefix_fp8(out, q, k_pool, v_pool, kv_scales, block_table, seq_lens,
                                             scale, partition_tokens, workspace, *, group_first,
                                             shared_tokens, num_kv_heads, block_size, num_blocks,
                                             block_stride, err_word=None, stream=None, prepare=False):
    """paged_attention_decode_shared_prefix over an fp8 (E4M3) cache with
    per-(block, kv head) scales (host group lists)."""
    return _shared_prefix_codes("paged_attention_decode_shared_prefix_fp8", out, q, k_pool, v_pool,
                                kv_scales, block_table, seq_lens, scale, partition_tokens, workspace,
                                group_first, shared_tokens, num_kv_heads, block_size, num_blocks,
                                block_stride, err_word, stream, prepare)
