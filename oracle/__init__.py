"""CPU oracle for decode attention over a block-paged KV cache (fp64).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA path: the arithmetic lives in ``pa_oracle.c``
(plain C, double precision), compiled here with gcc; this module only
marshals numpy/torch CPU arrays into it.

Every function states the passage of the source pages it follows:

* "KV Cache and BlockManager" (dpshk.com/news/5906718), abbreviated [BM]
* vLLM memory-management course, ch. 3 "KV Block design", abbreviated [KB]
* "A strange KV Cache bug" (dpshk.com/news/5937191), abbreviated [BUG]
* "KV Cache paging in LLM inference" (intelliparadigm.com), abbreviated [PG]

Parity is pinned for every function (tests/test_oracle.py); none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pa_oracle.c"
_LIBDIR = _HERE / "_lib"
_LIB = _LIBDIR / "libpa_oracle.so"

F32, F16, BF16 = 0, 1, 2
SEQ_BAD_LEN, SEQ_BAD_BLOCK, SEQ_BAD_POS = 1, 2, 4

_lock = threading.Lock()
_handle = None


def build(force: bool = False) -> Path:
    """Compile pa_oracle.c into oracle/_lib/libpa_oracle.so (gcc, OpenMP)."""
    _LIBDIR.mkdir(exist_ok=True)
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIBDIR / f".libpa_oracle.{os.getpid()}.so"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
             "-o", str(tmp), str(_SRC), "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            build()
            lib = ctypes.CDLL(str(_LIB))
            i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.pao_blocks_needed.restype = i64
            lib.pao_blocks_needed.argtypes = [i64, i64]
            lib.pao_kv_bytes.restype = i64
            lib.pao_kv_bytes.argtypes = [i64, i64, i64, i64, i64]
            lib.pao_convert.restype = None
            lib.pao_convert.argtypes = [vp, i64, i32, vp]
            lib.pao_gather.restype = None
            lib.pao_gather.argtypes = [i32, i32, i32, i64, i32, vp, vp, vp, i32, i64, vp, vp]
            lib.pao_attention_contiguous.restype = None
            lib.pao_attention_contiguous.argtypes = [i64, i32, vp, vp, vp, dbl, vp]
            lib.pao_attention_decode.restype = i32
            lib.pao_attention_decode.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                 vp, vp, vp, vp, vp, dbl, vp, vp, i32]
            lib.pao_attention_partial.restype = i32
            lib.pao_attention_partial.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                  vp, vp, vp, vp, vp, dbl, i64, i64,
                                                  vp, vp, vp, vp, i32]
            lib.pao_merge_partials.restype = None
            lib.pao_merge_partials.argtypes = [i32, i32, vp, vp, vp, vp]
            lib.pao_kv_append_tokens.restype = i32
            lib.pao_kv_append_tokens.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                 vp, vp, vp, vp, vp, vp, vp, vp]
            lib.pao_attention_decode_window.restype = i32
            lib.pao_attention_decode_window.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                        vp, vp, vp, vp, vp, dbl, i64, vp, vp, i32]
            lib.pao_quantize_i8.restype = ctypes.c_byte
            lib.pao_quantize_i8.argtypes = [ctypes.c_float, ctypes.c_float]
            lib.pao_quantize_i8_array.restype = None
            lib.pao_quantize_i8_array.argtypes = [vp, i64, ctypes.c_float, vp]
            lib.pao_kv_append_i8.restype = i32
            lib.pao_kv_append_i8.argtypes = [i32, i32, i32, i32, i32, i64, i64, i32,
                                             vp, vp, vp, vp, vp, vp, vp, vp]
            lib.pao_gather_i8.restype = None
            lib.pao_gather_i8.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp, i32, i64, vp, vp]
            lib.pao_attention_decode_i8.restype = i32
            lib.pao_attention_decode_i8.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                    vp, vp, vp, vp, vp, vp, dbl, vp, vp, i32]
            lib.pao_kv_append.restype = i32
            lib.pao_kv_append.argtypes = [i32, i32, i32, i32, i32, i64, i64, i32,
                                          vp, vp, vp, vp, vp, vp, vp]
            lib.pao_e4m3_value.restype = dbl
            lib.pao_e4m3_value.argtypes = [ctypes.c_ubyte]
            lib.pao_e4m3_encode.restype = ctypes.c_ubyte
            lib.pao_e4m3_encode.argtypes = [ctypes.c_float]
            lib.pao_quantize_fp8.restype = ctypes.c_ubyte
            lib.pao_quantize_fp8.argtypes = [ctypes.c_float, ctypes.c_float]
            lib.pao_quantize_fp8_array.restype = None
            lib.pao_quantize_fp8_array.argtypes = [vp, i64, ctypes.c_float, vp]
            lib.pao_kv_append_fp8.restype = i32
            lib.pao_kv_append_fp8.argtypes = [i32, i32, i32, i32, i32, i64, i64, i32,
                                              vp, vp, vp, vp, vp, vp, vp, vp]
            lib.pao_gather_fp8.restype = None
            lib.pao_gather_fp8.argtypes = [i32, i32, i32, i64, vp, vp, vp, vp, i32, i64, vp, vp]
            lib.pao_attention_decode_fp8.restype = i32
            lib.pao_attention_decode_fp8.argtypes = [i32, i32, i32, i32, i32, i32, i64, i64, i32,
                                                     vp, vp, vp, vp, vp, vp, dbl, vp, vp, i32]
            _handle = lib
    return _handle


# ---------------------------------------------------------------------------
# marshalling helpers: accept numpy arrays or torch CPU tensors
# ---------------------------------------------------------------------------

def _dtype_code(x) -> int:
    name = str(getattr(x, "dtype", ""))
    if name in ("float32", "torch.float32"):
        return F32
    if name in ("float16", "torch.float16"):
        return F16
    if name in ("torch.bfloat16", "bfloat16"):
        return BF16
    raise TypeError(f"oracle: unsupported element type {name}")


def _ptr(x) -> int:
    """Address of a C-contiguous CPU buffer (numpy array or torch tensor)."""
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle: array must be C-contiguous")
        return x.ctypes.data
    if getattr(x, "is_cuda", False):
        raise ValueError("oracle: inputs must live in host memory")
    if not x.is_contiguous():
        raise ValueError("oracle: tensor must be contiguous")
    return x.data_ptr()


def _f32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


# ---------------------------------------------------------------------------
# public oracle functions
# ---------------------------------------------------------------------------

def blocks_needed(length: int, block_size: int) -> int:
    """Blocks a sequence of `length` tokens occupies ([BM] s2 example)."""
    return int(_lib().pao_blocks_needed(int(length), int(block_size)))


def kv_bytes(seqs: int, heads: int, tokens_per_seq: int, head_dim: int, dtype_bytes: int) -> int:
    """KV-cache bytes per layer, the [BM] s1 formula (heads = KV heads)."""
    return int(_lib().pao_kv_bytes(seqs, heads, tokens_per_seq, head_dim, dtype_bytes))


def to_double(x) -> np.ndarray:
    """Decode f32/f16/bf16 elements to float64 with the oracle's own decoder."""
    n = int(np.prod(x.shape)) if len(x.shape) else 1
    out = np.empty(n, dtype=np.float64)
    _lib().pao_convert(_ptr(x), n, _dtype_code(x), out.ctypes.data)
    return out.reshape(tuple(x.shape))


def gather(k_pool, v_pool, table_row, kv_head: int, length: int, *, block_size: int,
           head_dim: int, num_kv_heads: int, block_stride: int):
    """Contiguous [length][head_dim] K and V of one kv head ([BM] s2, [KB] s3.3)."""
    row = _i32(table_row)
    Kc = np.empty((max(length, 1), head_dim), dtype=np.float64)
    Vc = np.empty_like(Kc)
    _lib().pao_gather(head_dim, block_size, num_kv_heads, block_stride, _dtype_code(k_pool),
                      _ptr(k_pool), _ptr(v_pool), row.ctypes.data, kv_head, length,
                      Kc.ctypes.data, Vc.ctypes.data)
    return Kc[:length], Vc[:length]


def attention_contiguous(q, Kc, Vc, scale: float) -> np.ndarray:
    """Textbook softmax attention of one query over contiguous K/V ([BUG] s4.1-4.2)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    Kc = np.ascontiguousarray(Kc, dtype=np.float64)
    Vc = np.ascontiguousarray(Vc, dtype=np.float64)
    L, D = Kc.shape
    o = np.empty(D, dtype=np.float64)
    _lib().pao_attention_contiguous(L, D, q.ctypes.data, Kc.ctypes.data, Vc.ctypes.data,
                                    float(scale), o.ctypes.data)
    return o


def attention_decode(q, k_pool, v_pool, block_table, seq_lens, scale: float, *,
                     num_kv_heads: int, block_size: int, block_stride: int,
                     num_blocks: int, threads: int = 0):
    """Decode attention over the paged cache, masked to seq_lens.

    q: [B][H][D] (f32/f16/bf16, host); pools: flat host buffers of the same
    dtype addressed as blk*block_stride + kv_head*block_size*D + slot*D + d;
    block_table: int32 [B][MB]; seq_lens: int32 [B] (valid lengths).
    Returns (out float64 [B][H][D], seq_err int32 [B]).
    """
    B, H, D = (int(s) for s in q.shape)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    MB = bt.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_attention_decode(B, H, num_kv_heads, D, block_size, MB, num_blocks, block_stride,
                                _dtype_code(q), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                bt.ctypes.data, sl.ctypes.data, float(scale),
                                out.ctypes.data, err.ctypes.data, int(threads))
    return out, err


def attention_partial(q, k_pool, v_pool, block_table, seq_lens, scale: float,
                      t_begin: int, t_end: int, *, num_kv_heads: int, block_size: int,
                      block_stride: int, num_blocks: int, threads: int = 0):
    """Partial softmax sums (m, l, acc) over tokens [t_begin, t_end) ([PG] s2.2)."""
    B, H, D = (int(s) for s in q.shape)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    MB = bt.shape[1]
    m = np.empty((B, H), dtype=np.float64)
    l = np.empty((B, H), dtype=np.float64)
    acc = np.empty((B, H, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_attention_partial(B, H, num_kv_heads, D, block_size, MB, num_blocks, block_stride,
                                 _dtype_code(q), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                 bt.ctypes.data, sl.ctypes.data, float(scale),
                                 int(t_begin), int(t_end), m.ctypes.data, l.ctypes.data,
                                 acc.ctypes.data, err.ctypes.data, int(threads))
    return m, l, acc, err


def merge_partials(m, l, acc) -> np.ndarray:
    """Log-sum-exp merge of partial results of one (b, h)."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    n, D = acc.shape
    o = np.empty(D, dtype=np.float64)
    _lib().pao_merge_partials(n, D, m.ctypes.data, l.ctypes.data, acc.ctypes.data, o.ctypes.data)
    return o


def kv_append(k_new, v_new, k_pool, v_pool, block_table, positions, *, block_size: int,
              block_stride: int, num_blocks: int):
    """Append one token's K/V row per (sequence, kv head), in place ([BM] s4.4).

    k_new, v_new: [B][Hkv][D]; the pools are modified in place (pass copies).
    Returns seq_err int32 [B].
    """
    B, Hkv, D = (int(s) for s in k_new.shape)
    bt = _i32(block_table)
    pos = _i32(positions)
    MB = bt.shape[1]
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_kv_append(B, Hkv, D, block_size, MB, num_blocks, block_stride, _dtype_code(k_new),
                         _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                         bt.ctypes.data, pos.ctypes.data, err.ctypes.data)
    return err


def kv_append_tokens(k_new, v_new, k_pool, v_pool, block_table, positions, counts, *,
                     block_size: int, block_stride: int, num_blocks: int):
    """Prefill write of counts[b] tokens per sequence from a padded batch
    k_new/v_new [B][T][Hkv][D], in place ([BUG] s2.3-2.4, s4.1)."""
    B, T, Hkv, D = (int(s) for s in k_new.shape)
    bt = _i32(block_table)
    pos = _i32(positions)
    cnt = _i32(counts)
    MB = bt.shape[1]
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_kv_append_tokens(B, T, Hkv, D, block_size, MB, num_blocks, block_stride,
                                _dtype_code(k_new), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                                _ptr(v_pool), bt.ctypes.data, pos.ctypes.data, cnt.ctypes.data,
                                err.ctypes.data)
    return err


def attention_decode_window(q, k_pool, v_pool, block_table, seq_lens, scale: float, window: int,
                            *, num_kv_heads: int, block_size: int, block_stride: int,
                            num_blocks: int, threads: int = 0):
    """Decode attention over the last `window` valid tokens ([BUG] s5.3)."""
    B, H, D = (int(s) for s in q.shape)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    MB = bt.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_attention_decode_window(B, H, num_kv_heads, D, block_size, MB, num_blocks,
                                       block_stride, _dtype_code(q), _ptr(q), _ptr(k_pool),
                                       _ptr(v_pool), bt.ctypes.data, sl.ctypes.data,
                                       float(scale), int(window), out.ctypes.data,
                                       err.ctypes.data, int(threads))
    return out, err


# ---------------------------------------------------------------------------
# int8 cache blocks with per-(block, kv head) scales
# ---------------------------------------------------------------------------
# The pages name int8-quantised cache blocks ("KV Cache and BlockManager"
# s6.3; the "quantized" element size of its s3 block-size rule) without a
# scheme.  The reading implemented in pa_oracle.c: a code c in [-127, 127]
# stands for c * s, with one fp32 scale s per (physical block, kv head) for K
# and one for V, kv_scales[(blk*2 + 0)*Hkv + hk] and [(blk*2 + 1)*Hkv + hk];
# writing x stores clamp(round_half_even(x / s), -127, 127), decided in IEEE
# binary32 (a NaN quotient stores 0).

def quantize_i8(x, scale: float) -> np.ndarray:
    """int8 codes of the float32 values x under one scale (binary32 x / s,
    ties to even, clamped to [-127, 127])."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xs.shape, dtype=np.int8)
    _lib().pao_quantize_i8_array(xs.ctypes.data, xs.size, float(np.float32(scale)), out.ctypes.data)
    return out


def kv_append_i8(k_new, v_new, k_pool, v_pool, kv_scales, block_table, positions, *,
                 block_size: int, block_stride: int, num_blocks: int):
    """Append one token per (sequence, kv head) into int8 pools, quantising
    with the scales of the target block (in place; returns seq_err)."""
    B, Hkv, D = (int(s) for s in k_new.shape)
    bt = _i32(block_table)
    pos = _i32(positions)
    sc = _f32(kv_scales)
    MB = bt.shape[1]
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_kv_append_i8(B, Hkv, D, block_size, MB, num_blocks, block_stride,
                            _dtype_code(k_new), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                            _ptr(v_pool), sc.ctypes.data, bt.ctypes.data, pos.ctypes.data,
                            err.ctypes.data)
    return err


def gather_i8(k_pool, v_pool, kv_scales, table_row, kv_head: int, length: int, *,
              block_size: int, head_dim: int, num_kv_heads: int, block_stride: int):
    """Contiguous [length][head_dim] dequantised K and V of one kv head."""
    row = _i32(table_row)
    sc = _f32(kv_scales)
    Kc = np.empty((max(length, 1), head_dim), dtype=np.float64)
    Vc = np.empty_like(Kc)
    _lib().pao_gather_i8(head_dim, block_size, num_kv_heads, block_stride, _ptr(k_pool),
                         _ptr(v_pool), sc.ctypes.data, row.ctypes.data, kv_head, length,
                         Kc.ctypes.data, Vc.ctypes.data)
    return Kc[:length], Vc[:length]


def attention_decode_i8(q, k_pool, v_pool, kv_scales, block_table, seq_lens, scale: float, *,
                        num_kv_heads: int, block_size: int, block_stride: int,
                        num_blocks: int, threads: int = 0):
    """Decode attention over an int8 cache (the values the codes stand for),
    masked to seq_lens.  Returns (out float64 [B][H][D], seq_err int32 [B])."""
    B, H, D = (int(s) for s in q.shape)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    sc = _f32(kv_scales)
    MB = bt.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_attention_decode_i8(B, H, num_kv_heads, D, block_size, MB, num_blocks,
                                   block_stride, _dtype_code(q), _ptr(q), _ptr(k_pool),
                                   _ptr(v_pool), sc.ctypes.data, bt.ctypes.data, sl.ctypes.data,
                                   float(scale), out.ctypes.data, err.ctypes.data, int(threads))
    return out, err


# ---------------------------------------------------------------------------
# fp8 (E4M3) cache blocks with per-(block, kv head) scales
# ---------------------------------------------------------------------------
# The second reading of quantised blocks implemented in pa_oracle.c: a code
# is an OCP FP8 E4M3 byte (bias 7, 3 mantissa bits, subnormals m * 2^-9, no
# infinities, 0x7F / 0xFF NaN, largest finite 448) standing for value(c) * s,
# scales laid out as for int8; writing x stores the code of the binary32
# quotient x / s, nearest value, ties to the even code, magnitudes beyond 448
# saturating to 448 (a NaN quotient stores 0x7F).

def e4m3_value(code: int) -> float:
    """The value an E4M3 code stands for."""
    return float(_lib().pao_e4m3_value(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """The E4M3 code of a binary32 value (nearest, ties to even, saturating)."""
    return int(_lib().pao_e4m3_encode(float(np.float32(x))))


def quantize_fp8(x, scale: float) -> np.ndarray:
    """E4M3 codes (uint8) of the float32 values x under one scale."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xs.shape, dtype=np.uint8)
    _lib().pao_quantize_fp8_array(xs.ctypes.data, xs.size, float(np.float32(scale)), out.ctypes.data)
    return out


def kv_append_fp8(k_new, v_new, k_pool, v_pool, kv_scales, block_table, positions, *,
                  block_size: int, block_stride: int, num_blocks: int):
    """Append one token per (sequence, kv head) into fp8 pools, quantising
    with the scales of the target block (in place; returns seq_err)."""
    B, Hkv, D = (int(s) for s in k_new.shape)
    bt = _i32(block_table)
    pos = _i32(positions)
    sc = _f32(kv_scales)
    MB = bt.shape[1]
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_kv_append_fp8(B, Hkv, D, block_size, MB, num_blocks, block_stride,
                             _dtype_code(k_new), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                             _ptr(v_pool), sc.ctypes.data, bt.ctypes.data, pos.ctypes.data,
                             err.ctypes.data)
    return err


def gather_fp8(k_pool, v_pool, kv_scales, table_row, kv_head: int, length: int, *,
               block_size: int, head_dim: int, num_kv_heads: int, block_stride: int):
    """Contiguous [length][head_dim] dequantised K and V of one kv head."""
    row = _i32(table_row)
    sc = _f32(kv_scales)
    Kc = np.empty((max(length, 1), head_dim), dtype=np.float64)
    Vc = np.empty_like(Kc)
    _lib().pao_gather_fp8(head_dim, block_size, num_kv_heads, block_stride, _ptr(k_pool),
                          _ptr(v_pool), sc.ctypes.data, row.ctypes.data, kv_head, length,
                          Kc.ctypes.data, Vc.ctypes.data)
    return Kc[:length], Vc[:length]


def attention_decode_fp8(q, k_pool, v_pool, kv_scales, block_table, seq_lens, scale: float, *,
                         num_kv_heads: int, block_size: int, block_stride: int,
                         num_blocks: int, threads: int = 0):
    """Decode attention over an fp8 cache (the values the codes stand for),
    masked to seq_lens.  Returns (out float64 [B][H][D], seq_err int32 [B])."""
    B, H, D = (int(s) for s in q.shape)
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    sc = _f32(kv_scales)
    MB = bt.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    err = np.zeros(B, dtype=np.int32)
    _lib().pao_attention_decode_fp8(B, H, num_kv_heads, D, block_size, MB, num_blocks,
                                    block_stride, _dtype_code(q), _ptr(q), _ptr(k_pool),
                                    _ptr(v_pool), sc.ctypes.data, bt.ctypes.data, sl.ctypes.data,
                                    float(scale), out.ctypes.data, err.ctypes.data, int(threads))
    return out, err
