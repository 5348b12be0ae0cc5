"""CPU oracle for the paged-KV hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product (the CUDA library and its Python binding) never imports, links or
calls it, and shares none of its code.

Numeric routines live in ``pa_oracle.c`` (plain C, double precision); the
block bookkeeping lives in ``blocks.py``.  The wrappers below take numpy
arrays (host memory) and return numpy arrays.  Element types: "f32",
"bf16", "f16"; 16-bit buffers are passed as raw uint16 bit patterns.

Pinned functions (see tests/test_oracle_pins.py): slot translation, write,
block copy, block swap, gather, attention, the FP8 E4M3 codes, the quantizing
write and attention over a quantized cache, and the block bookkeeping.  None
is unpinned.
"""
import ctypes
import os

import numpy as np

from . import blocks  # noqa: F401  (re-exported)
from .build import build as _build

DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
ELT = {"f32": 4, "bf16": 2, "f16": 2}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build()
        L = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        L.oracle_slot_mapping.argtypes = [vp, i32, vp, vp, i64, i32, vp]
        L.oracle_slot_mapping.restype = None
        L.oracle_write_kv.argtypes = [vp, vp, vp, i64, vp, vp, i64]
        L.oracle_write_kv.restype = None
        L.oracle_copy_blocks.argtypes = [vp, vp, i32, vp, i32, i64]
        L.oracle_copy_blocks.restype = None
        L.oracle_swap_blocks.argtypes = [vp, vp, vp, vp, i32, vp, i32, i64]
        L.oracle_swap_blocks.restype = None
        L.oracle_gather.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.c_int, vp]
        L.oracle_gather.restype = None
        L.oracle_paged_attention.argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32,
                                             ctypes.c_float, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int]
        L.oracle_paged_attention.restype = None
        L.oracle_decode.argtypes = [vp, i64, ctypes.c_int, vp]
        L.oracle_decode.restype = None
        L.oracle_e4m3_encode_array.argtypes = [vp, i64, vp]
        L.oracle_e4m3_encode_array.restype = None
        L.oracle_e4m3_decode_array.argtypes = [vp, i64, vp]
        L.oracle_e4m3_decode_array.restype = None
        L.oracle_quant_rows.argtypes = [vp, ctypes.c_int, i64, i32, vp, vp]
        L.oracle_quant_rows.restype = None
        L.oracle_write_kv_fp8.argtypes = [vp, vp, ctypes.c_int, vp, i64, i32, i32, i32, vp, vp, vp, vp]
        L.oracle_write_kv_fp8.restype = None
        L.oracle_paged_attention_fp8.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32,
                                                 i32, i32, i32, ctypes.c_float, ctypes.c_int, ctypes.c_int]
        L.oracle_paged_attention_fp8.restype = None
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _c(a, dtype=None):
    a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype=dtype))
    return a


def max_threads() -> int:
    return lib().oracle_max_threads()


def decode(raw, dtype: str) -> np.ndarray:
    """Raw element buffer (float32 array or uint16 bit patterns) -> float64."""
    raw = _c(raw)
    out = np.empty(raw.shape, dtype=np.float64)
    lib().oracle_decode(_ptr(raw), raw.size, DTYPES[dtype], _ptr(out))
    return out


def slot_mapping(block_tables, seq_idx, positions, block_size: int) -> np.ndarray:
    bt = _c(block_tables, np.int32)
    si = _c(seq_idx, np.int32)
    pos = _c(positions, np.int64)
    out = np.empty(pos.shape[0], dtype=np.int64)
    lib().oracle_slot_mapping(_ptr(bt), bt.shape[1], _ptr(si), _ptr(pos), pos.shape[0], block_size, _ptr(out))
    return out


def write_kv(k, v, slot_mapping_, k_cache, v_cache) -> None:
    """In-place row scatter into numpy caches [NB, bs, Hkv, hd] (any element type)."""
    k, v = _c(k), _c(v)
    sm = _c(slot_mapping_, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    row_bytes = k.nbytes // max(k.shape[0], 1) if k.shape[0] else 0
    lib().oracle_write_kv(_ptr(k), _ptr(v), _ptr(sm), sm.shape[0], _ptr(k_cache), _ptr(v_cache), row_bytes)


def copy_blocks(k_caches, v_caches, block_pairs) -> None:
    """In-place whole-block copies over every layer's numpy caches."""
    pairs = _c(block_pairs, np.int64).reshape(-1, 2)
    n = len(k_caches)
    for c in list(k_caches) + list(v_caches):
        assert c.flags.c_contiguous
    block_bytes = k_caches[0].nbytes // k_caches[0].shape[0]
    kp = (ctypes.c_void_p * n)(*[c.ctypes.data for c in k_caches])
    vp = (ctypes.c_void_p * n)(*[c.ctypes.data for c in v_caches])
    lib().oracle_copy_blocks(kp, vp, n, _ptr(pairs), pairs.shape[0], block_bytes)


def swap_blocks(src_k, src_v, dst_k, dst_v, block_pairs) -> None:
    """In-place: dst pools' blocks receive the src pools' blocks, every layer."""
    pairs = _c(block_pairs, np.int64).reshape(-1, 2)
    n = len(src_k)
    for c in list(src_k) + list(src_v) + list(dst_k) + list(dst_v):
        assert c.flags.c_contiguous
    block_bytes = src_k[0].nbytes // src_k[0].shape[0]
    arr = lambda cs: (ctypes.c_void_p * n)(*[c.ctypes.data for c in cs])  # noqa: E731
    lib().oracle_swap_blocks(arr(src_k), arr(src_v), arr(dst_k), arr(dst_v), n, _ptr(pairs), pairs.shape[0],
                             block_bytes)


def gather(cache, block_table, seq_len: int, dtype: str) -> np.ndarray:
    """First seq_len tokens of one sequence, [seq_len, Hkv, hd] float64."""
    cache = _c(cache)
    nb, bs, hkv, hd = cache.shape
    bt = _c(block_table, np.int32)
    out = np.empty((seq_len, hkv, hd), dtype=np.float64)
    lib().oracle_gather(_ptr(cache), _ptr(bt), seq_len, bs, hkv, hd, DTYPES[dtype], _ptr(out))
    return out


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale: float,
                    dtype: str, causal: bool = True, seq_select=None, num_threads: int = 0) -> np.ndarray:
    """Varlen paged causal attention, float64 output [total_q, Hq, hd]."""
    q = _c(q)
    kc, vc = _c(k_cache), _c(v_cache)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    total_q, hq, hd = q.shape
    nb, bs, hkv, hd2 = kc.shape
    assert hd2 == hd and hq % hkv == 0
    sel = None if seq_select is None else _c(seq_select, np.uint8)
    out = np.full((total_q, hq, hd), np.nan, dtype=np.float64)
    lib().oracle_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl),
                                 _ptr(qsl), sl.shape[0], hq, hkv, hd, bs, ctypes.c_float(scale),
                                 1 if causal else 0, DTYPES[dtype], _ptr(sel), num_threads)
    return out


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: str,
                     seq_select=None, num_threads: int = 0) -> np.ndarray:
    """One query per sequence: the num_new = 1 case of paged_attention."""
    s = np.asarray(context_lens).shape[0]
    qsl = np.arange(s + 1, dtype=np.int32)
    return paged_attention(q, k_cache, v_cache, block_tables, context_lens, qsl, scale, dtype, True,
                           seq_select, num_threads)


# ---- quantized (FP8 E4M3) cache --------------------------------------------

def e4m3_encode(x) -> np.ndarray:
    """float32 values -> E4M3 codes (nearest, ties to even, held at +-448)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def quant_rows(x, dtype: str):
    """Rows [..., row_len] (raw element buffer) -> (codes uint8 same shape, scales float32 [...])."""
    x = _c(x)
    row_len = x.shape[-1]
    n = x.size // row_len
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    lib().oracle_quant_rows(_ptr(x), DTYPES[dtype], n, row_len, _ptr(codes), _ptr(scales))
    return codes, scales


def write_kv_fp8(k, v, dtype: str, slot_mapping_, k_codes, v_codes, k_scales, v_scales) -> None:
    """In place: k, v [n, Hkv, hd] (raw, `dtype`) quantized into codes [NB, bs, Hkv, hd] and
    scales [NB, Hkv, bs] at the slots (negative slots skipped)."""
    k, v = _c(k), _c(v)
    sm = _c(slot_mapping_, np.int64)
    for a in (k_codes, v_codes, k_scales, v_scales):
        assert a.flags.c_contiguous
    n, hkv, hd = k.shape
    nb, bs = k_codes.shape[:2]
    assert k_codes.shape == (nb, bs, hkv, hd) and k_scales.shape == (nb, hkv, bs)
    lib().oracle_write_kv_fp8(_ptr(k), _ptr(v), DTYPES[dtype], _ptr(sm), sm.shape[0], hkv, hd, bs, _ptr(k_codes),
                              _ptr(v_codes), _ptr(k_scales), _ptr(v_scales))


def paged_attention_fp8(q, q_dtype: str, k_codes, v_codes, k_scales, v_scales, block_tables, seq_lens,
                        query_start_loc, scale: float, causal: bool = True, num_threads: int = 0) -> np.ndarray:
    """Varlen paged attention over a quantized cache, float64 [total_q, Hq, hd]."""
    q = _c(q)
    kc, vc = _c(k_codes, np.uint8), _c(v_codes, np.uint8)
    ks, vs = _c(k_scales, np.float32), _c(v_scales, np.float32)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    qsl = _c(query_start_loc, np.int32)
    total_q, hq, hd = q.shape
    nb, bs, hkv, hd2 = kc.shape
    assert hd2 == hd and hq % hkv == 0 and ks.shape == (nb, hkv, bs) and vs.shape == ks.shape
    out = np.full((total_q, hq, hd), np.nan, dtype=np.float64)
    lib().oracle_paged_attention_fp8(_ptr(out), _ptr(q), DTYPES[q_dtype], _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                     _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl), sl.shape[0], hq, hkv, hd, bs,
                                     ctypes.c_float(scale), 1 if causal else 0, num_threads)
    return out
