"""ctypes binding of libpa.so: the C ABI's entry points under the same names.

Argument marshalling only -- torch tensors become device pointers, sizes and
the current CUDA stream; every step of the path runs in the library's CUDA
kernels.  There is no fallback: if the library is missing the first call
raises, and every non-OK status raises PAError with the library's reason.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpa.so")

PA_F32, PA_BF16, PA_F16, PA_FP8_E4M3 = 0, 1, 2, 3
PA_OPT_CHECK_MODE, PA_OPT_DECODE_KERNEL, PA_OPT_DECODE_CTAS, PA_OPT_VARLEN_KERNEL, PA_OPT_FP8_PAIR_STEP = 0, 1, 2, 3, 4
DTYPE_CODE = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16}
# pools that only move bytes (copy, swap) may also hold E4M3 codes
POOL_DTYPE_CODE = {**DTYPE_CODE, torch.uint8: PA_FP8_E4M3, torch.float8_e4m3fn: PA_FP8_E4M3}

EXPORTS = ("pa_status_string", "pa_last_error", "pa_set_option", "pa_get_option", "pa_set_check_mode",
           "pa_device_status", "pa_slot_mapping", "pa_write_kv", "pa_copy_blocks", "pa_decode_workspace_size",
           "pa_decode", "pa_decode_append", "pa_varlen_workspace_size", "pa_varlen", "pa_decode_noalloc",
           "pa_swap_blocks", "pa_write_kv_fp8", "pa_decode_fp8_workspace_size", "pa_decode_fp8",
           "pa_decode_append_fp8", "pa_selftest_wait_timeout", "pa_varlen_fp8_workspace_size", "pa_varlen_fp8")


class PAError(RuntimeError):
    def __init__(self, status, name, reason):
        super().__init__("%s failed: %s (%s)" % (name, name_of(status), reason))
        self.status = status


_lib = None


def lib():
    """The loaded library (loads it on first use; raises if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpa.so is not built (%s); run __graft_entry__.build() first" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    ci, cf = ctypes.c_int, ctypes.c_float
    sig = {
        "pa_status_string": ([ci], ctypes.c_char_p),
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_set_option": ([ci, i64], ci),
        "pa_get_option": ([ci], i64),
        "pa_set_check_mode": ([ci], ci),
        "pa_device_status": ([ci], ci),
        "pa_selftest_wait_timeout": ([i32, vp], ci),
        "pa_slot_mapping": ([vp, i32, i32, vp, vp, i64, i32, vp, vp], ci),
        "pa_write_kv": ([vp, vp, vp, i64, vp, vp, i32, i32, i32, i32, ci, vp], ci),
        "pa_write_kv_fp8": ([vp, vp, vp, i64, vp, vp, vp, vp, i32, i32, i32, i32, ci, vp], ci),
        "pa_decode_fp8_workspace_size": ([i32, i32, i32, i32, i32, i32, ci], sz),
        "pa_decode_append_fp8": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, cf,
                                  ci, vp, sz, vp], ci),
        "pa_decode_fp8": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, cf, ci, vp, sz,
                           vp], ci),
        "pa_copy_blocks": ([vp, vp, i32, vp, i32, i32, i32, i32, i32, ci, vp], ci),
        "pa_swap_blocks": ([vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, ci, vp], ci),
        "pa_decode_workspace_size": ([i32, i32, i32, i32, i32, i32, ci], sz),
        "pa_decode": ([vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, cf, ci, vp, sz, vp], ci),
        "pa_decode_append": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, cf, ci, vp, sz,
                              vp], ci),
        "pa_varlen_workspace_size": ([i32, i32, i32, i32, i32, i32, i32, i32, ci], sz),
        "pa_decode_noalloc": ([vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32, cf, ci, vp], ci),
        "pa_varlen": ([vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, cf, ci, ci, vp,
                       sz, vp], ci),
        "pa_varlen_fp8_workspace_size": ([i32, i32, i32, i32, i32, i32, i32, i32, ci], sz),
        "pa_varlen_fp8": ([vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, cf,
                           ci, ci, vp, sz, vp], ci),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def name_of(status):
    return lib().pa_status_string(status).decode()


def _check(status, name):
    if status != 0:
        raise PAError(status, name, lib().pa_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype(t):
    try:
        return DTYPE_CODE[t.dtype]
    except KeyError:
        raise TypeError("unsupported dtype %s" % t.dtype)


def _pool_dtype(t):
    try:
        return POOL_DTYPE_CODE[t.dtype]
    except KeyError:
        raise TypeError("unsupported pool dtype %s" % t.dtype)


def _dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def pa_set_option(option, value):
    _check(lib().pa_set_option(option, value), "pa_set_option")


def pa_get_option(option):
    return lib().pa_get_option(option)


def pa_set_check_mode(on):
    _check(lib().pa_set_check_mode(1 if on else 0), "pa_set_check_mode")


def pa_selftest_wait_timeout(polls=1000, stream=None):
    """Run the bounded-wait self-test (a wait nothing completes gives up and sets the
    timeout bit that pa_device_status reports)."""
    _check(lib().pa_selftest_wait_timeout(polls, _stream(stream)), "pa_selftest_wait_timeout")


def pa_device_status(clear=True):
    _check(lib().pa_device_status(1 if clear else 0), "pa_device_status")


def pa_slot_mapping(block_tables, seq_idx, positions, block_size, slot_out=None, stream=None):
    """slot_out[i] = block_tables[seq_idx[i], positions[i] // bs] * bs + positions[i] % bs (-1 for pos < 0)."""
    if slot_out is None:
        slot_out = torch.empty(positions.shape[0], dtype=torch.int64, device=positions.device)
    _dev(block_tables, seq_idx, positions, slot_out)
    st = lib().pa_slot_mapping(_ptr(block_tables), block_tables.shape[0], block_tables.shape[1], _ptr(seq_idx),
                               _ptr(positions), positions.shape[0], block_size, _ptr(slot_out), _stream(stream))
    _check(st, "pa_slot_mapping")
    return slot_out


def pa_write_kv(k, v, slot_mapping, k_cache, v_cache, stream=None):
    """Row scatter of k, v [N, Hkv, hd] into caches [NB, bs, Hkv, hd] at slot_mapping [N]."""
    _dev(k, v, slot_mapping, k_cache, v_cache)
    nb, bs, hkv, hd = k_cache.shape
    st = lib().pa_write_kv(_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.shape[0], _ptr(k_cache),
                           _ptr(v_cache), nb, bs, hkv, hd, _dtype(k_cache), _stream(stream))
    _check(st, "pa_write_kv")


def pa_write_kv_fp8(k, v, slot_mapping, k_codes, v_codes, k_scales, v_scales, stream=None):
    """Quantizing write: rows of k, v [N, Hkv, hd] -> E4M3 codes [NB, bs, Hkv, hd] (uint8) at
    slot_mapping [N] and one fp32 scale per row in scales [NB, Hkv, bs]."""
    _dev(k, v, slot_mapping, k_codes, v_codes, k_scales, v_scales)
    nb, bs, hkv, hd = k_codes.shape
    if tuple(k_scales.shape) != (nb, hkv, bs) or tuple(v_scales.shape) != (nb, hkv, bs):
        raise ValueError("scales must be [num_blocks, num_kv_heads, block_size]")
    if k_scales.dtype != torch.float32 or v_scales.dtype != torch.float32:
        raise TypeError("scales must be float32")
    st = lib().pa_write_kv_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.shape[0], _ptr(k_codes),
                               _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), nb, bs, hkv, hd, _dtype(k),
                               _stream(stream))
    _check(st, "pa_write_kv_fp8")


def pa_copy_blocks(k_caches, v_caches, block_pairs, stream=None):
    """Copy block pairs [P, 2] (src, dst) in every layer's K and V cache.  Pools are
    [NB, bs, Hkv, hd] (uint8: E4M3 codes) or a quantized cache's scales [NB, Hkv, bs]."""
    if isinstance(k_caches, torch.Tensor):
        k_caches, v_caches = [k_caches], [v_caches]
    _dev(block_pairs, *k_caches, *v_caches)
    n = len(k_caches)
    kp = (ctypes.c_void_p * n)(*[c.data_ptr() for c in k_caches])
    vp = (ctypes.c_void_p * n)(*[c.data_ptr() for c in v_caches])
    if k_caches[0].dim() == 3:  # scale pools of a quantized cache: [NB, Hkv, bs]
        nb, hkv, bs = k_caches[0].shape
        hd = 1
    else:
        nb, bs, hkv, hd = k_caches[0].shape
    st = lib().pa_copy_blocks(kp, vp, n, _ptr(block_pairs), block_pairs.shape[0], nb, bs, hkv, hd,
                              _pool_dtype(k_caches[0]), _stream(stream))
    _check(st, "pa_copy_blocks")


def pa_swap_blocks(src_k, src_v, dst_k, dst_v, block_pairs, stream=None):
    """Copy blocks between two pools (device or pinned host tensors), every layer:
    dst[pairs[p, 1]] = src[pairs[p, 0]]."""
    if isinstance(src_k, torch.Tensor):
        src_k, src_v, dst_k, dst_v = [src_k], [src_v], [dst_k], [dst_v]
    for t in list(src_k) + list(src_v) + list(dst_k) + list(dst_v) + [block_pairs]:
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("pools and pairs must be contiguous CUDA or pinned host tensors")
    n = len(src_k)
    arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])  # noqa: E731
    nbs, bs, hkv, hd = src_k[0].shape
    st = lib().pa_swap_blocks(arr(src_k), arr(src_v), arr(dst_k), arr(dst_v), n, _ptr(block_pairs),
                              block_pairs.shape[0], nbs, dst_k[0].shape[0], bs, hkv, hd, _pool_dtype(src_k[0]),
                              _stream(stream))
    _check(st, "pa_swap_blocks")


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context, dtype):
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else dtype
    return lib().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context, code)


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context, scale, workspace=None,
              stream=None):
    """One query per sequence: out, q [S, Hq, hd]; context_lens [S]; tables [S, max_blocks]."""
    _dev(out, q, k_cache, v_cache, block_tables, context_lens, workspace)
    nb, bs, hkv, hd = k_cache.shape
    S, hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                         block_tables.shape[1], _ptr(context_lens), S, hq, hkv, hd, nb, bs, max_context,
                         float(scale), _dtype(q), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_decode_fp8_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context, dtype):
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else dtype
    return lib().pa_decode_fp8_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context,
                                              code)


def pa_decode_fp8(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, max_context, scale,
                  workspace=None, stream=None):
    """Decode over a quantized cache: codes [NB, bs, Hkv, hd] uint8, scales [NB, Hkv, bs] fp32;
    out, q [S, Hq, hd] of the query type."""
    _dev(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, workspace)
    nb, bs, hkv, hd = k_codes.shape
    S, hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_decode_fp8(_ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
                             _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), S, hq, hkv, hd, nb, bs,
                             max_context, float(scale), _dtype(q), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pa_decode_fp8")
    return out


def pa_decode_append_fp8(out, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                         max_context, scale, workspace=None, stream=None):
    """The generation step over a quantized cache: each sequence's new rows k_new, v_new
    [S, Hkv, hd] (query type) are quantized into the slot of position L-1, then decoded."""
    _dev(out, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, workspace)
    nb, bs, hkv, hd = k_codes.shape
    S, hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_decode_append_fp8(_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(v_codes),
                                    _ptr(k_scales), _ptr(v_scales), _ptr(block_tables), block_tables.shape[1],
                                    _ptr(context_lens), S, hq, hkv, hd, nb, bs, max_context, float(scale), _dtype(q),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pa_decode_append_fp8")
    return out


def pa_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, max_context, scale,
                     workspace=None, stream=None):
    """Write each sequence's new token (position L-1) into the pool and
    decode: out, q [S, Hq, hd]; k_new, v_new [S, Hkv, hd]."""
    _dev(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, workspace)
    nb, bs, hkv, hd = k_cache.shape
    S, hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_decode_append(_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), S, hq, hkv, hd, nb,
                                bs, max_context, float(scale), _dtype(q), _ptr(workspace), ws_bytes,
                                _stream(stream))
    _check(st, "pa_decode_append")
    return out


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, max_context, scale, stream=None):
    """pa_decode without a workspace: the scratch is the library's fixed
    per-device array (for callers that cannot allocate device memory)."""
    _dev(out, q, k_cache, v_cache, block_tables, context_lens)
    nb, bs, hkv, hd = k_cache.shape
    S, hq, _ = q.shape
    st = lib().pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 block_tables.shape[1], _ptr(context_lens), S, hq, hkv, hd, nb, bs, max_context,
                                 float(scale), _dtype(q), _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out


def pa_varlen_workspace_size(num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim, block_size, max_context,
                             dtype):
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else dtype
    return lib().pa_varlen_workspace_size(num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim, block_size,
                                          max_context, code)


def pa_varlen(out, q, k_cache, v_cache, block_tables, seq_lens, cu_seqlens_q, max_q, max_context, scale,
              causal=True, workspace=None, stream=None):
    """Mixed prefill/decode: q, out [T, Hq, hd]; cu_seqlens_q [S+1]; seq_lens [S]."""
    _dev(out, q, k_cache, v_cache, block_tables, seq_lens, cu_seqlens_q, workspace)
    nb, bs, hkv, hd = k_cache.shape
    T, hq, _ = q.shape
    S = seq_lens.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_varlen(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                         block_tables.shape[1], _ptr(seq_lens), _ptr(cu_seqlens_q), S, T, max_q, hq, hkv, hd, nb,
                         bs, max_context, float(scale), 1 if causal else 0, _dtype(q), _ptr(workspace), ws_bytes,
                         _stream(stream))
    _check(st, "pa_varlen")
    return out


def pa_varlen_fp8_workspace_size(num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim, block_size,
                                 max_context, dtype):
    code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else dtype
    return lib().pa_varlen_fp8_workspace_size(num_seqs, total_q, max_q, num_heads, num_kv_heads, head_dim,
                                              block_size, max_context, code)


def pa_varlen_fp8(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, seq_lens, cu_seqlens_q, max_q,
                  max_context, scale, causal=True, workspace=None, stream=None):
    """Mixed prefill/decode over a quantized cache: codes [NB, bs, Hkv, hd] uint8, scales [NB, Hkv, bs] fp32;
    q, out [T, Hq, hd] of the query type; cu_seqlens_q [S+1]; seq_lens [S]."""
    _dev(out, q, k_codes, v_codes, k_scales, v_scales, block_tables, seq_lens, cu_seqlens_q, workspace)
    nb, bs, hkv, hd = k_codes.shape
    T, hq, _ = q.shape
    S = seq_lens.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pa_varlen_fp8(_ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
                             _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), _ptr(cu_seqlens_q), S, T, max_q,
                             hq, hkv, hd, nb, bs, max_context, float(scale), 1 if causal else 0, _dtype(q),
                             _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pa_varlen_fp8")
    return out
