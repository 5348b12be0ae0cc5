"""The C-ABI library: it builds, loads, exports every entry point include/pa.h
declares, and its host-side argument checks answer without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_116_gb300 import build

    build.build()
    from paged_kv_cache_116_gb300 import _binding

    return _binding.lib()


def test_header_declares_the_path(lib):
    names = _declared()
    for must in ("pa_slot_mapping", "pa_write_kv", "pa_copy_blocks", "pa_decode", "pa_varlen",
                 "pa_decode_workspace_size", "pa_varlen_workspace_size"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_116_gb300 import _binding

    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(_binding.EXPORTS) == _declared()


def test_status_strings_and_options(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(3) == b"PA_ERR_INDEX"
    assert lib.pa_set_option(2, 17) == 0 and lib.pa_get_option(2) == 17
    assert lib.pa_set_option(2, 0) == 0
    assert lib.pa_set_option(99, 1) == 1  # unknown option
    assert lib.pa_set_option(4, 2) == 0 and lib.pa_get_option(4) == 2  # FP8 pair step: always
    assert lib.pa_set_option(4, 3) == 1  # no such choice
    assert lib.pa_set_option(4, 0) == 0
    assert lib.pa_set_option(0, -1) == 1  # negative value
    assert lib.pa_set_option(3, 2) == 0 and lib.pa_get_option(3) == 2  # varlen: the tcgen05 kernel
    assert lib.pa_set_option(3, 3) == 1  # no such varlen kernel
    assert lib.pa_set_option(3, 0) == 0


def test_argument_errors_need_no_gpu(lib):
    vp = ctypes.c_void_p
    one = vp(16)
    # num_heads not a multiple of num_kv_heads
    st = lib.pa_decode(one, one, one, one, one, 4, one, 2, 6, 4, 128, 10, 16, 64, 1.0, 1, None, 0, None)
    assert st == 1 and b"multiple" in lib.pa_last_error()
    # unknown dtype
    st = lib.pa_write_kv(one, one, one, 1, one, one, 10, 16, 2, 128, 7, None)
    assert st == 1
    # misaligned cache pointer
    st = lib.pa_write_kv(one, one, one, 1, one, vp(18), 10, 16, 2, 128, 1, None)
    assert st == 1 and b"aligned" in lib.pa_last_error()
    # a row that is not a multiple of 16 bytes
    st = lib.pa_write_kv(one, one, one, 1, one, one, 10, 16, 1, 6, 1, None)
    assert st == 2
    # too many layers for one copy call
    arr = (vp * 1)(16)
    st = lib.pa_copy_blocks(arr, arr, 129, one, 1, 10, 16, 2, 128, 1, None)
    assert st == 1
    # empty work is a no-op that touches nothing
    assert lib.pa_write_kv(None, None, None, 0, None, None, 10, 16, 2, 128, 1, None) == 0
    assert lib.pa_decode(None, None, None, None, None, 4, None, 0, 8, 2, 128, 10, 16, 64, 1.0, 1, None, 0,
                         None) == 0


def test_varlen_workspace_holds_an_item_for_every_prefill_slot(lib):
    """The tensor-core varlen kernel reads the plan item of every prefill
    slot of its grid (total_q / (P T) + num_seqs slots; P query tiles per
    CTA, T = 128 / G tokens per tile) before it knows how many hold work, so
    the workspace must hold that many 16-byte items after its 256-byte
    header, and the decode-row list (4 bytes per request) after them."""
    import numpy as np

    bf16 = 1
    rng = np.random.default_rng(5)
    lib.pa_varlen_workspace_size.restype = ctypes.c_size_t
    for _ in range(300):
        hd = int(rng.choice([64, 128, 256]))
        g = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
        hkv = int(rng.integers(1, 5))
        S = int(rng.integers(1, 5000))
        total_q = int(rng.integers(S, 40 * S + 2))
        ws = lib.pa_varlen_workspace_size(S, total_q, total_q, g * hkv, hkv, hd, 16, 4096, bf16)
        P, T = (1 if hd == 256 else 2), 128 // g
        slots = total_q // (P * T) + S
        assert ws >= 256 + 16 * slots + 4 * S, (hd, g, S, total_q, ws)
