"""GB300-native paged-KV attention.

The product is the C-ABI library ``libpa.so`` (include/pa.h); this package
holds its CUDA sources (``csrc/``), the nvcc build (``build.py``), a ctypes
binding with the C entry points' names (``_binding``), and seeded synthetic
inputs (``workloads``).
"""
from ._binding import (  # noqa: F401
    PA_BF16, PA_F16, PA_F32, PA_FP8_E4M3, PA_OPT_CHECK_MODE, PA_OPT_DECODE_CTAS, PA_OPT_DECODE_KERNEL,
    PA_OPT_FP8_PAIR_STEP, PA_OPT_VARLEN_KERNEL, PAError, lib, pa_copy_blocks, pa_decode, pa_decode_append, pa_decode_append_fp8,
    pa_decode_fp8, pa_decode_fp8_workspace_size, pa_decode_noalloc, pa_decode_workspace_size, pa_device_status,
    pa_get_option, pa_selftest_wait_timeout, pa_set_check_mode, pa_set_option, pa_slot_mapping, pa_swap_blocks,
    pa_varlen, pa_varlen_fp8, pa_varlen_fp8_workspace_size, pa_varlen_workspace_size, pa_write_kv, pa_write_kv_fp8)
