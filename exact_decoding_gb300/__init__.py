"""GB300-native lookahead decoding: the `la_step` hot path as sm_103a CUDA
kernels behind the C ABI in include/la.h, with a thin ctypes binding.

PyTorch is used only for device memory and streams; every step of the path
runs in libla.so.  Import fails loudly if the library has not been built
(`python -m exact_decoding_gb300.build` or `__graft_entry__.build()`).
"""
from .la import (LaError, Decoder, DeviceWeights, la_create, la_prefill, la_step, la_ar_step, la_generate, la_stats,
                 la_export_state, la_import_state, la_debug_logits, la_gemm_bf16, la_gemm_bf16_noalloc, la_gemm_status,
                 la_selftest_timeout, la_gemm_schedule, la_step_tables, la_destroy, la_strerror, load_library, LIB_PATH)

__all__ = ["LaError", "Decoder", "DeviceWeights", "la_create", "la_prefill", "la_step", "la_ar_step", "la_generate", "la_stats",
           "la_export_state", "la_import_state", "la_debug_logits", "la_gemm_bf16", "la_gemm_bf16_noalloc", "la_gemm_status",
           "la_selftest_timeout", "la_gemm_schedule", "la_step_tables", "la_destroy",
           "la_strerror", "load_library", "LIB_PATH"]
