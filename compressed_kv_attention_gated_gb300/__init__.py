"""Gated-softmax KV compression for NVIDIA GB300 (sm_103a).

The CUDA library ``_lib/libckv.so`` (C ABI in ``include/ckv.h``) holds the
kernels; ``ckv`` is its thin ctypes binding; ``synth`` builds seeded synthetic
inputs of the workloads the library is measured on.
"""
from .ckv import (  # noqa: F401
    CkvError,
    ckv_c128_online_decode,
    ckv_c128_online_decode_fp8,
    ckv_c128_online_prefill,
    ckv_c128_online_prefill_fp8,
    ckv_c128_online_prefill_counted,
    ckv_c128_online_prefill_counted_fp8,
    ckv_c128_prefill_set_variant,
    ckv_check_distinct,
    ckv_check_distinct_noalloc,
    ckv_expand_pools_and_append_tail,
    ckv_kpool_compress,
    ckv_kpool_compress_set_variant,
    ckv_kpool_decode_update,
    ckv_kpool_seed_tail,
    ckv_latency_probe,
    ckv_plan_online_prefill,
    ckv_plan_online_prefill_device,
    ckv_wait_timeout_selftest,
    load,
)
