"""libfusedxtx for GB300: ``out = alpha * X^T (v * (X y)) + beta * z`` in one pass over X.

The pattern and its instantiations come from "On optimizing machine learning
workloads via kernel fusion" (abstract). Every step of the computation runs in the
CUDA kernels of ``libfusedxtx.so`` (sources in ``csrc/``, C ABI in
``include/fxtx.h``); this package only marshals arguments. There is no CPU
fallback: if the library cannot be loaded, importing the binding fails.

Raw C-ABI calls (pointers as ints, stream as a cudaStream_t int) carry the C names:
``fxtx_dense_f32``, ``fxtx_dense_f64``, ``fxtx_dense_bf16``, ``fxtx_dense_f32_noalloc``,
``fxtx_dense_multi_f32``, ``fxtx_dense_multi_f64``, ``fxtx_csr_f32``, ``fxtx_csr_f64``,
``fxtx_csr_validate``, ``fxtx_csr_analyze``, ``fxtx_csr_analysis_clear``,
``fxtx_csr_plan_describe_host``, ``fxtx_epilogue_f32``, ``fxtx_epilogue_f64``, ``fxtx_device_error``,
``fxtx_status_string``,
``fxtx_plan_describe``, ``fxtx_multi_plan_describe`` and the ``fxtx_autotune_*`` calls. ``dense``, ``dense_multi`` and
``csr`` take torch CUDA tensors; ``epilogue`` applies alpha * w + beta * z. The module
``distributed`` runs one call across ranks, each holding a block of X's rows.
"""
from ._lib import (  # noqa: F401
    FXTX_ERR_ALLOC,
    FXTX_ERR_BAD_CSR,
    FXTX_ERR_CUDA,
    FXTX_ERR_INVALID_ARG,
    FXTX_ERR_TIMEOUT,
    FXTX_ERR_TOO_LARGE,
    FXTX_ERR_UNSUPPORTED,
    FXTX_OK,
    FxtxError,
    autotune,
    autotune_candidates,
    autotune_clear,
    autotune_entries,
    autotune_load,
    autotune_mode,
    autotune_save,
    csr,
    csr_analysis_clear,
    csr_analyze,
    csr_plan_describe_host,
    csr_validate,
    CsrStats,
    dense,
    dense_multi,
    device_error,
    epilogue,
    fxtx_autotune_candidates,
    fxtx_autotune_clear,
    fxtx_autotune_entries,
    fxtx_autotune_get,
    fxtx_autotune_load,
    fxtx_autotune_save,
    fxtx_autotune_set,
    fxtx_csr_analysis_clear,
    fxtx_csr_analyze,
    fxtx_csr_f32,
    fxtx_csr_f64,
    fxtx_csr_plan_describe_host,
    fxtx_csr_validate,
    fxtx_dense_f32,
    fxtx_dense_f32_noalloc,
    fxtx_dense_bf16,
    fxtx_dense_f64,
    fxtx_dense_multi_f32,
    fxtx_dense_multi_f64,
    fxtx_device_error,
    fxtx_epilogue_f32,
    fxtx_epilogue_f64,
    fxtx_multi_plan_describe,
    fxtx_plan_describe,
    fxtx_status_string,
    library_path,
    multi_plan_describe,
    plan_describe,
)
