"""GB300 (sm_103a) Q4_K mixture-of-experts layer: CUDA kernels behind a C ABI.

The compute lives in libq4kmoe.so (csrc/, declared in include/q4kmoe.h); this
package is the thin ctypes binding (``_lib``), the library build (``build``),
the seeded synthetic-input generators (``inputs``) and the workload table
(``workloads``). Importing the package does not load the CUDA library; the
first call does, and raises if it cannot.
"""
from ._lib import (  # noqa: F401
    FMT_AFFINE4,
    FMT_Q4TP,
    PATH_PERSISTENT,
    PATH_PERSISTENT_WIDE,
    PATH_TWO_LAUNCH,
    Q4KError,
    ROUTE_SIGMOID_GROUPED,
    ROUTE_SOFTMAX,
    SHARED_NONE,
    SHARED_SIGMOID,
    SHARED_UNSCALED,
    load,
    lib_path,
    moe_combine_residual,
    q4k_expert_ffn_forward,
    q4k_expert_ffn_forward_noalloc,
    q4k_expert_ffn_noalloc_max_scratch_bytes,
    q4k_moe_bucket,
    q4k_moe_id_gemv,
    q4k_moe_id_gemv_fmt,
    q4k_moe_layer_forward,
    q4k_moe_layer_down,
    q4k_moe_layer_forward_host,
    q4k_moe_layer_gate_up,
    q4k_moe_layer_half_workspace_size,
    q4k_moe_layer_launch_count,
    q4k_moe_layer_forward_routed,
    q4k_moe_layer_path,
    q4k_moe_layer_routed_workspace_size,
    q4k_moe_layer_host_staging_size,
    q4k_moe_layer_workspace_size,
    q4k_moe_router,
    q4k_rms_norm,
    q4k_moe_workspace_size,
    q4k_quantize_rows,
    q4k_stream_ceiling,
    q4k_stream_ceiling_sink_words,
    q4k_version,
)
