"""ctypes binding of libq4kmoe.so: argument marshalling only.

Every function here forwards torch tensors (as raw pointers) and sizes to the C
ABI of include/q4kmoe.h, on the current torch CUDA stream unless one is given,
and raises Q4KError on any non-OK status. There is no fallback: if the CUDA
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

Q4K_OK = 0
STATUS_NAMES = {
    0: "Q4K_OK", 1: "Q4K_ERR_NULL", 2: "Q4K_ERR_SHAPE", 3: "Q4K_ERR_TOPK", 4: "Q4K_ERR_WORKSPACE",
    5: "Q4K_ERR_CUDA", 6: "Q4K_ERR_EXPERT_ID", 7: "Q4K_ERR_ALIGN", 8: "Q4K_ERR_MODE", 9: "Q4K_ERR_LIMIT",
    10: "Q4K_ERR_TIMEOUT",
}
SHARED_NONE, SHARED_SIGMOID, SHARED_UNSCALED = 0, 1, 2
PATH_TWO_LAUNCH, PATH_PERSISTENT, PATH_PERSISTENT_WIDE = 0, 1, 2
ROUTE_SOFTMAX, ROUTE_SIGMOID_GROUPED = 0, 1
FMT_AFFINE4, FMT_Q4TP = 1, 2

# Exported C symbols and their signatures (restype, argtypes).
_P, _I, _I64, _U64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
SIGNATURES = {
    "q4k_last_error_string": (ctypes.c_char_p, []),
    "q4k_version": (ctypes.c_char_p, []),
    "q4k_moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "q4k_moe_layer_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "q4k_moe_layer_host_staging_size": (_SZ, [_I, _I, _I]),
    "q4k_moe_bucket": (_I, [_P, _I, _I, _P, _P, _P, _P, _P]),
    "q4k_moe_id_gemv": (_I, [_P, _U64, _I, _P, _I64, _I64, _P, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "q4k_expert_ffn_forward": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "q4k_expert_ffn_noalloc_max_scratch_bytes": (_SZ, []),
    "q4k_expert_ffn_forward_noalloc": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_combine_residual": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "q4k_moe_layer_forward": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P,
                                   _P, _SZ, _P, _P]),
    "q4k_moe_layer_forward_host": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                        _P, _P, _SZ, _P, _P]),
    "q4k_moe_layer_gate_up": (_I, [_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P, _P]),
    "q4k_moe_layer_down": (_I, [_P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P, _P]),
    "q4k_moe_layer_half_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "q4k_moe_layer_launch_count": (_I, [_I, _I, _I, _I, _I, _I]),
    "q4k_moe_layer_path": (_I, [_I, _I, _I, _I, _I, _I]),
    "q4k_moe_id_gemv_fmt": (_I, [_I, _P, _P, _U64, _U64, _U64, _U64, _I, _I, _P, _I64, _I64, _P, _I, _I, _I, _I, _P,
                                 _P, _P]),
    "q4k_moe_layer_routed_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "q4k_moe_layer_forward_routed": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I,
                                          ctypes.c_float, _I, _I, _I, _I, _I, _I, _P, _P, ctypes.c_float, _P, _P,
                                          _P, _P, _SZ, _P, _P]),
    "q4k_moe_router": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _I, _P, _P, _P, _P, _P]),
    "q4k_rms_norm": (_I, [_P, _P, _I, _I, ctypes.c_float, _P, _P]),
    "q4k_quantize_rows": (_I, [_P, _I64, _I, _P, _P]),
    "q4k_stream_ceiling_sink_words": (_I, []),
    "q4k_stream_ceiling": (_I, [_P, _U64, _P, _P]),
}


class Q4KError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_needed: bool = True):
    """Load libq4kmoe.so (building it with nvcc first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_needed and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"CUDA library missing: {_build.LIB_PATH} (build with python -m bit_quantized_moe_q4k_gb300.build)")
        lib = ctypes.CDLL(_build.LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int) -> None:
    if status != Q4K_OK:
        msg = load().q4k_last_error_string().decode()
        raise Q4KError(status, msg)


def _cuda(*tensors) -> None:
    for t in tensors:
        if t is not None and not isinstance(t, int) and not t.is_cuda:
            raise ValueError("device tensor expected")


# ---- sizes -------------------------------------------------------------------------------------

def q4k_moe_workspace_size(m, top_k, num_experts, n_max, k_max) -> int:
    return int(load().q4k_moe_workspace_size(m, top_k, num_experts, n_max, k_max))


def q4k_moe_layer_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter) -> int:
    return int(load().q4k_moe_layer_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter))


def q4k_moe_layer_host_staging_size(m, top_k, hidden) -> int:
    return int(load().q4k_moe_layer_host_staging_size(m, top_k, hidden))


def q4k_version() -> str:
    return load().q4k_version().decode()


# ---- calls -------------------------------------------------------------------------------------

def q4k_moe_bucket(ids, n_pairs, num_experts, counts, offsets, perm, err_flag=None, stream=None):
    _cuda(ids, counts, offsets, perm, err_flag)
    _check(load().q4k_moe_bucket(_ptr(ids), n_pairs, num_experts, _ptr(counts), _ptr(offsets), _ptr(perm),
                                 _ptr(err_flag), _stream(stream)))


def q4k_moe_id_gemv(w_stacked, w_byte_offset, num_experts, a, src1_outer_stride, src1_inner_stride, ids, m, top_k,
                    n, k, out, workspace=None, ws_bytes=0, err_flag=None, stream=None):
    _cuda(w_stacked, a, ids, out, workspace, err_flag)
    _check(load().q4k_moe_id_gemv(_ptr(w_stacked), w_byte_offset, num_experts, _ptr(a), src1_outer_stride,
                                  src1_inner_stride, _ptr(ids), m, top_k, n, k, _ptr(out), _ptr(workspace), ws_bytes,
                                  _ptr(err_flag), _stream(stream)))


def q4k_expert_ffn_forward(w_gate, w_up, w_down, num_experts, h_post, ids, m, top_k, hidden, inter, expert_out,
                           workspace, ws_bytes, err_flag=None, stream=None):
    _cuda(w_gate, w_up, w_down, h_post, ids, expert_out, workspace, err_flag)
    _check(load().q4k_expert_ffn_forward(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(h_post), _ptr(ids),
                                         m, top_k, hidden, inter, _ptr(expert_out), _ptr(workspace), ws_bytes,
                                         _ptr(err_flag), _stream(stream)))


def q4k_expert_ffn_noalloc_max_scratch_bytes() -> int:
    return int(load().q4k_expert_ffn_noalloc_max_scratch_bytes())


def q4k_expert_ffn_forward_noalloc(w_gate, w_up, w_down, num_experts, h_post, ids, m, top_k, hidden, inter,
                                   expert_out, err_flag=None, stream=None):
    """The routed FFN with its scratch in the library's static device array (no allocation)."""
    _cuda(w_gate, w_up, w_down, h_post, ids, expert_out, err_flag)
    _check(load().q4k_expert_ffn_forward_noalloc(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(h_post),
                                                 _ptr(ids), m, top_k, hidden, inter, _ptr(expert_out),
                                                 _ptr(err_flag), _stream(stream)))


def moe_combine_residual(h_mid, expert_out, weights, shared_out, shared_gate, shared_mode, m, top_k, hidden,
                         hidden_out, stream=None):
    _cuda(h_mid, expert_out, weights, shared_out, shared_gate, hidden_out)
    _check(load().moe_combine_residual(_ptr(h_mid), _ptr(expert_out), _ptr(weights), _ptr(shared_out),
                                       _ptr(shared_gate), shared_mode, m, top_k, hidden, _ptr(hidden_out),
                                       _stream(stream)))


def q4k_moe_id_gemv_fmt(fmt, w, w2, w_byte_offset, expert_stride, scales_offset, biases_offset, group_size,
                        num_experts, a, outer, inner, ids, m, top_k, n, k, out, err_flag=None, stream=None):
    """Batched id-GEMV over an MLX-affine (FMT_AFFINE4) or q4tp (FMT_Q4TP) slab; w2: fused gate|up."""
    _cuda(w, w2, a, ids, out, err_flag)
    _check(load().q4k_moe_id_gemv_fmt(fmt, _ptr(w), _ptr(w2), w_byte_offset, expert_stride, scales_offset,
                                      biases_offset, group_size, num_experts, _ptr(a), outer, inner, _ptr(ids), m,
                                      top_k, n, k, _ptr(out), _ptr(err_flag), _stream(stream)))


def q4k_moe_layer_routed_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter) -> int:
    return int(load().q4k_moe_layer_routed_workspace_size(m, top_k, num_experts, hidden, inter, shared_inter))


def q4k_moe_layer_forward_routed(w_gate, w_up, w_down, num_experts, ws_gate, ws_up, ws_down, shared_inter,
                                 shared_mode, h_post, h_mid, w_router, bias, w_shared_gate, scoring, normalize, scale,
                                 n_group, topk_group, m, top_k, hidden, inter, y, w_norm, eps, normed, ids_out,
                                 weights_out, workspace, ws_bytes, err_flag=None, stream=None):
    """Router -> layer -> (optional) RMSNorm from the layer input; one launch for a decode layer."""
    _cuda(w_gate, w_up, w_down, ws_gate, ws_up, ws_down, h_post, h_mid, w_router, bias, w_shared_gate, y, w_norm,
          normed, ids_out, weights_out, workspace, err_flag)
    _check(load().q4k_moe_layer_forward_routed(
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(ws_gate), _ptr(ws_up), _ptr(ws_down), shared_inter,
        shared_mode, _ptr(h_post), _ptr(h_mid), _ptr(w_router), _ptr(bias), _ptr(w_shared_gate), scoring,
        1 if normalize else 0, float(scale), n_group, topk_group, m, top_k, hidden, inter, _ptr(y), _ptr(w_norm),
        float(eps), _ptr(normed), _ptr(ids_out), _ptr(weights_out), _ptr(workspace), ws_bytes, _ptr(err_flag),
        _stream(stream)))


def q4k_moe_router(x, w_router, bias, w_shared_gate, m, num_experts, hidden, top_k, scoring, normalize, scale,
                   n_group, topk_group, ids, weights, logits, shared_gate=None, stream=None):
    """Gate logits, top-k choice and routing weights on the device (w_router / w_shared_gate: bf16 bits as
    int16/uint16 tensors)."""
    _cuda(x, w_router, bias, w_shared_gate, ids, weights, logits, shared_gate)
    _check(load().q4k_moe_router(_ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_shared_gate), m, num_experts, hidden,
                                 top_k, scoring, 1 if normalize else 0, float(scale), n_group, topk_group, _ptr(ids),
                                 _ptr(weights), _ptr(logits), _ptr(shared_gate), _stream(stream)))


def q4k_rms_norm(x, w, m, hidden, eps, out, stream=None):
    """out = x / sqrt(mean(x^2) + eps) * bf16(w), row by row (w: bf16 bits)."""
    _cuda(x, w, out)
    _check(load().q4k_rms_norm(_ptr(x), _ptr(w), m, hidden, float(eps), _ptr(out), _stream(stream)))


def q4k_moe_layer_forward(w_gate, w_up, w_down, num_experts, ws_gate, ws_up, ws_down, shared_inter, shared_mode,
                          h_post, h_mid, ids, weights, shared_gate, m, top_k, hidden, inter, y, workspace, ws_bytes,
                          err_flag=None, stream=None):
    _cuda(w_gate, w_up, w_down, ws_gate, ws_up, ws_down, h_post, h_mid, ids, weights, shared_gate, y, workspace,
          err_flag)
    _check(load().q4k_moe_layer_forward(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(ws_gate),
                                        _ptr(ws_up), _ptr(ws_down), shared_inter, shared_mode, _ptr(h_post),
                                        _ptr(h_mid), _ptr(ids), _ptr(weights), _ptr(shared_gate), m, top_k, hidden,
                                        inter, _ptr(y), _ptr(workspace), ws_bytes, _ptr(err_flag), _stream(stream)))


def q4k_moe_layer_forward_host(w_gate, w_up, w_down, num_experts, ws_gate, ws_up, ws_down, shared_inter, shared_mode,
                               h_post, h_mid, ids, weights, shared_gate, m, top_k, hidden, inter, y, workspace,
                               ws_bytes, err_flag=None, stream=None):
    """h_post, h_mid, ids, weights, shared_gate and y are HOST tensors. Page-locked (pinned) ones are
    read and written by the kernels directly; pageable ones are copied, one transfer per buffer."""
    _cuda(w_gate, w_up, w_down, ws_gate, ws_up, ws_down, workspace, err_flag)
    _check(load().q4k_moe_layer_forward_host(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(ws_gate),
                                             _ptr(ws_up), _ptr(ws_down), shared_inter, shared_mode, _ptr(h_post),
                                             _ptr(h_mid), _ptr(ids), _ptr(weights), _ptr(shared_gate), m, top_k,
                                             hidden, inter, _ptr(y), _ptr(workspace), ws_bytes, _ptr(err_flag),
                                             _stream(stream)))


def q4k_moe_layer_launch_count(m, top_k, num_experts, hidden, inter, shared_inter) -> int:
    return int(load().q4k_moe_layer_launch_count(m, top_k, num_experts, hidden, inter, shared_inter))


def q4k_moe_layer_path(m, top_k, num_experts, hidden, inter, shared_inter) -> int:
    """PATH_PERSISTENT_WIDE, PATH_PERSISTENT or PATH_TWO_LAUNCH: the kernels one layer call runs."""
    return int(load().q4k_moe_layer_path(m, top_k, num_experts, hidden, inter, shared_inter))


def q4k_moe_layer_half_workspace_size(m, top_k, k_routed, shared_inter, k_shared) -> int:
    return int(load().q4k_moe_layer_half_workspace_size(m, top_k, k_routed, shared_inter, k_shared))


def q4k_moe_layer_gate_up(w_gate, w_up, num_experts, ws_gate, ws_up, shared_inter, h_post, ids, m, top_k, hidden,
                          inter, act, act_shared, workspace=None, ws_bytes=0, err_flag=None, stream=None):
    _cuda(w_gate, w_up, ws_gate, ws_up, h_post, ids, act, act_shared, workspace, err_flag)
    _check(load().q4k_moe_layer_gate_up(_ptr(w_gate), _ptr(w_up), num_experts, _ptr(ws_gate), _ptr(ws_up),
                                        shared_inter, _ptr(h_post), _ptr(ids), m, top_k, hidden, inter, _ptr(act),
                                        _ptr(act_shared), _ptr(workspace), ws_bytes, _ptr(err_flag),
                                        _stream(stream)))


def q4k_moe_layer_down(w_down, num_experts, ws_down, shared_inter, act, act_shared, ids, m, top_k, hidden, inter,
                       expert_out, shared_out, workspace=None, ws_bytes=0, err_flag=None, stream=None):
    _cuda(w_down, ws_down, act, act_shared, ids, expert_out, shared_out, workspace, err_flag)
    _check(load().q4k_moe_layer_down(_ptr(w_down), num_experts, _ptr(ws_down), shared_inter, _ptr(act),
                                     _ptr(act_shared), _ptr(ids), m, top_k, hidden, inter, _ptr(expert_out),
                                     _ptr(shared_out), _ptr(workspace), ws_bytes, _ptr(err_flag), _stream(stream)))


def q4k_quantize_rows(x, rows, k, out, stream=None):
    _cuda(x, out)
    _check(load().q4k_quantize_rows(_ptr(x), rows, k, _ptr(out), _stream(stream)))


def q4k_stream_ceiling_sink_words() -> int:
    return int(load().q4k_stream_ceiling_sink_words())


def q4k_stream_ceiling(src, nbytes, sink, stream=None):
    _cuda(src, sink)
    _check(load().q4k_stream_ceiling(_ptr(src), nbytes, _ptr(sink), _stream(stream)))
