"""CPU oracle for the Q4_K mixture-of-experts id-GEMV layer (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import this package. The product path (the
CUDA library and its Python binding) never does, and the two share no code.

The arithmetic lives in ``q4k_oracle.c`` (plain C, fp64 accumulation); this
module builds it with gcc on first use and wraps each entry point for numpy
arrays. Definitions and their sources are documented in ``q4k_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("q4k_oracle.c", "q4o_route.c", "q4o_fmt4.c")]
_HDR = os.path.join(_HERE, "q4k_oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 256
BLOCK_BYTES = 144


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP when available). Returns its path."""
    with _lock:
        fresh = (os.path.exists(_LIB_PATH)
                 and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS + [_HDR]))
        if fresh and not force:
            return _LIB_PATH
        base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                "-Wall", "-Wextra", "-Wno-unused-parameter"]
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        for extra in (["-fopenmp"], []):
            cmd = base + extra + ["-o", tmp] + _SRCS + ["-lm"]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode == 0:
                os.replace(tmp, _LIB_PATH)
                return _LIB_PATH
        raise RuntimeError("oracle build failed:\n" + res.stderr)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    sig = {
        "q4o_half_to_float": (ctypes.c_float, [ctypes.c_uint16]),
        "q4o_float_to_half_rne": (ctypes.c_uint16, [ctypes.c_float]),
        "q4o_half_to_float_n": (None, [P, P, i64]),
        "q4o_float_to_half_rne_n": (None, [P, P, i64]),
        "q4o_block_scale_min": (None, [P, i32, P, P]),
        "q4o_dequant_block": (None, [P, P]),
        "q4o_weight_at": (ctypes.c_float, [P, i64]),
        "q4o_dequant_rows": (None, [P, i64, i64, P, i32]),
        "q4o_quantize_rows": (None, [P, i64, i64, P]),
        "q4o_moe_id_gemv": (i32, [P, i32, P, i64, i64, P, i32, i32, i32, i32, P]),
        "q4o_moe_id_gemv_f64": (i32, [P, i32, P, i64, i64, P, i32, i32, i32, i32, P]),
        "q4o_silu": (ctypes.c_double, [ctypes.c_double]),
        "q4o_expert_ffn": (i32, [P, P, P, i32, P, P, i32, i32, i32, i32, P]),
        "q4o_moe_combine": (None, [P, P, P, P, P, i32, i32, i32, i32, P]),
        "q4o_moe_layer": (i32, [P, P, P, i32, P, P, P, i32, i32, P, P, P, P, P, i32, i32, i32, i32, P]),
        "q4o_bucket": (i32, [P, i32, i32, P, P, P]),
        "q4o_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
        "q4o_router_logits": (None, [P, P, i32, i32, i32, P]),
        "q4o_route_softmax": (i32, [P, i32, i32, i32, i32, P, P]),
        "q4o_route_sigmoid_grouped": (i32, [P, P, i32, i32, i32, i32, i32, i32, ctypes.c_double, P, P]),
        "q4o_rms_norm": (None, [P, P, i32, i32, ctypes.c_double, P]),
        "q4o_affine4_dequant": (None, [P, ctypes.c_uint64, ctypes.c_uint64, i64, i64, i32, P]),
        "q4o_q4tp_dequant": (None, [P, i64, i64, P]),
        "q4o_fmt4_matrix_bytes": (ctypes.c_uint64, [i32, i64, i64, i32]),
        "q4o_moe_id_gemv_fmt4": (i32, [i32, P, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, i32, i32, P,
                                       i64, i64, P, i32, i32, i32, i32, P]),
        "q4o_set_threads": (i32, [i32]),
        "q4o_get_threads": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(arr):
    return None if arr is None else arr.ctypes.data


def _c(arr, dtype):
    return np.ascontiguousarray(arr, dtype=dtype)


# ---- binary16 ------------------------------------------------------------------------------

def half_to_float(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _load().q4o_half_to_float_n(_ptr(h), _ptr(out), h.size)
    return out


def float_to_half_bits(f) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().q4o_float_to_half_rne_n(_ptr(f), _ptr(out), f.size)
    return out


# ---- Q4_K decode ----------------------------------------------------------------------------

def scale_min(block, j: int):
    block = _c(block, np.uint8)
    sc, mn = ctypes.c_int(), ctypes.c_int()
    _load().q4o_block_scale_min(_ptr(block), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def dequant_block(block) -> np.ndarray:
    block = _c(block, np.uint8)
    assert block.size == BLOCK_BYTES
    out = np.empty(QK, np.float32)
    _load().q4o_dequant_block(_ptr(block), _ptr(out))
    return out


def weight_at(row, k: int) -> float:
    row = _c(row, np.uint8)
    return float(_load().q4o_weight_at(_ptr(row), k))


def dequant_rows(w, rows: int, k: int, elementwise: bool = False) -> np.ndarray:
    w = _c(w, np.uint8)
    assert w.size == rows * (k // QK) * BLOCK_BYTES
    out = np.empty((rows, k), np.float32)
    _load().q4o_dequant_rows(_ptr(w), rows, k, _ptr(out), 1 if elementwise else 0)
    return out


def quantize_rows(x) -> np.ndarray:
    """Quantize a [rows, k] float32 matrix to Q4_K bytes [rows, k/256*144]."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % QK == 0
    out = np.empty((rows, (k // QK) * BLOCK_BYTES), np.uint8)
    _load().q4o_quantize_rows(_ptr(x), rows, k, _ptr(out))
    return out


# ---- MoE id-GEMV / FFN / combine / layer -----------------------------------------------------

def moe_id_gemv(w, num_experts, a, outer, inner, ids, m, top_k, n, k):
    """fp64 out[m*top_k, n] and the count of out-of-range ids."""
    w = _c(w, np.uint8)
    ids = _c(ids, np.int32)
    out = np.empty((m * top_k, n), np.float64)
    if np.asarray(a).dtype == np.float64:
        a = _c(a, np.float64)
        bad = _load().q4o_moe_id_gemv_f64(_ptr(w), num_experts, _ptr(a), outer, inner, _ptr(ids),
                                          m, top_k, n, k, _ptr(out))
    else:
        a = _c(a, np.float32)
        bad = _load().q4o_moe_id_gemv(_ptr(w), num_experts, _ptr(a), outer, inner, _ptr(ids),
                                      m, top_k, n, k, _ptr(out))
    return out, bad


def silu(x: float) -> float:
    return float(_load().q4o_silu(float(x)))


def expert_ffn(w_gate, w_up, w_down, num_experts, h_post, ids, m, top_k, hidden, inter):
    """fp64 expert_out[m*top_k, hidden] and the count of out-of-range ids."""
    w_gate, w_up, w_down = (_c(x, np.uint8) for x in (w_gate, w_up, w_down))
    h_post = _c(h_post, np.float32)
    ids = _c(ids, np.int32)
    out = np.empty((m * top_k, hidden), np.float64)
    bad = _load().q4o_expert_ffn(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(h_post),
                                 _ptr(ids), m, top_k, hidden, inter, _ptr(out))
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return out, bad


def moe_combine(h_mid, expert_out, weights, shared_out, shared_gate, shared_mode, m, top_k, hidden):
    h_mid = _c(h_mid, np.float64)
    expert_out = _c(expert_out, np.float64)
    weights = _c(weights, np.float64)
    shared_out = None if shared_out is None else _c(shared_out, np.float64)
    shared_gate = None if shared_gate is None else _c(shared_gate, np.float64)
    y = np.empty((m, hidden), np.float64)
    _load().q4o_moe_combine(_ptr(h_mid), _ptr(expert_out), _ptr(weights), _ptr(shared_out),
                            _ptr(shared_gate), shared_mode, m, top_k, hidden, _ptr(y))
    return y


def moe_layer(w_gate, w_up, w_down, num_experts, shared, shared_inter, shared_mode,
              h_post, h_mid, ids, weights, shared_gate, m, top_k, hidden, inter):
    """fp64 y[m, hidden] for the whole layer. ``shared`` = (gate, up, down) slabs or None."""
    w_gate, w_up, w_down = (_c(x, np.uint8) for x in (w_gate, w_up, w_down))
    if shared is None:
        sg = su = sd = None
        shared_mode = 0
    else:
        sg, su, sd = (_c(x, np.uint8) for x in shared)
    h_post = _c(h_post, np.float32)
    h_mid = _c(h_mid, np.float32)
    ids = _c(ids, np.int32)
    weights = _c(weights, np.float32)
    shared_gate = None if shared_gate is None else _c(shared_gate, np.float32)
    y = np.empty((m, hidden), np.float64)
    bad = _load().q4o_moe_layer(_ptr(w_gate), _ptr(w_up), _ptr(w_down), num_experts, _ptr(sg), _ptr(su),
                                _ptr(sd), shared_inter, shared_mode, _ptr(h_post), _ptr(h_mid), _ptr(ids),
                                _ptr(weights), _ptr(shared_gate), m, top_k, hidden, inter, _ptr(y))
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return y, bad


def bucket(ids, num_experts):
    """(counts[E], offsets[E+1], perm[P], n_invalid): stable counting sort of pairs by expert."""
    ids = _c(ids, np.int32)
    P = ids.size
    counts = np.empty(num_experts, np.int32)
    offsets = np.empty(num_experts + 1, np.int32)
    perm = np.empty(P, np.int32)
    bad = _load().q4o_bucket(_ptr(ids), P, num_experts, _ptr(counts), _ptr(offsets), _ptr(perm))
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return counts, offsets, perm, bad


# ---- router and chained norm ---------------------------------------------------------------

FMT_AFFINE = 0
FMT_Q4TP = 1


def bf16_to_double(b: int) -> float:
    return float(_load().q4o_bf16_to_double(int(b)))


def router_logits(x, w_bf16, m, num_experts, hidden):
    """fp64 logits[m, num_experts] = x . bf16(w)^T (w given as uint16 bits)."""
    x = _c(x, np.float32)
    w_bf16 = _c(w_bf16, np.uint16)
    out = np.empty((m, num_experts), np.float64)
    _load().q4o_router_logits(_ptr(x), _ptr(w_bf16), m, num_experts, hidden, _ptr(out))
    return out


def route_softmax(logits, top_k, normalize=True):
    """(ids[m, top_k] int32, weights[m, top_k] fp64): softmax top-k routing."""
    logits = _c(logits, np.float64)
    m, E = logits.shape
    ids = np.empty((m, top_k), np.int32)
    w = np.empty((m, top_k), np.float64)
    rc = _load().q4o_route_softmax(_ptr(logits), m, E, top_k, 1 if normalize else 0, _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("route_softmax: bad arguments")
    return ids, w


def route_sigmoid_grouped(logits, bias, top_k, n_group=1, topk_group=1, normalize=True, scale=1.0):
    """(ids, weights): sigmoid scores, bias-corrected, group-limited top-k (noaux_tc)."""
    logits = _c(logits, np.float64)
    m, E = logits.shape
    bias = None if bias is None else _c(bias, np.float32)
    ids = np.empty((m, top_k), np.int32)
    w = np.empty((m, top_k), np.float64)
    rc = _load().q4o_route_sigmoid_grouped(_ptr(logits), _ptr(bias), m, E, top_k, n_group, topk_group,
                                           1 if normalize else 0, float(scale), _ptr(ids), _ptr(w))
    if rc != 0:
        raise ValueError("route_sigmoid_grouped: bad arguments")
    return ids, w


def rms_norm(x, w_bf16, eps):
    """fp64 x / sqrt(mean(x^2) + eps) * bf16(w), row by row."""
    x = _c(x, np.float64)
    m, H = x.shape
    w_bf16 = _c(w_bf16, np.uint16)
    out = np.empty((m, H), np.float64)
    _load().q4o_rms_norm(_ptr(x), _ptr(w_bf16), m, H, float(eps), _ptr(out))
    return out


# ---- other 4-bit formats ---------------------------------------------------------------------

def affine4_dequant(mat, s_off, b_off, n, k, gs):
    mat = _c(mat, np.uint8)
    out = np.empty((n, k), np.float64)
    _load().q4o_affine4_dequant(_ptr(mat), int(s_off), int(b_off), n, k, gs, _ptr(out))
    return out


def q4tp_dequant(mat, n, k):
    mat = _c(mat, np.uint8)
    out = np.empty((n, k), np.float64)
    _load().q4o_q4tp_dequant(_ptr(mat), n, k, _ptr(out))
    return out


def fmt4_matrix_bytes(fmt, n, k, gs=64):
    return int(_load().q4o_fmt4_matrix_bytes(fmt, n, k, gs))


def moe_id_gemv_fmt4(fmt, w, expert_stride, s_off, b_off, gs, num_experts, a, outer, inner, ids, m, top_k, n, k):
    """fp64 out[m*top_k, n] and the count of out-of-range ids, for an affine or q4tp slab."""
    w = _c(w, np.uint8)
    a = _c(a, np.float32)
    ids = _c(ids, np.int32)
    out = np.empty((m * top_k, n), np.float64)
    bad = _load().q4o_moe_id_gemv_fmt4(fmt, _ptr(w), int(expert_stride), int(s_off), int(b_off), gs, num_experts,
                                       _ptr(a), outer, inner, _ptr(ids), m, top_k, n, k, _ptr(out))
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return out, bad


def set_threads(n: int) -> int:
    return int(_load().q4o_set_threads(int(n)))


def get_threads() -> int:
    return int(_load().q4o_get_threads())
