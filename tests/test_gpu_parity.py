"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Sizes are chosen so the oracle finishes in seconds while the launches still span
several row tiles, several 4-token chunks of one bucket and ragged tails.
Integer results (bucketing, quantizer bytes) must be bit-exact; float results
meet the per-row acceptance of helpers.rows_close.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from bit_quantized_moe_q4k_gb300 import inputs
import bit_quantized_moe_q4k_gb300 as q4k

from helpers import dev, err_flag, host, oracle_slab, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _empty(shape, dtype=None):
    return torch.empty(shape, dtype=dtype or torch.float32, device="cuda")


# ---------------------------------------------------------------------------------------------
# bucketing (bit-exact)

@pytest.mark.parametrize("P,E,bad", [(0, 4, False), (1, 1, False), (6, 4, False), (8, 128, False), (128, 128, True),
                                     (512, 256, False), (3000, 7, True), (37, 4096, True)])
def test_bucket_bit_exact(P, E, bad):
    rng = np.random.default_rng(P + 7 * E)
    lo, hi = (-3, E + 3) if bad else (0, E)
    ids = rng.integers(lo, hi, size=P).astype(np.int32)
    counts, offsets, perm, nbad = oracle.bucket(ids, E)
    d_ids = dev(ids) if P else torch.zeros(1, dtype=torch.int32, device="cuda")
    c, o, p = (_empty(E, torch.int32), _empty(E + 1, torch.int32), _empty(max(P, 1), torch.int32))
    f = err_flag()
    q4k.q4k_moe_bucket(d_ids, P, E, c, o, p, f)
    assert np.array_equal(host(c), counts)
    assert np.array_equal(host(o), offsets)
    assert np.array_equal(host(p)[:P], perm)
    assert int(host(f)[0]) == (6 if nbad else 0)


# ---------------------------------------------------------------------------------------------
# quantizer (bit-exact: both sides take every rounding decision in binary32)

def test_quantizer_bytes_bit_exact():
    rows, k = 96, 2048
    parts = [inputs.normal(31, "qz", (rows, k), 0.02),
             inputs.normal(32, "qz", (8, k), 3.0),
             np.abs(inputs.normal(33, "qz", (4, k), 0.01)),
             -np.abs(inputs.normal(34, "qz", (4, k), 0.01)),
             np.zeros((2, k), np.float32), np.full((2, k), 0.125, np.float32)]
    x = np.concatenate(parts).astype(np.float32)
    ref = oracle.quantize_rows(x)
    out = _empty(ref.shape, torch.uint8)
    q4k.q4k_quantize_rows(dev(x), x.shape[0], k, out)
    got = host(out)
    assert np.array_equal(got, ref), f"{(got != ref).sum()} bytes differ"


# ---------------------------------------------------------------------------------------------
# id-GEMV

def _gemv_case(seed, E, n, k, m, T, mode, ids=None):
    w = oracle_slab(seed, "g", E, n, k)
    if ids is None:
        ids = inputs.ids_uniform_distinct(seed, m, T, E)
    if mode == "gate_up":
        a = inputs.normal(seed, "a", (m, k))
        outer, inner = k, 0
    else:
        a = inputs.normal(seed, "a", (m, T, k))
        outer, inner = T * k, k
    return w, np.asarray(ids, np.int32), a, outer, inner


def _run_gemv(w, E, a, outer, inner, ids, m, T, n, k, flag=None):
    out = _empty((m * T, n))
    q4k.q4k_moe_id_gemv(dev(w), 0, E, dev(a), outer, inner, dev(ids), m, T, n, k, out, err_flag=flag)
    return host(out)


@pytest.mark.parametrize("mode", ["gate_up", "down"])
@pytest.mark.parametrize("E,n,k,m,T", [(4, 64, 256, 3, 2),      # the pages' tiny case shape
                                       (8, 68, 768, 5, 3),      # ragged rows, 3 blocks per row
                                       (6, 100, 1280, 7, 2),    # 4 row tiles, ragged
                                       (3, 32, 2048, 9, 3),     # buckets of 9 pairs -> 3 chunks
                                       (2, 24, 4096, 2, 2),     # 64 threads per row: cross-warp sums
                                       (1, 40, 7168, 2, 1),     # 112 of 128 threads per row, ragged tile
                                       (2, 20, 10240, 1, 2)])   # two 64-weight groups per thread
def test_id_gemv_matches_oracle(mode, E, n, k, m, T):
    w, ids, a, outer, inner = _gemv_case(100 + n, E, n, k, m, T, mode)
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    got = _run_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    rows_close(got, ref, what=f"id-gemv {mode}")


@pytest.mark.parametrize("mode", ["gate_up", "down"])
@pytest.mark.parametrize("E,n,k,m,T", [(64, 36, 256, 2, 16),    # top_k at its limit, one block per row
                                       (64, 36, 256, 5, 16),    # 80 pairs: bucketed path, top_k 16
                                       (4096, 8, 256, 3, 4),    # the expert-count limit
                                       (1, 4, 256, 7, 1)])      # one expert, the smallest n
def test_id_gemv_limits(mode, E, n, k, m, T):
    w, ids, a, outer, inner = _gemv_case(300 + E + m, E, n, k, m, T, mode)
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    got = _run_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    rows_close(got, ref, what=f"id-gemv limits {mode} E={E} T={T}")


@pytest.mark.parametrize("mode", ["gate_up", "down"])
def test_pages_tiny_case(mode):
    """The ferrum-kernels tiny case: its ids and input recipes, against the oracle, and
    batched == per-token calls on the GPU bit for bit."""
    with open(os.path.join(GOLDEN, "ferrum_tiny_case.json")) as f:
        case = json.load(f)
    E, n, k, m, T = case["num_experts"], case["n"], case["k"], case["m"], case["top_k"]
    ids = np.array(case["ids"], np.int32)
    spec = case[mode]
    wp, ap = spec["weight_params"], spec["activation_params"]
    fn, gn = (math.sin, math.cos) if mode == "gate_up" else (math.cos, math.sin)
    w = np.concatenate([oracle.quantize_rows(np.array(
        [wp["amp"] * fn(wp["freq"] * ((i + e * wp["shift"]) % wp["period"])) + wp["bias"] for i in range(n * k)],
        np.float32).reshape(n, k)) for e in range(E)])
    rows = m if mode == "gate_up" else m * T
    a = np.array([ap["amp"] * gn(ap["freq"] * i) for i in range(rows * k)], np.float32)
    outer, inner = (k, 0) if mode == "gate_up" else (T * k, k)
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    batched = _run_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    rows_close(batched, ref, what="tiny case")
    d_w, d_a = dev(w), dev(a)
    per_token = []
    for t in range(m):
        out = _empty((T, n))
        q4k.q4k_moe_id_gemv(d_w, 0, E, d_a[t * outer:], 0, inner, dev(ids[t * T:(t + 1) * T]), 1, T, n, k, out)
        per_token.append(host(out))
    assert np.array_equal(batched, np.concatenate(per_token))


def test_id_gemv_weight_byte_offset_and_duplicates():
    E, n, k, m, T = 5, 64, 512, 4, 3
    w, _, a, outer, inner = _gemv_case(7, E, n, k, m, T, "gate_up")
    ids = np.array([1, 1, 4, 0, 0, 0, 2, 1, 2, 3, 3, 3], np.int32)  # same expert twice in one token
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    pad = 4096
    big = np.zeros(pad + w.size, np.uint8)
    big[pad:] = w.reshape(-1)
    out = _empty((m * T, n))
    q4k.q4k_moe_id_gemv(dev(big), pad, E, dev(a), outer, inner, dev(ids), m, T, n, k, out)
    rows_close(host(out), ref, what="offset+duplicates")


def test_id_gemv_out_of_range_ids_flag_and_zero_rows():
    E, n, k, m, T = 4, 64, 256, 3, 2
    w, _, a, outer, inner = _gemv_case(9, E, n, k, m, T, "gate_up")
    ids = np.array([0, 9, -1, 2, 3, 1], np.int32)
    ref, bad = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    f = err_flag()
    got = _run_gemv(w, E, a, outer, inner, ids, m, T, n, k, flag=f)
    assert bad == 2 and int(host(f)[0]) == 6  # Q4K_ERR_EXPERT_ID
    assert np.all(got[[1, 2]] == 0)
    rows_close(got, ref, what="invalid ids")


def test_id_gemv_empty_batch():
    w, ids, a, outer, inner = _gemv_case(10, 4, 64, 256, 1, 2, "gate_up")
    out = torch.full((2, 64), 7.0, device="cuda")
    q4k.q4k_moe_id_gemv(dev(w), 0, 4, dev(a), outer, inner, dev(ids), 0, 2, 64, 256, out)
    assert np.all(host(out) == 7.0)


def test_id_gemv_skewed_bucket_many_chunks():
    """One expert takes every pair (a Zipf head): 20 pairs -> 5 chunks over the same tiles."""
    E, n, k, m, T = 16, 96, 1024, 20, 1
    w, _, a, outer, inner = _gemv_case(11, E, n, k, m, T, "gate_up")
    ids = np.full(m, 13, np.int32)
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    rows_close(_run_gemv(w, E, a, outer, inner, ids, m, T, n, k), ref, what="skewed")


# ---------------------------------------------------------------------------------------------
# FFN, combine, layer

def _ffn_case(seed, E, H, I, m, T):
    wg, wu = oracle_slab(seed, "gate", E, I, H), oracle_slab(seed, "up", E, I, H)
    wd = oracle_slab(seed, "down", E, H, I)
    ids = inputs.ids_uniform_distinct(seed, m, T, E)
    x = inputs.normal(seed, "h_post", (m, H))
    return wg, wu, wd, ids, x


@pytest.mark.parametrize("E,H,I,m,T", [(8, 512, 256, 5, 2), (16, 1024, 768, 3, 4), (4, 256, 512, 9, 2)])
def test_expert_ffn_matches_oracle(E, H, I, m, T):
    wg, wu, wd, ids, x = _ffn_case(40 + E, E, H, I, m, T)
    ref, _ = oracle.expert_ffn(wg, wu, wd, E, x, ids, m, T, H, I)
    ws_bytes = q4k.q4k_moe_workspace_size(m, T, E, max(H, I), max(H, I))
    ws = _empty(ws_bytes // 4 + 64)
    out = _empty((m * T, H))
    q4k.q4k_expert_ffn_forward(dev(wg), dev(wu), dev(wd), E, dev(x), dev(ids), m, T, H, I, out, ws, ws_bytes)
    rows_close(host(out), ref, what="ffn")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_combine_matches_oracle(mode):
    m, T, H = 5, 3, 520
    rng = np.random.default_rng(mode)
    eo = rng.standard_normal((m * T, H)).astype(np.float32)
    hm = rng.standard_normal((m, H)).astype(np.float32)
    so = rng.standard_normal((m, H)).astype(np.float32)
    w = inputs.routing_weights(mode, m, T)
    g = rng.standard_normal(m).astype(np.float32)
    ref = oracle.moe_combine(hm, eo, w, so if mode else None, g if mode == 1 else None, mode, m, T, H)
    d_hm = dev(hm)
    q4k.moe_combine_residual(d_hm, dev(eo), dev(w), dev(so) if mode else None, dev(g) if mode == 1 else None,
                             mode, m, T, H, d_hm)  # in place: y aliases h_mid
    np.testing.assert_allclose(host(d_hm), ref, rtol=1e-5, atol=1e-5)


def _layer_inputs(W, experts_seed=None):
    seed = W.seed
    ids = inputs.make_ids(seed, W.ids, W.m, W.top_k, W.num_experts)
    used = sorted(set(ids.tolist()))
    wg = oracle_slab(seed, "gate", W.num_experts, W.inter, W.hidden, used)
    wu = oracle_slab(seed, "up", W.num_experts, W.inter, W.hidden, used)
    wd = oracle_slab(seed, "down", W.num_experts, W.hidden, W.inter, used)
    shared = None
    if W.shared_inter:
        shared = (oracle_slab(seed, "sgate", 1, W.shared_inter, W.hidden),
                  oracle_slab(seed, "sup", 1, W.shared_inter, W.hidden),
                  oracle_slab(seed, "sdown", 1, W.hidden, W.shared_inter))
    x = inputs.normal(seed, "h_post", (W.m, W.hidden))
    hm = inputs.normal(seed, "h_mid", (W.m, W.hidden))
    rw = inputs.routing_weights(seed, W.m, W.top_k)
    gl = inputs.normal(seed, "shared_gate", (W.m,))
    return wg, wu, wd, shared, ids, x, hm, rw, gl


def _run_layer_device(W, wg, wu, wd, shared, ids, x, hm, rw, gl):
    sh = W.shared_inter if shared is not None else 0
    ws_bytes = q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, W.num_experts, W.hidden, W.inter, sh)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = _empty((W.m, W.hidden))
    sg, su, sd = (dev(s) for s in shared) if shared is not None else (None, None, None)
    f = err_flag()
    q4k.q4k_moe_layer_forward(dev(wg), dev(wu), dev(wd), W.num_experts, sg, su, sd, sh, W.shared_mode, dev(x),
                              dev(hm), dev(ids), dev(rw), dev(gl), W.m, W.top_k, W.hidden, W.inter, y, ws, ws_bytes, f)
    assert int(host(f)[0]) == 0
    return host(y)


@pytest.mark.parametrize("name", ["qwen3moe_h2048_i768_e128_t8_m1", "qwen3moe_h2048_i768_e128_t8_m16_zipf"])
def test_layer_full_size_qwen3_like(name):
    """The Qwen3-MoE-like layer at its full size (m=1 and m=16 Zipf), in the launch
    configuration the benchmark times, against the oracle's whole layer."""
    from bit_quantized_moe_q4k_gb300.workloads import WORKLOADS
    W = WORKLOADS[name]
    args = _layer_inputs(W)
    wg, wu, wd, shared, ids, x, hm, rw, gl = args
    ref, bad = oracle.moe_layer(wg, wu, wd, W.num_experts, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw, gl,
                                W.m, W.top_k, W.hidden, W.inter)
    got = _run_layer_device(W, *args)
    rows_close(got, ref, what=name)


def test_layer_separate_combine_out_of_range_ids():
    """Beyond 4 tokens the two-launch layer combines in a launch of its own; pairs whose id is out
    of range contribute nothing there too (their rows are zero, and the flag is raised)."""
    from bit_quantized_moe_q4k_gb300.workloads import Workload
    W = Workload("sepcomb", 512, 256, 12, 3, 12, "uniform", 256, 1, 990)  # 36 pairs: two launches
    assert q4k.q4k_moe_layer_path(W.m, W.top_k, W.num_experts, W.hidden, W.inter, W.shared_inter) == \
        q4k.PATH_TWO_LAUNCH
    args = list(_layer_inputs(W))
    ids = args[4].reshape(-1).copy()
    ids[[1, 7, 14]] = [W.num_experts, -2, W.num_experts + 40]
    args[4] = ids
    wg, wu, wd, shared, ids, x, hm, rw, gl = args
    ref, bad = oracle.moe_layer(wg, wu, wd, W.num_experts, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw, gl,
                                W.m, W.top_k, W.hidden, W.inter)
    assert bad == 3
    sh = W.shared_inter
    ws_bytes = q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, W.num_experts, W.hidden, W.inter, sh)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = _empty((W.m, W.hidden))
    f = err_flag()
    q4k.q4k_moe_layer_forward(dev(wg), dev(wu), dev(wd), W.num_experts, *(dev(s) for s in shared), sh, W.shared_mode,
                              dev(x), dev(hm), dev(ids), dev(rw), dev(gl), W.m, W.top_k, W.hidden, W.inter, y, ws,
                              ws_bytes, f)
    assert int(host(f)[0]) == 6  # Q4K_ERR_EXPERT_ID
    rows_close(host(y), ref, what="separate combine, out-of-range ids")


def test_layer_top_k_16():
    """The combine at the top_k limit (16 slots per token), with a sigmoid-gated shared expert."""
    from bit_quantized_moe_q4k_gb300.workloads import Workload
    W = Workload("topk16", 256, 256, 32, 16, 3, "uniform", 256, 1, 950)
    args = _layer_inputs(W)
    wg, wu, wd, shared, ids, x, hm, rw, gl = args
    ref, _ = oracle.moe_layer(wg, wu, wd, W.num_experts, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw, gl,
                              W.m, W.top_k, W.hidden, W.inter)
    rows_close(_run_layer_device(W, *args), ref, what="layer top_k 16")


def test_layer_small_all_shared_modes_and_host_variant():
    from bit_quantized_moe_q4k_gb300.workloads import Workload
    for mode in (0, 1, 2):
        W = Workload("small", 512, 256, 12, 3, 6, "uniform", 0 if mode == 0 else 512, mode, 900 + mode)
        args = _layer_inputs(W)
        wg, wu, wd, shared, ids, x, hm, rw, gl = args
        ref, _ = oracle.moe_layer(wg, wu, wd, W.num_experts, shared, W.shared_inter, W.shared_mode, x, hm, ids, rw,
                                  gl, W.m, W.top_k, W.hidden, W.inter)
        got = _run_layer_device(W, *args)
        rows_close(got, ref, what=f"layer mode {mode}")
        # the host-buffer entry point gives the same bytes
        sh = W.shared_inter
        ws_bytes = (q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, W.num_experts, W.hidden, W.inter, sh)
                    + q4k.q4k_moe_layer_host_staging_size(W.m, W.top_k, W.hidden))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        y = torch.empty((W.m, W.hidden), dtype=torch.float32).pin_memory()
        sg, su, sd = (dev(s) for s in shared) if shared is not None else (None, None, None)
        q4k.q4k_moe_layer_forward_host(dev(wg), dev(wu), dev(wd), W.num_experts, sg, su, sd, sh, mode, pin(x),
                                       pin(hm), pin(ids), pin(rw), pin(gl), W.m, W.top_k, W.hidden, W.inter, y, ws,
                                       ws_bytes)
        torch.cuda.synchronize()
        assert np.array_equal(y.numpy(), got)
        # pageable host buffers take the copy-engine route: the same bytes
        pg = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        y2 = torch.empty((W.m, W.hidden), dtype=torch.float32)
        q4k.q4k_moe_layer_forward_host(dev(wg), dev(wu), dev(wd), W.num_experts, sg, su, sd, sh, mode, pg(x),
                                       pg(hm), pg(ids), pg(rw), pg(gl), W.m, W.top_k, W.hidden, W.inter, y2, ws,
                                       ws_bytes)
        torch.cuda.synchronize()
        assert np.array_equal(y2.numpy(), got)
