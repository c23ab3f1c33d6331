"""Pins for the oracle's router, chained RMSNorm and other 4-bit formats.

Each check ties the oracle to something other than itself: numpy's view of bf16 bits, a
dense matmul, closed forms of softmax / sigmoid / RMSNorm, brute force over all expert
subsets, hand-worked golden fixtures (tests/golden/*_handbuilt.json) and invariants of the
id-GEMV walk (batched == per-token, zero rows for bad ids). No GPU is used.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _hexbytes(s):
    return [int(x, 16) for x in s.split()]


def _bf16_bits(x):
    """bf16 bits of float32 values, round to nearest even (input builder, not the method)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------------
# router

def test_bf16_decode_all_patterns_match_numpy_view():
    bits = np.arange(65536, dtype=np.uint16)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    with np.errstate(invalid="ignore"):
        ref = _bf16_values(bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # the page's synthetic scale
    assert oracle.bf16_to_double(0x3C00) == 0.0078125


def test_router_logits_equal_dense_matmul():
    rng = np.random.default_rng(3)
    m, E, H = 3, 16, 96
    x = rng.standard_normal((m, H)).astype(np.float32)
    w = _bf16_bits(rng.standard_normal((E, H)) / math.sqrt(H))
    got = oracle.router_logits(x, w, m, E, H)
    ref = x.astype(np.float64) @ _bf16_values(w).reshape(E, H).T
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_softmax_routing_closed_form():
    """logits ln(1..E): softmax p_e = (e+1)/sum; the top k are the last k, largest first."""
    E, k = 10, 3
    logits = np.log(np.arange(1, E + 1, dtype=np.float64))[None, :]
    ids, w = oracle.route_softmax(logits, k, normalize=False)
    assert ids.tolist() == [[9, 8, 7]]
    np.testing.assert_allclose(w[0], np.array([10, 9, 8]) / 55.0, rtol=1e-14)
    ids, w = oracle.route_softmax(logits, k, normalize=True)
    np.testing.assert_allclose(w[0], np.array([10, 9, 8]) / 27.0, rtol=1e-14)


def test_softmax_routing_ties_go_to_the_lower_id():
    E, k = 12, 4
    ids, w = oracle.route_softmax(np.full((1, E), 0.3), k, normalize=False)
    assert ids.tolist() == [[0, 1, 2, 3]]
    np.testing.assert_allclose(w[0], np.full(k, 1.0 / E), rtol=1e-15)
    ids, w = oracle.route_softmax(np.full((1, E), -2.0), k, normalize=True)
    np.testing.assert_allclose(w[0], np.full(k, 1.0 / k), rtol=1e-15)
    # a tie across the boundary: experts 2 and 5 equal, only one fits
    l = np.array([[5.0, 4.0, 1.0, 0.0, -1.0, 1.0]])
    ids, _ = oracle.route_softmax(l, 3)
    assert ids.tolist() == [[0, 1, 2]]


def test_softmax_routing_brute_force_over_subsets():
    rng = np.random.default_rng(11)
    E, k = 7, 3
    for _ in range(20):
        l = rng.standard_normal((1, E))
        ids, w = oracle.route_softmax(l, k, normalize=False)
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(l[0, list(s)]))
        assert sorted(ids[0].tolist()) == sorted(best)
        assert all(l[0, ids[0, j]] > l[0, ids[0, j + 1]] for j in range(k - 1))
        p = np.exp(l[0]) / np.exp(l[0]).sum()
        np.testing.assert_allclose(w[0], p[ids[0]], rtol=1e-13)
        _, wn = oracle.route_softmax(l, k, normalize=True)
        np.testing.assert_allclose(wn[0], p[ids[0]] / p[ids[0]].sum(), rtol=1e-13)


def test_sigmoid_grouped_routing_handbuilt_case():
    g = _golden("router_noaux_handbuilt.json")
    E = g["num_experts"]
    for tok in g["tokens"]:
        s = np.array(tok["affinities"], np.float64)
        logits = np.log(s / (1.0 - s))[None, :]
        bias = np.array(tok["bias"], np.float32)
        ids, w = oracle.route_sigmoid_grouped(logits, bias, g["top_k"], g["n_group"], g["topk_group"],
                                              normalize=g["normalize"], scale=g["scale"])
        assert ids[0].tolist() == tok["ids"], tok["worked"]
        np.testing.assert_allclose(w[0], tok["weights"], rtol=1e-12)
    assert E == 8


def test_sigmoid_grouped_routing_reduces_to_plain_topk():
    """One group (or one expert per group with topk_group = top_k) is plain top-k on
    sigmoid(l) + bias; brute force over subsets. Unnormalised weights are sigmoid(l)*scale;
    normalised ones sum to scale."""
    rng = np.random.default_rng(5)
    E, k = 8, 3
    for _ in range(10):
        l = rng.standard_normal((1, E))
        bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
        c = 1.0 / (1.0 + np.exp(-l[0])) + bias.astype(np.float64)
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(c[list(s)]))
        for n_group, topk_group in ((1, 1), (E, k)):
            ids, w = oracle.route_sigmoid_grouped(l, bias, k, n_group, topk_group, normalize=False, scale=1.5)
            assert sorted(ids[0].tolist()) == sorted(best)
            assert all(c[ids[0, j]] > c[ids[0, j + 1]] for j in range(k - 1))
            np.testing.assert_allclose(w[0], 1.5 / (1.0 + np.exp(-l[0, ids[0]])), rtol=1e-14)
        _, wn = oracle.route_sigmoid_grouped(l, bias, k, 1, 1, normalize=True, scale=2.5)
        assert abs(wn.sum() - 2.5) < 1e-13


def test_sigmoid_grouped_routing_without_bias_matches_softmax_choice():
    """bias 0 and no group limit: sigmoid is increasing, so the choice is the softmax one."""
    rng = np.random.default_rng(9)
    l = rng.standard_normal((6, 32))
    a, _ = oracle.route_sigmoid_grouped(l, None, 6, 1, 1)
    b, _ = oracle.route_softmax(l, 6)
    assert np.array_equal(a, b)


def test_routing_rejects_bad_arguments():
    l = np.zeros((1, 8))
    with pytest.raises(ValueError):
        oracle.route_softmax(l, 9)
    with pytest.raises(ValueError):
        oracle.route_sigmoid_grouped(l, None, 2, n_group=3, topk_group=1)  # 8 % 3 != 0
    with pytest.raises(ValueError):
        oracle.route_sigmoid_grouped(l, None, 6, n_group=4, topk_group=2)  # 6 > 2 groups of 2 ... per=3 > 2


# ---------------------------------------------------------------------------------------------
# RMSNorm

def test_rms_norm_worked_example():
    x = np.array([[3.0, 4.0]])
    one = np.array([0x3F80, 0x3F80], np.uint16)  # bf16 1.0
    out = oracle.rms_norm(x, one, 0.0)
    r = math.sqrt((9.0 + 16.0) / 2.0)
    np.testing.assert_allclose(out[0], [3.0 / r, 4.0 / r], rtol=1e-15)


def test_rms_norm_closed_forms():
    H, eps = 64, 1e-6
    c = 0.37
    w = np.full(H, 0x4000, np.uint16)  # bf16 2.0
    out = oracle.rms_norm(np.full((1, H), c), w, eps)
    np.testing.assert_allclose(out[0], np.full(H, 2.0 * c / math.sqrt(c * c + eps)), rtol=1e-14)
    # alternating signs, weights that differ per column
    x = np.where(np.arange(H) % 2 == 0, 1.5, -1.5)[None, :]
    wb = _bf16_bits(np.linspace(-1, 1, H))
    out = oracle.rms_norm(x, wb, 0.0)
    np.testing.assert_allclose(out[0], np.sign(x[0]) * _bf16_values(wb), rtol=1e-15)
    # scale invariance with eps 0
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, H))
    np.testing.assert_allclose(oracle.rms_norm(x * 1024.0, wb, 0.0), oracle.rms_norm(x, wb, 0.0), rtol=1e-13)


# ---------------------------------------------------------------------------------------------
# other 4-bit formats

def _affine_fixture():
    g = _golden("affine4_handbuilt.json")
    n, k, gs = g["n"], g["k"], g["gs"]
    codes = [b for row in g["codes_hex"] for b in _hexbytes(row)]
    sc = [int(h, 16) for row in g["scales_bf16_hex"] for h in row.split()]
    bi = [int(h, 16) for row in g["biases_bf16_hex"] for h in row.split()]
    raw = bytearray(codes)
    s_off = len(raw)
    for v in sc:
        raw += bytes([v & 0xFF, v >> 8])
    b_off = len(raw)
    for v in bi:
        raw += bytes([v & 0xFF, v >> 8])
    return g, np.frombuffer(bytes(raw), np.uint8), s_off, b_off


def test_affine4_handbuilt_matrix():
    g, mat, s_off, b_off = _affine_fixture()
    w = oracle.affine4_dequant(mat, s_off, b_off, g["n"], g["k"], g["gs"])
    for key, val in g["expected"].items():
        r, c = (int(v) for v in key.split(","))
        assert w[r, c] == val, key
    # the bf16 fields decode to the listed values
    for r in range(2):
        for j in range(2):
            assert w[r, 32 * j] == g["scales_values"][r][j] * ((32 * j + 5 * r) % 16) + g["biases_values"][r][j]


def test_affine4_page_synthetic_scale():
    """bf16 scale 0x3C00 with bias 0 (the page's synthetic expert data): w = q / 128."""
    n, k, gs = 1, 64, 64
    codes = np.array([(2 * i) % 16 | (((2 * i + 1) % 16) << 4) for i in range(32)], np.uint8)
    mat = np.concatenate([codes, np.array([0x00, 0x3C, 0x00, 0x00], np.uint8)])
    w = oracle.affine4_dequant(mat, 32, 34, n, k, gs)
    assert np.array_equal(w[0], (np.arange(64) % 16) / 128.0)


def test_q4tp_handbuilt_matrix():
    g = _golden("q4tp_handbuilt.json")
    raw = [b for grp in g["group_codes_hex"] for b in _hexbytes(grp)]
    raw += _hexbytes(g["params_hex"]) + _hexbytes(g["scale_codes_hex"])
    mat = np.array(raw, np.uint8)
    assert mat.size == oracle.fmt4_matrix_bytes(oracle.FMT_Q4TP, g["n"], g["k"])
    w = oracle.q4tp_dequant(mat, g["n"], g["k"])
    for key, val in g["expected"].items():
        assert w[0, int(key)] == pytest.approx(val, rel=1e-15), key


def _rand_slab(rng, fmt, E, n, k, gs=64, pad=0):
    """A random slab of E matrices with sane scales: affine scales ~ 1/64, biases ~ -1/8..;
    q4tp base in [-8, -5], step in [0, 1/8]."""
    mb = oracle.fmt4_matrix_bytes(fmt, n, k, gs)
    stride = mb + pad
    slab = np.zeros(E * stride, np.uint8)
    for e in range(E):
        mat = rng.integers(0, 256, mb, dtype=np.uint8)
        if fmt == oracle.FMT_AFFINE:
            ng = n * (k // gs)
            sc = _bf16_bits(rng.uniform(0.005, 0.03, ng)).view(np.uint8)
            bi = _bf16_bits(rng.uniform(-0.15, 0.05, ng)).view(np.uint8)
            mat[n * k // 2: n * k // 2 + 2 * ng] = sc
            mat[n * k // 2 + 2 * ng: n * k // 2 + 4 * ng] = bi
        else:
            gpr = k // 32
            p0 = n * gpr * 16
            base = rng.uniform(-8, -5, n).astype(np.float16)
            step = rng.uniform(0, 0.125, n).astype(np.float16)
            prm = np.stack([base, step], 1).reshape(-1).view(np.uint8)
            mat[p0: p0 + 4 * n] = prm
        slab[e * stride: e * stride + mb] = mat
    return slab, stride


@pytest.mark.parametrize("fmt", [0, 1])
def test_fmt4_id_gemv_is_the_dense_product_of_the_decoded_expert(fmt):
    rng = np.random.default_rng(21 + fmt)
    E, n, k, m, T, gs = 3, 8, 256, 2, 2, 64
    slab, stride = _rand_slab(rng, fmt, E, n, k, gs, pad=16)
    mb = oracle.fmt4_matrix_bytes(fmt, n, k, gs)
    s_off, b_off = n * k // 2, n * k // 2 + 2 * n * (k // gs)
    a = rng.standard_normal((m * T, k)).astype(np.float32)
    ids = np.array([2, 0, 7, 2], np.int32)  # 7 is out of range
    out, bad = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs, E, a, T * k, k, ids, m, T, n, k)
    assert bad == 1
    for p, e in enumerate(ids):
        if e >= E:
            assert not out[p].any()
            continue
        mat = slab[e * stride: e * stride + mb]
        dense = (oracle.affine4_dequant(mat, s_off, b_off, n, k, gs) if fmt == 0 else oracle.q4tp_dequant(mat, n, k))
        np.testing.assert_allclose(out[p], dense @ a[p].astype(np.float64), rtol=1e-12, atol=1e-12)
    # batched == per token, broadcast rows (outer = k, inner = 0)
    x = rng.standard_normal((m, k)).astype(np.float32)
    full, _ = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    for t in range(m):
        one, _ = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs, E, x[t:t + 1], k, 0,
                                         ids[t * T:(t + 1) * T], 1, T, n, k)
        assert np.array_equal(one, full[t * T:(t + 1) * T])
