"""Pins for the CPU oracle: each check ties it to something other than itself.

Closed forms on hand-built blocks, a hand-worked golden scale field, library
routines (numpy's binary16 conversion, dense matmul, Python's sort), the
mathematics of SiLU and sigmoid, round-trip error bounds of the quantizer, and
the batched == per-token invariant of the ferrum-kernels batched id-GEMV tests.
No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from bit_quantized_moe_q4k_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------------
# helpers that build blocks byte by byte (independent of the oracle's quantizer)

def _block(d_bits, dmin_bits, scales12, qs128):
    b = np.zeros(144, np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2], b[3] = dmin_bits & 0xFF, dmin_bits >> 8
    b[4:16] = np.asarray(scales12, np.uint8)
    b[16:144] = np.asarray(qs128, np.uint8)
    return b


ONE = 0x3C00        # binary16 1.0
HALF = 0x3800       # binary16 0.5
QUARTER = 0x3400    # binary16 0.25
# scale field with scale 1 and min 0 for all eight sub-blocks:
# bytes 0..3 hold scales 0..3, bytes 8..11 low nibbles hold scales 4..7
UNIT_SCALES = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]


def _read_golden_scale_field():
    fields = {}
    with open(os.path.join(GOLDEN, "q4k_scale_field_handbuilt.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            key, val = line.split(":", 1)
            fields[key.strip()] = val.split()
    scales = [int(x, 16) for x in fields["scales_hex"]]
    pairs = [tuple(int(v) for v in p.split(",")) for p in fields["pairs"]]
    w15 = [float(x) for x in fields["w_all_codes_15"]]
    w0 = [float(x) for x in fields["w_all_codes_0"]]
    return scales, pairs, w15, w0


# ---------------------------------------------------------------------------------------------
# binary16

def test_half_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.half_to_float(bits)
    ref = bits.view(np.float16).astype(np.float32)
    assert np.array_equal(ours, ref, equal_nan=True)


def test_half_encode_matches_numpy_rne():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(0.02),
        (rng.standard_normal(200000) * 3000).astype(np.float32),
        np.ldexp(rng.random(100000), rng.integers(-30, 17, 100000)).astype(np.float32),
    ])
    # exact halfway cases between neighbouring binary16 values, both parities, normal and subnormal
    h = np.arange(0, 0x7BFF, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                     2.0 ** -25 * 1.0001, 2.0 ** -26, 6.1e-5, np.inf, -np.inf], np.float32)
    for v in (vals, mid, -mid, edge):
        ours = oracle.float_to_half_bits(v)
        with np.errstate(over="ignore"):
            ref = v.astype(np.float16).view(np.uint16)
        assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------------------------
# Q4_K unpack (closed forms on hand-built blocks)

def test_unit_scale_block_reads_codes_in_layout_order():
    # every code byte b holds low nibble b % 16 and high nibble (b + 5) % 16
    qs = [(b % 16) | (((b + 5) % 16) << 4) for b in range(128)]
    blk = _block(ONE, 0, UNIT_SCALES, qs)
    w = oracle.dequant_block(blk)
    # 64-weight group c: weights 64c..64c+31 are the low nibbles of bytes 32c..32c+31,
    # weights 64c+32..64c+63 the high nibbles of the same bytes
    expected = []
    for c in range(4):
        expected += [float((32 * c + i) % 16) for i in range(32)]
        expected += [float((32 * c + i + 5) % 16) for i in range(32)]
    assert w.tolist() == expected
    # spot values worked by hand
    assert (w[0], w[1], w[31], w[32], w[33], w[63], w[64], w[96], w[255]) == (0, 1, 15, 5, 6, 4, 0, 5, 4)


def test_golden_scale_field_pairs_and_weights():
    scales, pairs, w15, w0 = _read_golden_scale_field()
    blk15 = _block(ONE, ONE, scales, [0xFF] * 128)
    blk0 = _block(ONE, ONE, scales, [0x00] * 128)
    for j in range(8):
        assert oracle.scale_min(blk15, j) == pairs[j]
    w = oracle.dequant_block(blk15)
    w_zero = oracle.dequant_block(blk0)
    for j in range(8):
        assert np.all(w[32 * j: 32 * j + 32] == w15[j])
        assert np.all(w_zero[32 * j: 32 * j + 32] == w0[j])


def test_d_and_dmin_scale_the_block():
    scales, pairs, _, _ = _read_golden_scale_field()
    qs = [0x3A] * 128  # low code 10, high code 3
    w = oracle.dequant_block(_block(HALF, QUARTER, scales, qs))
    for j, (sc, mn) in enumerate(pairs):
        q = 10 if j % 2 == 0 else 3
        assert np.all(w[32 * j: 32 * j + 32] == np.float32(0.5 * sc * q - 0.25 * mn))


def test_two_unpackers_agree_bit_for_bit():
    rng = np.random.default_rng(11)
    rows, k = 7, 1024
    w = rng.integers(0, 256, size=(rows, (k // 256) * 144), dtype=np.uint8)
    # sane binary16 d / dmin (random exponents in [-16, 0], positive)
    dd = (rng.random((rows, k // 256, 2)) * 0.5 + 0.5) * np.exp2(rng.integers(-16, 1, (rows, k // 256, 2)))
    bits = dd.astype(np.float16).view(np.uint16)
    blocks = w.reshape(rows, k // 256, 144)
    blocks[:, :, 0] = bits[:, :, 0] & 0xFF
    blocks[:, :, 1] = bits[:, :, 0] >> 8
    blocks[:, :, 2] = bits[:, :, 1] & 0xFF
    blocks[:, :, 3] = bits[:, :, 1] >> 8
    a = oracle.dequant_rows(w, rows, k, elementwise=False)
    b = oracle.dequant_rows(w, rows, k, elementwise=True)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ---------------------------------------------------------------------------------------------
# quantizer

def _fields(block):
    d = float(oracle.half_to_float(np.array([int(block[0]) | (int(block[1]) << 8)], np.uint16))[0])
    dmin = float(oracle.half_to_float(np.array([int(block[2]) | (int(block[3]) << 8)], np.uint16))[0])
    return d, dmin, [oracle.scale_min(block, j) for j in range(8)]


def test_quantizer_round_trip_bound_and_rms():
    x = inputs.normal(1, "pin_q", (64, 2048), 0.02)
    q = oracle.quantize_rows(x)
    w = oracle.dequant_rows(q, 64, 2048)
    blocks = q.reshape(64, 8, 144)
    for r in range(0, 64, 5):
        for b in range(8):
            d, dmin, sm = _fields(blocks[r, b])
            for j, (sc, mn) in enumerate(sm):
                xs = x[r, 256 * b + 32 * j: 256 * b + 32 * j + 32].astype(np.float64)
                ws = w[r, 256 * b + 32 * j: 256 * b + 32 * j + 32].astype(np.float64)
                step, off = d * sc, dmin * mn
                lo, hi = min(0.0, xs.min()), xs.max()
                bound = (0.5 * step + max(0.0, hi + off - 15 * step) + max(0.0, -lo - off)
                         + 1e-6 * max(abs(lo), abs(hi)))
                assert np.all(np.abs(xs - ws) <= bound)
    rel_rms = np.sqrt(np.mean((w.astype(np.float64) - x) ** 2) / np.mean(x.astype(np.float64) ** 2))
    assert 0.05 < rel_rms <= 0.12


def test_quantizer_header_follows_definition():
    x = inputs.normal(2, "pin_q2", (3, 512), 0.02)
    q = oracle.quantize_rows(x).reshape(3, 2, 144)
    for r in range(3):
        for b in range(2):
            xb = x[r, 256 * b: 256 * b + 256].reshape(8, 32)
            lo = np.minimum(0, xb.min(axis=1))
            hi = xb.max(axis=1)
            scale = ((hi - lo).astype(np.float32) / np.float32(15)).astype(np.float32)
            d_exp = np.float16(np.float32(scale.max()) / np.float32(63))
            dmin_exp = np.float16(np.float32((-lo).max()) / np.float32(63))
            d, dmin, sm = _fields(q[r, b])
            assert d == float(d_exp) and dmin == float(dmin_exp)
            for j, (sc, mn) in enumerate(sm):
                assert 0 <= sc <= 63 and 0 <= mn <= 63
                assert sc == min(63, int(np.rint(np.float32(scale[j]) / np.float32(d))))


def test_quantizer_mins_and_codes_follow_definition():
    """Every 6-bit min m_j and every 4-bit code q_i against the definition recomputed with
    numpy float32 (one rounding per step, round-half-even):
    m_j = min(63, rint(mn_j / dmin)) (0 when dmin = 0),
    q_i = clamp(rint((x_i + dmin*m_j) / (d*sc_j)), 0, 15) (0 when d*sc_j = 0).
    Rows include a sub-block of zeros and an all-positive row (dmin = 0)."""
    x = inputs.normal(4, "pin_q3", (5, 768), 0.02)
    x[1, 256:288] = 0.0                                       # one sub-block of zeros
    x[2] = np.abs(x[2]) + np.float32(0.001)                   # nothing below zero: dmin = 0
    q = oracle.quantize_rows(x).reshape(5, 3, 144)
    f32 = np.float32
    for r in range(5):
        for b in range(3):
            d, dmin, sm = _fields(q[r, b])
            codes = np.empty(256, np.int64)
            qs = q[r, b, 16:]
            for c in range(4):
                codes[64 * c: 64 * c + 32] = qs[32 * c: 32 * c + 32] & 0x0F
                codes[64 * c + 32: 64 * c + 64] = qs[32 * c: 32 * c + 32] >> 4
            for j, (sc, mn) in enumerate(sm):
                xs = x[r, 256 * b + 32 * j: 256 * b + 32 * j + 32].astype(f32)
                mn_j = f32(-min(f32(0), xs.min()))
                m_exp = 0 if dmin == 0 else min(63, int(np.rint(f32(mn_j / f32(dmin)))))
                assert mn == m_exp, (r, b, j, mn, m_exp)
                ds = f32(f32(d) * f32(sc))
                dm = f32(f32(dmin) * f32(mn))
                if ds == 0:
                    want = np.zeros(32, np.int64)
                else:
                    want = np.clip(np.rint(((xs + dm).astype(f32) / ds).astype(f32)), 0, 15).astype(np.int64)
                assert np.array_equal(codes[32 * j: 32 * j + 32], want), (r, b, j)


def test_quantizer_special_cases():
    z = np.zeros((1, 256), np.float32)
    assert not oracle.quantize_rows(z).any()  # all fields zero, all weights zero
    pos = np.abs(inputs.normal(3, "pin_pos", (1, 256), 0.02)) + np.float32(0.01)
    qp = oracle.quantize_rows(pos)
    assert qp[0, 2] == 0 and qp[0, 3] == 0  # dmin = 0 when nothing is below zero
    wp = oracle.dequant_rows(qp, 1, 256)
    assert np.all(wp >= 0)
    const = np.full((1, 256), -0.03, np.float32)
    wc = oracle.dequant_rows(oracle.quantize_rows(const), 1, 256)
    assert np.allclose(wc, -0.03, rtol=0.02)


# ---------------------------------------------------------------------------------------------
# id-GEMV

def _slab(seed, E, n, k):
    return np.concatenate([oracle.quantize_rows(inputs.expert_weights(seed, "pin", e, n, k)) for e in range(E)])


def test_gemv_equals_dense_matmul_both_stride_modes():
    E, n, k, m, T = 5, 32, 512, 4, 3
    w = _slab(5, E, n, k)
    W = oracle.dequant_rows(w, E * n, k, elementwise=True).astype(np.float64).reshape(E, n, k)
    ids = inputs.ids_uniform_distinct(5, m, T, E)
    # gate/up: every slot of token t reads row t
    a = inputs.normal(5, "pin_a", (m, k))
    out, bad = oracle.moe_id_gemv(w, E, a, k, 0, ids, m, T, n, k)
    X = np.repeat(a.astype(np.float64), T, axis=0)
    ref = np.stack([W[ids[p]] @ X[p] for p in range(m * T)])
    assert bad == 0 and np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    # down: pair p reads its own row of [m, T, k]
    a2 = inputs.normal(5, "pin_a2", (m, T, k))
    out2, _ = oracle.moe_id_gemv(w, E, a2, T * k, k, ids, m, T, n, k)
    X2 = a2.reshape(m * T, k).astype(np.float64)
    ref2 = np.stack([W[ids[p]] @ X2[p] for p in range(m * T)])
    assert np.allclose(out2, ref2, rtol=1e-12, atol=1e-12)


def test_gemv_factored_form_identity():
    """sum_b sum_j [d*sc_j * sum_i q_i x_i - dmin*m_j * sum_i x_i] equals the dense dot product."""
    k = 768
    w = oracle.quantize_rows(inputs.expert_weights(6, "pin", 0, 3, k))
    x = inputs.normal(6, "pin_x", (k,)).astype(np.float64)
    out, _ = oracle.moe_id_gemv(w, 1, x.astype(np.float32), k, 0, np.zeros(1, np.int32), 1, 1, 3, k)
    for r in range(3):
        acc = 0.0
        for b in range(k // 256):
            blk = w[r, 144 * b: 144 * b + 144]
            d, dmin, sm = _fields(blk)
            codes = np.concatenate([np.concatenate([blk[16 + 32 * c: 48 + 32 * c] & 15,
                                                    blk[16 + 32 * c: 48 + 32 * c] >> 4]) for c in range(4)])
            for j, (sc, mn) in enumerate(sm):
                xs = x[256 * b + 32 * j: 256 * b + 32 * j + 32]
                acc += np.float32(d * sc) * np.dot(codes[32 * j: 32 * j + 32], xs) - np.float32(dmin * mn) * xs.sum()
        assert abs(acc - out[0, r]) <= 1e-9 * max(1.0, abs(acc))


@pytest.mark.parametrize("mode", ["gate_up", "down"])
def test_pages_tiny_case_batched_equals_per_token(mode):
    """The batched walk equals m per-token calls on the ferrum-kernels tiny case (exact in the oracle)."""
    with open(os.path.join(GOLDEN, "ferrum_tiny_case.json")) as f:
        case = json.load(f)
    E, n, k, m, T = case["num_experts"], case["n"], case["k"], case["m"], case["top_k"]
    ids = np.array(case["ids"], np.int32)
    spec = case[mode]
    wp, ap = spec["weight_params"], spec["activation_params"]
    fn = math.sin if mode == "gate_up" else math.cos
    gn = math.cos if mode == "gate_up" else math.sin
    slabs = []
    for e in range(E):
        raw = np.array([wp["amp"] * fn(wp["freq"] * ((i + e * wp["shift"]) % wp["period"])) + wp["bias"]
                        for i in range(n * k)], np.float32).reshape(n, k)
        slabs.append(oracle.quantize_rows(raw))
    w = np.concatenate(slabs)
    rows = m if mode == "gate_up" else m * T
    a = np.array([ap["amp"] * gn(ap["freq"] * i) for i in range(rows * k)], np.float32)
    outer, inner = (k, 0) if mode == "gate_up" else (T * k, k)
    batched, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    per_token = []
    for t in range(m):
        o, _ = oracle.moe_id_gemv(w, E, a[t * outer:], 0, inner, ids[t * T:(t + 1) * T], 1, T, n, k)
        per_token.append(o)
    assert np.array_equal(batched, np.concatenate(per_token))
    assert np.isfinite(batched).all() and np.abs(batched).max() > 0


def test_gemv_out_of_range_ids_zero_rows():
    E, n, k = 3, 8, 256
    w = _slab(8, E, n, k)
    ids = np.array([0, -1, 2, 3, 1, 7], np.int32)
    a = inputs.normal(8, "pin_a", (3, k))
    out, bad = oracle.moe_id_gemv(w, E, a, k, 0, ids, 3, 2, n, k)
    assert bad == 3
    for p in (1, 3, 5):
        assert np.all(out[p] == 0)
    assert np.all(out[[0, 2, 4]] != 0)


def test_gemv_all_ids_equal_is_dense_gemm():
    E, n, k, m = 4, 16, 256, 5
    w = _slab(9, E, n, k)
    W2 = oracle.dequant_rows(w[2 * n:3 * n], n, k).astype(np.float64)
    a = inputs.normal(9, "pin_a", (m, k))
    out, _ = oracle.moe_id_gemv(w, E, a, k, 0, np.full(m, 2, np.int32), m, 1, n, k)
    assert np.allclose(out, a.astype(np.float64) @ W2.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# SwiGLU, FFN, combine, layer

def test_silu_identities():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(1.0) == pytest.approx(0.7310585786300049, abs=1e-16)  # sigmoid(1)
    for x in (0.3, 1.7, 4.0, 11.0):
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, rel=1e-15)  # x*s(x) + x*s(-x) = x
    assert oracle.silu(60.0) == pytest.approx(60.0, rel=1e-15)
    assert abs(oracle.silu(-60.0)) < 1e-24


def _const_rows_slab(values, k):
    """Q4_K rows whose every weight equals an integer value in [0, 15] (d=1, dmin=0, scale 1)."""
    rows = []
    for v in values:
        blk = _block(ONE, 0, UNIT_SCALES, [int(v) | (int(v) << 4)] * 128)
        rows.append(np.tile(blk, k // 256))
    return np.stack(rows)


def test_ffn_closed_form_constant_rows():
    H, I = 512, 256  # both are K of some projection, so multiples of 256
    cg = [(3 * n) % 8 for n in range(I)]
    cu = [(5 * n + 1) % 4 for n in range(I)]
    rd = [(h * 7) % 16 for h in range(H)]
    wg, wu, wd = _const_rows_slab(cg, H), _const_rows_slab(cu, H), _const_rows_slab(rd, I)
    x = inputs.normal(12, "pin_x", (1, H), 0.01)
    sx = float(x.astype(np.float64).sum())
    out, _ = oracle.expert_ffn(wg, wu, wd, 1, x, np.zeros(1, np.int32), 1, 1, H, I)
    act = [(c * sx) / (1 + math.exp(-c * sx)) * (u * sx) for c, u in zip(cg, cu)]
    expected = np.array([r * sum(act) for r in rd])
    assert np.allclose(out[0], expected, rtol=1e-12, atol=1e-15)


def test_ffn_slots_are_independent_experts():
    E, H, I, m, T = 4, 256, 256, 2, 3
    wg, wu, wd = (_slab(s, E, n, k) for s, n, k in ((13, I, H), (14, I, H), (15, H, I)))
    ids = inputs.ids_uniform_distinct(13, m, T, E)
    x = inputs.normal(13, "pin_x", (m, H))
    full, _ = oracle.expert_ffn(wg, wu, wd, E, x, ids, m, T, H, I)
    for p in range(m * T):
        single, _ = oracle.expert_ffn(wg, wu, wd, E, x[p // T:p // T + 1], ids[p:p + 1], 1, 1, H, I)
        assert np.array_equal(full[p], single[0])


def test_combine_special_cases():
    rng = np.random.default_rng(3)
    m, T, H = 3, 2, 16
    eo = rng.standard_normal((m * T, H))
    hm = rng.standard_normal((m, H))
    so = rng.standard_normal((m, H))
    w = rng.random(m * T)
    # identity: top_k = 1, weight 1, no residual, no shared term
    y = oracle.moe_combine(np.zeros((m * T, H)), eo, np.ones(m * T), None, None, 0, m * T, 1, H)
    assert np.array_equal(y, eo)
    # gate logit 0 -> shared weight exactly one half
    y0 = oracle.moe_combine(hm, eo, w, so, np.zeros(m), 1, m, T, H)
    y_none = oracle.moe_combine(hm, eo, w, None, None, 0, m, T, H)
    assert np.allclose(y0 - y_none, 0.5 * so, rtol=0, atol=1e-14)
    # unscaled equals sigmoid with a very large logit
    y_unscaled = oracle.moe_combine(hm, eo, w, so, None, 2, m, T, H)
    y_big = oracle.moe_combine(hm, eo, w, so, np.full(m, 800.0), 1, m, T, H)
    assert np.array_equal(y_unscaled, y_big)
    # closed form of the routed sum for one token
    t = 1
    ref = hm[t] + w[2 * t] * eo[2 * t] + w[2 * t + 1] * eo[2 * t + 1]
    assert np.allclose(y_none[t], ref, rtol=1e-15, atol=1e-15)
    # permuting tokens permutes outputs
    perm = np.array([2, 0, 1])
    pairs = np.concatenate([[2 * p, 2 * p + 1] for p in perm])
    yp = oracle.moe_combine(hm[perm], eo[pairs], w[pairs], so[perm], np.linspace(-1, 1, 3)[perm], 1, m, T, H)
    yr = oracle.moe_combine(hm, eo, w, so, np.linspace(-1, 1, 3), 1, m, T, H)
    assert np.array_equal(yp, yr[perm])


def test_layer_reduces_to_its_parts():
    E, H, I, Is, m, T = 4, 256, 256, 512, 2, 2
    wg, wu, wd = (_slab(s, E, n, k) for s, n, k in ((21, I, H), (22, I, H), (23, H, I)))
    sg, su, sd = (_slab(s, 1, n, k) for s, n, k in ((24, Is, H), (25, Is, H), (26, H, Is)))
    ids = inputs.ids_uniform_distinct(21, m, T, E)
    x = inputs.normal(21, "pin_x", (m, H))
    hm = inputs.normal(21, "pin_hm", (m, H))
    w = inputs.routing_weights(21, m, T)
    gl = inputs.normal(21, "pin_g", (m,))
    y, bad = oracle.moe_layer(wg, wu, wd, E, (sg, su, sd), Is, 1, x, hm, ids, w, gl, m, T, H, I)
    eo, _ = oracle.expert_ffn(wg, wu, wd, E, x, ids, m, T, H, I)
    so, _ = oracle.expert_ffn(sg, su, sd, 1, x, np.zeros(m, np.int32), m, 1, H, Is)
    sig = 1 / (1 + np.exp(-gl.astype(np.float64)))
    ref = hm + (w.reshape(m, T, 1) * eo.reshape(m, T, H)).sum(axis=1) + sig[:, None] * so
    assert bad == 0 and np.allclose(y, ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# bucketing

@pytest.mark.parametrize("P,E", [(1, 1), (6, 4), (128, 128), (512, 256), (1000, 7), (37, 300)])
def test_bucket_matches_library_sort(P, E):
    rng = np.random.default_rng(P * 131 + E)
    ids = rng.integers(-2, E + 2, size=P).astype(np.int32)
    counts, offsets, perm, bad = oracle.bucket(ids, E)
    valid = [p for p in range(P) if 0 <= ids[p] < E]
    ref = sorted(valid, key=lambda p: (int(ids[p]), p)) + [p for p in range(P) if not 0 <= ids[p] < E]
    assert perm.tolist() == ref
    assert bad == P - len(valid)
    assert counts.tolist() == [int((ids == e).sum()) for e in range(E)]
    assert offsets[0] == 0 and offsets[-1] == len(valid)
    assert np.array_equal(np.diff(offsets), counts)
