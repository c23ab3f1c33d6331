"""GPU parity of the id-GEMV over the MLX-style affine 4-bit and q4tp formats
(q4k_moe_id_gemv_fmt) with the oracle, through the C ABI: both stride walks, the fused
gate|up form, group sizes 32/64/128, the bucketing paths (at most 32 pairs and more), ragged
row tiles, several lane splits, padded expert strides, the pages' expert-blob layout (gate,
up and down of an expert in one blob), and out-of-range ids. Acceptance per output row is
moeflux's tolerance (cosine >= 0.9999, max_abs_diff <= 1e-3 * max|out|).
"""
import numpy as np
import pytest

import oracle
import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import inputs

from helpers import dev, err_flag, fmt4_slab, host, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ABI_FMT = {0: q4k.FMT_AFFINE4, 1: q4k.FMT_Q4TP}


def _silu(v):
    return np.vectorize(oracle.silu)(v)


def _run(fmt, w, w2, off, stride, s_off, b_off, gs, E, a, outer, inner, ids, m, T, n, k):
    out = torch.full((m * T, n), float("nan"), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_moe_id_gemv_fmt(ABI_FMT[fmt], w, w2, off, stride, s_off, b_off, gs, E, dev(a), outer, inner, dev(ids),
                            m, T, n, k, out, f)
    got = host(out)
    return got, int(host(f)[0])


CASES = [
    # (fmt, gs, E, n, k, m, T, pad)
    (0, 64, 8, 64, 256, 1, 2, 0),
    (0, 32, 8, 68, 2048, 3, 4, 16),
    (0, 128, 16, 128, 4096, 5, 8, 0),
    (0, 64, 4, 96, 1024, 40, 2, 32),
    (1, 0, 8, 64, 256, 1, 2, 0),
    (1, 0, 8, 68, 2048, 3, 4, 16),
    (1, 0, 16, 128, 4096, 5, 8, 0),
    (1, 0, 4, 96, 1024, 40, 2, 32),
]


@pytest.mark.parametrize("fmt,gs,E,n,k,m,T,pad", CASES)
def test_fmt4_id_gemv_matches_oracle(fmt, gs, E, n, k, m, T, pad):
    gs_eff = gs or 64
    slab, stride, s_off, b_off = fmt4_slab(900 + m, fmt, E, n, k, gs_eff, pad)
    ids = inputs.ids_uniform_distinct(900 + m, m, T, E)
    x = inputs.normal(900 + m, "x", (m, k))
    wd = dev(slab)
    # gate/up walk: a token's row broadcast to its slots
    got, flag = _run(fmt, wd, None, 0, stride, s_off, b_off, gs_eff, E, x, k, 0, ids, m, T, n, k)
    ref, bad = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs_eff, E, x, k, 0, ids, m, T, n, k)
    assert flag == 0 and bad == 0
    rows_close(got, ref, what="broadcast walk")
    # down walk: one row per pair
    a = inputs.normal(901 + m, "act", (m * T, k))
    got, _ = _run(fmt, wd, None, 0, stride, s_off, b_off, gs_eff, E, a, T * k, k, ids, m, T, n, k)
    ref, _ = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs_eff, E, a, T * k, k, ids, m, T, n, k)
    rows_close(got, ref, what="per-pair walk")


@pytest.mark.parametrize("fmt", [0, 1])
def test_fmt4_fused_gate_up_matches_oracle(fmt):
    E, n, k, m, T, gs = 8, 256, 2048, 4, 4, 64
    wg, stride, s_off, b_off = fmt4_slab(910, fmt, E, n, k, gs, name="gate")
    wu, stride2, _, _ = fmt4_slab(910, fmt, E, n, k, gs, name="up")
    assert stride == stride2
    ids = inputs.ids_uniform_distinct(910, m, T, E)
    x = inputs.normal(910, "x", (m, k))
    got, flag = _run(fmt, dev(wg), dev(wu), 0, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    g, _ = oracle.moe_id_gemv_fmt4(fmt, wg, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    u, _ = oracle.moe_id_gemv_fmt4(fmt, wu, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    assert flag == 0
    rows_close(got, _silu(g) * u, what="fused gate|up")


def test_fmt4_bad_ids_give_zero_rows_and_the_flag():
    fmt, E, n, k, m, T, gs = 0, 4, 64, 512, 3, 2, 32
    slab, stride, s_off, b_off = fmt4_slab(920, fmt, E, n, k, gs)
    ids = np.array([0, 9, 3, -1, 2, 1], np.int32)
    x = inputs.normal(920, "x", (m, k))
    got, flag = _run(fmt, dev(slab), None, 0, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    ref, bad = oracle.moe_id_gemv_fmt4(fmt, slab, stride, s_off, b_off, gs, E, x, k, 0, ids, m, T, n, k)
    assert bad == 2 and flag == 6  # Q4K_ERR_EXPERT_ID
    assert not got[1].any() and not got[3].any()
    rows_close(got, ref, what="bad ids")


def test_fmt4_expert_blob_layout():
    """The pages' affine expert blob: an expert is [gate | up | down], each weights | scales |
    biases; the gate|up call reads gate and up of the chosen experts out of the blobs, the
    down call the down matrices (k = inter)."""
    E, H, I, m, T, gs = 6, 1024, 512, 3, 2, 64
    def block_bytes(n, k):
        return n * k // 2 + 4 * n * (k // gs)
    gate_b, up_b, down_b = block_bytes(I, H), block_bytes(I, H), block_bytes(H, I)
    blob = ((gate_b + up_b + down_b + 15) // 16) * 16
    rng = np.random.default_rng(930)
    slab = rng.integers(0, 256, E * blob, dtype=np.uint8)
    mats = {}
    for name, off, n, k in (("gate", 0, I, H), ("up", gate_b, I, H), ("down", gate_b + up_b, H, I)):
        one, _, s_off, b_off = fmt4_slab(930, 0, E, n, k, gs, name=name)
        mb = oracle.fmt4_matrix_bytes(0, n, k, gs)
        stride_one = len(one) // E
        for e in range(E):
            slab[e * blob + off: e * blob + off + mb] = one[e * stride_one: e * stride_one + mb]
        mats[name] = (off, n, k, s_off, b_off)
    ids = inputs.ids_uniform_distinct(930, m, T, E)
    x = inputs.normal(930, "x", (m, H))
    wd = dev(slab)
    goff, _, _, s_off, b_off = mats["gate"]
    uoff = mats["up"][0]
    base = wd.data_ptr()
    got, flag = _run(0, wd, base + uoff - goff, goff, blob, s_off, b_off, gs, E, x, H, 0, ids, m, T, I, H)
    g, _ = oracle.moe_id_gemv_fmt4(0, slab[goff:], blob, s_off, b_off, gs, E, x, H, 0, ids, m, T, I, H)
    u, _ = oracle.moe_id_gemv_fmt4(0, slab[uoff:], blob, s_off, b_off, gs, E, x, H, 0, ids, m, T, I, H)
    assert flag == 0
    rows_close(got, _silu(g) * u, what="blob gate|up")
    act = (_silu(g) * u).astype(np.float32)
    doff, _, _, ds, db = mats["down"]
    got_d, _ = _run(0, wd, None, doff, blob, ds, db, gs, E, act, T * I, I, ids, m, T, H, I)
    ref_d, _ = oracle.moe_id_gemv_fmt4(0, slab[doff:], blob, ds, db, gs, E, act, T * I, I, ids, m, T, H, I)
    rows_close(got_d, ref_d, what="blob down")


@pytest.mark.parametrize("fmt", [0, 1])
def test_fmt4_qwen3_like_expert_shapes(fmt):
    """Qwen3-like routed experts (128 experts, hidden 2048, expert width 768, top-8) at m = 1
    and m = 16: the gate|up projection in each format."""
    E, n, k, T = 128, 768, 2048, 8
    wg, stride, s_off, b_off = fmt4_slab(940, fmt, E, n, k, 64, name="gate")
    wu, _, _, _ = fmt4_slab(940, fmt, E, n, k, 64, name="up")
    wgd, wud = dev(wg), dev(wu)
    for m in (1, 16):
        ids = inputs.ids_uniform_distinct(940 + m, m, T, E)
        x = inputs.normal(940 + m, "x", (m, k))
        got, flag = _run(fmt, wgd, wud, 0, stride, s_off, b_off, 64, E, x, k, 0, ids, m, T, n, k)
        g, _ = oracle.moe_id_gemv_fmt4(fmt, wg, stride, s_off, b_off, 64, E, x, k, 0, ids, m, T, n, k)
        u, _ = oracle.moe_id_gemv_fmt4(fmt, wu, stride, s_off, b_off, 64, E, x, k, 0, ids, m, T, n, k)
        assert flag == 0
        rows_close(got, _silu(g) * u, what=f"m={m}")
