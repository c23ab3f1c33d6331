"""Test helpers: acceptance check, slab builders, device plumbing."""
from __future__ import annotations

import numpy as np

import oracle
from bit_quantized_moe_q4k_gb300 import inputs

# Acceptance per output row (moeflux expert_forward.rs, module doc "Tolerance regime"):
# cosine >= 0.9999 and max_abs_diff <= 1e-3 * max_abs_out.
ROW_REL_MAX = 1e-3
ROW_COS_MIN = 0.9999


def rows_close(got, ref, rel=ROW_REL_MAX, cos_min=ROW_COS_MIN, what=""):
    got = np.asarray(got, np.float64).reshape(len(ref), -1)
    ref = np.asarray(ref, np.float64).reshape(len(ref), -1)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    worst = 0.0
    for i in range(ref.shape[0]):
        r, g = ref[i], got[i]
        mx = np.abs(r).max()
        if mx == 0.0:
            assert np.abs(g).max() == 0.0, f"{what}: row {i} should be all zero"
            continue
        d = np.abs(g - r).max() / mx
        cos = float(np.dot(g, r) / (np.linalg.norm(g) * np.linalg.norm(r)))
        assert d <= rel and cos >= cos_min, f"{what}: row {i}: max_abs_diff/max|out| = {d:.3e}, cosine = {cos:.7f}"
        worst = max(worst, d)
    return worst


def oracle_slab(seed, proj, num_experts, n, k, experts=None):
    """Q4_K bytes [num_experts * n, k/256*144] quantized by the oracle from N(0, 0.02) weights.
    Experts outside `experts` (when given) are left zero."""
    nb = (k // 256) * 144
    out = np.zeros((num_experts * n, nb), np.uint8)
    for e in (range(num_experts) if experts is None else experts):
        out[e * n:(e + 1) * n] = oracle.quantize_rows(inputs.expert_weights(seed, proj, e, n, k))
    return out


def dev(x, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def err_flag():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def fmt4_slab(seed, fmt, E, n, k, gs=64, pad=0, name="w"):
    """A seeded slab of E [n, k] matrices in an other 4-bit format (oracle numbering: fmt 0
    MLX-affine, 1 q4tp), laid out as the header documents: random code bytes; affine bf16
    scales U(0.005, 0.03) and biases U(-0.15, 0.05) per group of gs; q4tp binary16 base
    U(-8, -5) and step U(0, 1/8) per row and random 5-bit group codes. Returns
    (slab uint8, expert_stride, scales_offset, biases_offset)."""
    mb = oracle.fmt4_matrix_bytes(fmt, n, k, gs)
    stride = ((mb + 15) // 16) * 16 + pad
    g = np.random.default_rng([seed, fmt, E, n, k, gs, pad, sum(name.encode())])
    slab = g.integers(0, 256, E * stride, dtype=np.uint8)
    s_off = n * k // 2
    b_off = s_off + 2 * n * (k // gs)
    for e in range(E):
        base = e * stride
        if fmt == 0:
            ng = n * (k // gs)
            sc = inputs.to_bf16_bits(g.uniform(0.005, 0.03, ng).astype(np.float32)).view(np.uint8)
            bi = inputs.to_bf16_bits(g.uniform(-0.15, 0.05, ng).astype(np.float32)).view(np.uint8)
            slab[base + s_off: base + s_off + 2 * ng] = sc
            slab[base + b_off: base + b_off + 2 * ng] = bi
        else:
            prm = np.stack([g.uniform(-8, -5, n), g.uniform(0, 0.125, n)], 1).astype(np.float16).reshape(-1)
            slab[base + s_off: base + s_off + 4 * n] = prm.view(np.uint8)
    return slab, stride, s_off, b_off
