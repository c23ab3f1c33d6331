"""Full-size parity for the layers the CPU oracle cannot run whole: DeepSeek-V3-like (m=64,
6.3 GB of slabs) and the Mixtral-like m sweep, in the launch configuration the benchmark
times (the whole layer through q4k_moe_layer_forward with its workspace, so large buckets
take the tensor-core path).

Weights are fp32 N(0, 0.02) drawn per (projection, expert) by a seeded device generator and
quantized on the GPU by q4k_quantize_rows. For sampled tokens (at least 8 per layer; for the
Mixtral-like layers the first and last pair of every 32-pair chunk of every expert, so each
tensor-core chunk is checked), the experts they use are drawn again, copied to the host and
quantized by the oracle: the bytes must be identical to the GPU's. The oracle then runs the
whole layer for those tokens on its own bytes, and the GPU rows (every row tile of hidden)
must meet the per-row acceptance.
"""
import numpy as np
import pytest

import oracle
import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import inputs
from bit_quantized_moe_q4k_gb300.workloads import MIXTRAL_M_SWEEP, PREFILL, WORKLOADS

from helpers import err_flag, host, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PROJ_SEED = {"gate": 1, "up": 2, "down": 3, "sgate": 4, "sup": 5, "sdown": 6}


def _fp32(seed, proj, e, n, k):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed * 1_000_003 + PROJ_SEED[proj] * 100_003 + e)
    return torch.randn(n, k, generator=g, device="cuda", dtype=torch.float32) * 0.02


def _slab(seed, proj, E, n, k):
    nb = (k // 256) * 144
    out = torch.empty(E * n * nb, dtype=torch.uint8, device="cuda")
    for e in range(E):
        q4k.q4k_quantize_rows(_fp32(seed, proj, e, n, k), n, k, out[e * n * nb:])
    return out


def _oracle_bytes(seed, proj, e, n, k, dev_slab):
    x = _fp32(seed, proj, e, n, k).cpu().numpy()
    ref = oracle.quantize_rows(x)
    nb = (k // 256) * 144
    got = dev_slab[e * n * nb:(e + 1) * n * nb].cpu().numpy().reshape(n, nb)
    assert np.array_equal(got, ref), f"{proj} expert {e}: GPU quantizer bytes differ from the oracle's"
    return ref


def _run(W, sample):
    seed = W.seed
    E, H, I, T, m, Is = W.num_experts, W.hidden, W.inter, W.top_k, W.m, W.shared_inter
    wg, wu, wd = _slab(seed, "gate", E, I, H), _slab(seed, "up", E, I, H), _slab(seed, "down", E, H, I)
    sg = su = sd = None
    if Is:
        sg, su, sd = _slab(seed, "sgate", 1, Is, H), _slab(seed, "sup", 1, Is, H), _slab(seed, "sdown", 1, H, Is)
    ids = inputs.make_ids(seed, W.ids, m, T, E)
    x = inputs.normal(seed, "h_post", (m, H))
    hm = inputs.normal(seed, "h_mid", (m, H))
    rw = inputs.routing_weights(seed, m, T)
    gl = inputs.normal(seed, "shared_gate", (m,))
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    nbytes = q4k.q4k_moe_layer_workspace_size(m, T, E, H, I, Is)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = torch.empty((m, H), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward(wg, wu, wd, E, sg, su, sd, Is, W.shared_mode, d(x), d(hm), d(ids), d(rw), d(gl), m, T,
                              H, I, y, ws, nbytes, f)
    got = host(y)
    assert int(host(f)[0]) == 0
    # oracle on the sampled tokens, with its own quantization of the experts they use
    ts = sorted(set(t for t in sample if t < m))
    used = sorted(set(int(e) for t in ts for e in ids[t * T:(t + 1) * T]))
    remap = {e: i for i, e in enumerate(used)}
    og = np.concatenate([_oracle_bytes(seed, "gate", e, I, H, wg) for e in used])
    ou = np.concatenate([_oracle_bytes(seed, "up", e, I, H, wu) for e in used])
    od = np.concatenate([_oracle_bytes(seed, "down", e, H, I, wd) for e in used])
    shared = None
    if Is:
        shared = (_oracle_bytes(seed, "sgate", 0, Is, H, sg), _oracle_bytes(seed, "sup", 0, Is, H, su),
                  _oracle_bytes(seed, "sdown", 0, H, Is, sd))
    sel_pairs = [t * T + s for t in ts for s in range(T)]
    cids = np.array([remap[int(ids[p])] for p in sel_pairs], np.int32)
    ref, _ = oracle.moe_layer(og, ou, od, len(used), shared, Is, W.shared_mode, x[ts], hm[ts], cids, rw[sel_pairs],
                              gl[ts], len(ts), T, H, I)
    rows_close(got[ts], ref, what=f"{W.name} m={m} tokens {ts}")
    assert np.isfinite(got).all()


def _chunk_sample(W, per_chunk=32, extra=8):
    """Tokens that reach every 32-pair chunk of every expert's bucket (the tensor-core path
    splits a bucket into chunks of 32 pairs, in pair order): the first and the last pair of each
    chunk, plus `extra` evenly spaced tokens and the last token."""
    ids = inputs.make_ids(W.seed, W.ids, W.m, W.top_k, W.num_experts)
    toks = set(range(0, W.m, max(1, W.m // extra))) | {W.m - 1}
    for e in range(W.num_experts):
        pairs = np.flatnonzero(ids == e)
        for c0 in range(0, len(pairs), per_chunk):
            chunk = pairs[c0:c0 + per_chunk]
            toks |= {int(chunk[0]) // W.top_k, int(chunk[-1]) // W.top_k}
    return sorted(toks)


def test_fullsize_deepseek_v3_like_m64():
    W = WORKLOADS["deepseekv3_h7168_i2048_e256_t8_m64"]
    _run(W, sample=list(range(0, 64, 7)) + [63])  # 11 tokens


@pytest.mark.parametrize("m", MIXTRAL_M_SWEEP)
def test_fullsize_mixtral_like_sweep(m):
    W = WORKLOADS["mixtral_h4096_i14336_e8_t2"].with_m(m)
    sample = _chunk_sample(W)
    assert len(sample) >= min(8, m)
    _run(W, sample=sample)


def _bucket_ends_sample(W, extra=8):
    """Tokens of the first and the last pair of every expert's bucket, plus `extra` evenly
    spaced tokens and the last token (prefill sizes: the oracle on every chunk would take
    minutes)."""
    ids = inputs.make_ids(W.seed, W.ids, W.m, W.top_k, W.num_experts)
    toks = set(range(0, W.m, max(1, W.m // extra))) | {W.m - 1}
    for e in range(W.num_experts):
        pairs = np.flatnonzero(ids == e)
        if len(pairs):
            toks |= {int(pairs[0]) // W.top_k, int(pairs[-1]) // W.top_k}
    return sorted(toks)


@pytest.mark.parametrize("name,m", PREFILL, ids=[f"{n.split('_')[0]}-m{m}" for n, m in PREFILL])
def test_fullsize_prefill(name, m):
    W = WORKLOADS[name].with_m(m)
    sample = _bucket_ends_sample(W)
    if W.num_experts > 16:  # keep the oracle's share to a few tens of tokens
        sample = sorted(set(sample[::max(1, len(sample) // 24)]) | {m - 1})
    _run(W, sample=sample)
