"""GPU parity of the routed decode block (q4k_moe_layer_forward_routed): router -> layer ->
RMSNorm from the layer input, through the C ABI.

The call runs the router's kernels, the layer and the norm. So the ids, weights, y and normed
output must equal, bit for bit, what q4k_moe_router, q4k_moe_layer_forward and q4k_rms_norm give
one after the other on the same inputs. Every case is also checked end to end against the
oracle: the oracle's routing (decisive under the logit bounds), its layer and its norm.
"""
import math

import numpy as np
import pytest

import oracle
import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import inputs

from helpers import dev, err_flag, host, oracle_slab, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _layer_case(seed, E, H, I, SI, m, with_bias):
    c = {"x": inputs.normal(seed, "h_post", (m, H)), "hm": inputs.normal(seed, "h_mid", (m, H)),
         "wr": inputs.bf16_normal(seed, "w_router", (E, H), 1.0 / math.sqrt(H)),
         "wsg": inputs.bf16_normal(seed, "w_shared_gate", (H,), 1.0 / math.sqrt(H)),
         "wn": inputs.bf16_normal(seed, "w_norm", (H,), 0.1, 1.0),
         "bias": inputs.uniform(seed, "router_bias", (E,), -0.05, 0.05) if with_bias else None}
    c["slabs"] = tuple(oracle_slab(seed, p, E, *((I, H) if p != "down" else (H, I))) for p in ("gate", "up", "down"))
    c["shared"] = (tuple(oracle_slab(seed + 1, p, 1, *((SI, H) if p != "down" else (H, SI)))
                         for p in ("gate", "up", "down")) if SI else None)
    return c


def _beta(x, w, H):
    d = 8 * math.ceil(H / 2048) + 16
    wv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return d * U * (np.abs(x.astype(np.float64)) @ np.abs(wv).T) + 1e-30


def _norm_rtol(H):
    return 2 * (H // 128 + 8 + 8) * U


CASES = [
    # (name, E, H, I, SI, shared_mode, m, top_k, scoring, n_group, topk_group, scale)
    ("softmax, sigmoid-gated shared, m=1", 16, 1024, 256, 256, 1, 1, 4, 0, 1, 1, 1.0),
    ("softmax, sigmoid-gated shared, m=3", 16, 1024, 256, 256, 1, 3, 4, 0, 1, 1, 1.0),
    ("noaux_tc 8 groups keep 4, unscaled shared, m=2", 64, 1024, 256, 512, 2, 2, 8, 1, 8, 4, 2.5),
    ("softmax, no shared expert, m=4", 8, 512, 512, 0, 0, 4, 2, 0, 1, 1, 1.0),
    ("two-launch layer (64 pairs), softmax, sigmoid-gated shared", 16, 1024, 256, 256, 1, 8, 8, 0, 1, 1, 1.0),
]


def _call_routed(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale, norm=True, ws=None):
    d = {k: dev(v) for k, v in (("x", c["x"]), ("hm", c["hm"]))}
    wg, wu, wd = (dev(a) for a in c["slabs"])
    sg_s = [dev(a) for a in c["shared"]] if c["shared"] else [None, None, None]
    y = torch.full((m, H), float("nan"), dtype=torch.float32, device="cuda")
    normed = torch.full((m, H), float("nan"), dtype=torch.float32, device="cuda") if norm else None
    ids = torch.full((m, K), -5, dtype=torch.int32, device="cuda")
    wts = torch.full((m, K), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = q4k.q4k_moe_layer_routed_workspace_size(m, K, E, H, I, SI)
    if ws is None:
        ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda")  # any contents
    f = err_flag()
    q4k.q4k_moe_layer_forward_routed(
        wg, wu, wd, E, sg_s[0], sg_s[1], sg_s[2], SI, mode, d["x"], d["hm"], dev(c["wr"].view(np.int16)),
        None if c["bias"] is None else dev(c["bias"]), dev(c["wsg"].view(np.int16)) if mode else None, scoring, True,
        scale, ng, tg, m, K, H, I, y, dev(c["wn"].view(np.int16)) if norm else None, 1e-6, normed, ids, wts, ws,
        nbytes, f)
    out = {"y": host(y), "ids": host(ids), "w": host(wts), "normed": host(normed) if norm else None}
    assert int(host(f)[0]) == 0
    return out, ws


def _call_separate(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale):
    wg, wu, wd = (dev(a) for a in c["slabs"])
    sg_s = [dev(a) for a in c["shared"]] if c["shared"] else [None, None, None]
    ids = torch.empty((m, K), dtype=torch.int32, device="cuda")
    wts = torch.empty((m, K), dtype=torch.float32, device="cuda")
    lg = torch.empty((m, E), dtype=torch.float32, device="cuda")
    sg = torch.empty((m,), dtype=torch.float32, device="cuda") if mode else None
    xd = dev(c["x"])
    q4k.q4k_moe_router(xd, dev(c["wr"].view(np.int16)), None if c["bias"] is None else dev(c["bias"]),
                       dev(c["wsg"].view(np.int16)) if mode else None, m, E, H, K, scoring, True, scale, ng, tg, ids,
                       wts, lg, sg)
    y = torch.empty((m, H), dtype=torch.float32, device="cuda")
    nbytes = q4k.q4k_moe_layer_workspace_size(m, K, E, H, I, SI)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward(wg, wu, wd, E, sg_s[0], sg_s[1], sg_s[2], SI, mode, xd, dev(c["hm"]), ids, wts, sg, m, K,
                              H, I, y, ws, nbytes, f)
    assert int(host(f)[0]) == 0
    return {"y": host(y), "ids": host(ids), "w": host(wts), "lg": host(lg), "sg": None if sg is None else host(sg)}


@pytest.mark.parametrize("name,E,H,I,SI,mode,m,K,scoring,ng,tg,scale", CASES, ids=[c[0] for c in CASES])
def test_routed_layer_matches_separate_calls_and_oracle(name, E, H, I, SI, mode, m, K, scoring, ng, tg, scale):
    c = _layer_case(800 + m + E, E, H, I, SI, m, scoring == q4k.ROUTE_SIGMOID_GROUPED)
    single = q4k.q4k_moe_layer_path(m, K, E, H, I, SI) in (q4k.PATH_PERSISTENT, q4k.PATH_PERSISTENT_WIDE)
    assert single == ("two-launch" not in name)
    got, ws = _call_routed(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale)
    sep = _call_separate(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale)
    assert np.array_equal(got["ids"], sep["ids"]), "choice differs from q4k_moe_router's"
    assert np.array_equal(got["w"], sep["w"]), "weights differ from q4k_moe_router's"
    assert np.array_equal(got["y"], sep["y"]), "y differs from router + q4k_moe_layer_forward"
    # the norm is q4k_rms_norm of the call's own y
    normed = torch.empty((m, H), dtype=torch.float32, device="cuda")
    q4k.q4k_rms_norm(dev(got["y"]), dev(c["wn"].view(np.int16)), m, H, 1e-6, normed)
    assert np.array_equal(got["normed"], host(normed))
    np.testing.assert_allclose(got["normed"], oracle.rms_norm(got["y"].astype(np.float64), c["wn"], 1e-6),
                               rtol=_norm_rtol(H), atol=1e-30)
    # end to end against the oracle, where the oracle's choice is decided by the logit bounds
    ref_lg = oracle.router_logits(c["x"], c["wr"], m, E, H)
    beta = _beta(c["x"], c["wr"], H)
    assert np.all(np.abs(sep["lg"] - ref_lg) <= beta)
    if scoring == q4k.ROUTE_SOFTMAX:
        ref_ids, ref_w = oracle.route_softmax(ref_lg, K, True)
    else:
        ref_ids, ref_w = oracle.route_sigmoid_grouped(ref_lg, c["bias"], K, ng, tg, True, scale)
    same = [t for t in range(m) if got["ids"][t].tolist() == ref_ids[t].tolist()]
    assert len(same) >= max(1, m - 1), f"choices differ from the oracle's on tokens {set(range(m)) - set(same)}"
    ref_sg = oracle.router_logits(c["x"], c["wsg"][None, :], m, 1, H)[:, 0].astype(np.float32) if mode else None
    ref_y, bad = oracle.moe_layer(*c["slabs"], E, c["shared"], SI, mode, c["x"][same], c["hm"][same],
                                  ref_ids[same].reshape(-1), ref_w[same].reshape(-1).astype(np.float32),
                                  None if ref_sg is None else ref_sg[same], len(same), K, H, I)
    assert bad == 0
    rows_close(got["y"][same], ref_y, what=f"{name}: y")
    rows_close(got["normed"][same], oracle.rms_norm(ref_y, c["wn"], 1e-6), what=f"{name}: normed")
    # the same workspace again (tags of the next launch), and a call without the norm
    again, _ = _call_routed(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale, ws=ws)
    for k in ("ids", "w", "y", "normed"):
        assert np.array_equal(again[k], got[k]), k
    plain, _ = _call_routed(c, E, H, I, SI, mode, m, K, scoring, ng, tg, scale, norm=False, ws=ws)
    assert np.array_equal(plain["y"], got["y"])


def test_routed_layer_normed_may_alias_y():
    E, H, I, SI, mode, m, K = 16, 1024, 256, 256, 1, 2, 4
    c = _layer_case(830, E, H, I, SI, m, False)
    got, ws = _call_routed(c, E, H, I, SI, mode, m, K, 0, 1, 1, 1.0)
    wg, wu, wd = (dev(a) for a in c["slabs"])
    sg_s = [dev(a) for a in c["shared"]]
    y = torch.empty((m, H), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward_routed(wg, wu, wd, E, *sg_s, SI, mode, dev(c["x"]), dev(c["hm"]),
                                     dev(c["wr"].view(np.int16)), None, dev(c["wsg"].view(np.int16)), 0, True, 1.0, 1,
                                     1, m, K, H, I, y, dev(c["wn"].view(np.int16)), 1e-6, y, None, None, ws, ws.numel(),
                                     f)
    assert int(host(f)[0]) == 0
    assert np.array_equal(host(y), got["normed"])
