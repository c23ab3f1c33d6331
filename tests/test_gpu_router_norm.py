"""GPU parity of the router (q4k_moe_router) and the chained RMSNorm (q4k_rms_norm) with the
oracle, through the C ABI.

Tolerances come from the kernels' arithmetic. A logit is an fp32 sum whose rounding depth
is at most d = 8*ceil(hidden/2048) + 16 additions (a thread's fma chain over its chunks, five
shuffle levels, eight warps), so |logit - exact| <= beta = d * 2^-24 * sum_h |w x| (a rigorous
bound for any summation tree of that depth, with margin). The choice is an integer decided
in floating point: where the oracle's scores are farther apart than the bounds allow the
kernel to confuse them, the ids must be equal; elsewhere (a near tie) any choice that the
bounds cannot rule out is valid, and the test checks exactly that. Weights are compared with
a tolerance derived from beta.
"""
import itertools
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


def _case(seed, m, E, H, with_bias=False, with_sg=False):
    x = inputs.normal(seed, "h_post", (m, H))
    w = inputs.bf16_normal(seed, "w_router", (E, H), 1.0 / math.sqrt(H))
    bias = inputs.uniform(seed, "router_bias", (E,), -0.05, 0.05) if with_bias else None
    wsg = inputs.bf16_normal(seed, "w_shared_gate", (H,), 1.0 / math.sqrt(H)) if with_sg else None
    return x, w, bias, wsg


def _run(x, w, bias, wsg, m, E, H, k, scoring, normalize=True, scale=1.0, n_group=1, topk_group=1):
    ids = torch.full((m, k), -7, dtype=torch.int32, device="cuda")
    wt = torch.full((m, k), float("nan"), dtype=torch.float32, device="cuda")
    lg = torch.full((m, E), float("nan"), dtype=torch.float32, device="cuda")
    sg = torch.full((m,), float("nan"), dtype=torch.float32, device="cuda") if wsg is not None else None
    q4k.q4k_moe_router(dev(x), dev(w.view(np.int16)), None if bias is None else dev(bias),
                       None if wsg is None else dev(wsg.view(np.int16)), m, E, H, k, scoring, normalize, scale,
                       n_group, topk_group, ids, wt, lg, sg)
    return host(ids), host(wt), host(lg), (None if sg is None else host(sg))


def _beta(x, w, H):
    """Per (token, expert) bound on the kernel's logit error."""
    d = 8 * math.ceil(H / 2048) + 16
    wv = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return d * U * (np.abs(x.astype(np.float64)) @ np.abs(wv).T) + 1e-30


def _valid_topk(chosen, score, beta, allowed, k):
    """True if `chosen` (in order) is a top-k of score over `allowed` for some perturbation of
    each score within its bound."""
    chosen = list(chosen)
    if len(set(chosen)) != k or not all(allowed[c] for c in chosen):
        return False
    rest = [e for e in range(len(score)) if allowed[e] and e not in chosen]
    for c in chosen:
        for e in rest:
            if score[c] + beta[c] < score[e] - beta[e]:
                return False
    for a, b in zip(chosen, chosen[1:]):
        if score[a] + beta[a] < score[b] - beta[b]:
            return False
    return True


def _decisive(ref_ids, score, beta, allowed, k):
    """The oracle's order is forced by the bounds: every chosen score is farther than the
    bounds from the next one and from every allowed unchosen score."""
    order = list(ref_ids)
    rest = [e for e in range(len(score)) if allowed[e] and e not in order]
    for a, b in zip(order, order[1:]):
        if score[a] - beta[a] <= score[b] + beta[b]:
            return False
    last = order[-1]
    return all(score[last] - beta[last] > score[e] + beta[e] for e in rest)


def _check_softmax(x, w, m, E, H, k, normalize, got_ids, got_w, got_lg):
    ref_lg = oracle.router_logits(x, w, m, E, H)
    beta = _beta(x, w, H)
    assert np.all(np.abs(got_lg - ref_lg) <= beta), float(np.max(np.abs(got_lg - ref_lg) / beta))
    ref_ids, ref_w = oracle.route_softmax(ref_lg, k, normalize)
    exact = 0
    for t in range(m):
        allowed = np.ones(E, bool)
        if _decisive(ref_ids[t], ref_lg[t], beta[t], allowed, k):
            assert got_ids[t].tolist() == ref_ids[t].tolist(), t
            exact += 1
        else:
            assert _valid_topk(got_ids[t], ref_lg[t], beta[t], allowed, k), (t, got_ids[t], ref_ids[t])
        # weights of the kernel's own choice, from the oracle's logits
        l = ref_lg[t]
        p = np.exp(l - l.max())
        p = p[got_ids[t]] / (p[got_ids[t]].sum() if normalize else p.sum())
        tol = 4.0 * beta[t].max() * max(1.0, p.max()) + 8 * E * U
        np.testing.assert_allclose(got_w[t], p, rtol=0, atol=tol)
    return exact


def _check_grouped(x, w, bias, m, E, H, k, n_group, topk_group, normalize, scale, got_ids, got_w, got_lg):
    ref_lg = oracle.router_logits(x, w, m, E, H)
    beta_l = _beta(x, w, H)
    assert np.all(np.abs(got_lg - ref_lg) <= beta_l)
    ref_ids, ref_w = oracle.route_sigmoid_grouped(ref_lg, bias, k, n_group, topk_group, normalize, scale)
    gsize = E // n_group
    per = max(1, k // topk_group)
    exact = 0
    for t in range(m):
        s = 1.0 / (1.0 + np.exp(-ref_lg[t]))
        c = s + (bias.astype(np.float64) if bias is not None else 0.0)
        beta = beta_l[t] / 4.0 + 4 * U  # sigmoid is 1/4-Lipschitz; its rounding and the bias add
        gsc = np.array([np.sort(c[g * gsize:(g + 1) * gsize])[::-1][:per].sum() for g in range(n_group)])
        gbeta = np.array([per * beta[g * gsize:(g + 1) * gsize].max() + per * 2 * U for g in range(n_group)])
        # group sets the bounds cannot rule out: the groups surely kept (fewer than
        # n_group - topk_group groups can reach them, so they beat enough others) plus any choice
        # among the groups that may be kept
        beats_surely = lambda a, b: gsc[a] - gbeta[a] > gsc[b] + gbeta[b]  # noqa: E731
        above = [sum(beats_surely(h, g) for h in range(n_group)) for g in range(n_group)]
        below = [sum(beats_surely(g, h) for h in range(n_group)) for g in range(n_group)]
        sure = [g for g in range(n_group) if below[g] >= n_group - topk_group]
        maybe = [g for g in range(n_group) if g not in sure and above[g] < topk_group]
        gsets = [tuple(sorted(sure + list(c))) for c in itertools.combinations(maybe, topk_group - len(sure))]
        ok_exact = len(gsets) == 1
        allowed_ref = np.zeros(E, bool)
        for g in gsets[0] if ok_exact else []:
            allowed_ref[g * gsize:(g + 1) * gsize] = True
        if ok_exact and _decisive(ref_ids[t], c, beta, allowed_ref, k):
            assert got_ids[t].tolist() == ref_ids[t].tolist(), t
            exact += 1
        else:
            good = False
            for gs in gsets:
                allowed = np.zeros(E, bool)
                for g in gs:
                    allowed[g * gsize:(g + 1) * gsize] = True
                if _valid_topk(got_ids[t], c, beta, allowed, k):
                    good = True
                    break
            assert good, (t, got_ids[t], ref_ids[t])
        sw = s[got_ids[t]]
        want = (sw / sw.sum() if normalize else sw) * scale
        tol = scale * (2.0 * beta.max() + 16 * U) * 4
        np.testing.assert_allclose(got_w[t], want, rtol=0, atol=tol)
    return exact


SOFTMAX_CASES = [
    # (name, m, E, H, k, normalize)
    ("qwen3-like m=1", 1, 128, 2048, 8, True),
    ("qwen3-like m=16", 16, 128, 2048, 8, True),
    ("qwen3-like m=37 (ragged tile)", 37, 128, 2048, 8, False),
    ("mixtral-like m=1", 1, 8, 4096, 2, True),
    ("mixtral-like m=64", 64, 8, 4096, 2, True),
    ("4096 experts", 5, 4096, 256, 16, True),
    ("hidden 16384", 3, 16, 16384, 4, False),
    ("hidden 7168 (ragged chunks)", 9, 64, 7168, 6, True),
]


@pytest.mark.parametrize("name,m,E,H,k,normalize", SOFTMAX_CASES, ids=[c[0] for c in SOFTMAX_CASES])
def test_router_softmax_matches_oracle(name, m, E, H, k, normalize):
    x, w, _, _ = _case(400 + m + E, m, E, H)
    ids, wt, lg, _ = _run(x, w, None, None, m, E, H, k, q4k.ROUTE_SOFTMAX, normalize)
    exact = _check_softmax(x, w, m, E, H, k, normalize, ids, wt, lg)
    assert exact >= m // 2, f"only {exact} of {m} tokens were decisive"


GROUPED_CASES = [
    # (name, m, E, H, k, n_group, topk_group, scale)
    ("deepseek-like m=1", 1, 256, 7168, 8, 8, 4, 2.5),
    ("deepseek-like m=3", 3, 256, 7168, 8, 8, 4, 2.5),
    ("deepseek-like m=64", 64, 256, 7168, 8, 8, 4, 2.5),
    ("no group limit", 11, 64, 1024, 6, 1, 1, 1.0),
    ("32 groups", 4, 512, 512, 16, 32, 8, 1.5),
]


@pytest.mark.parametrize("name,m,E,H,k,ng,tg,scale", GROUPED_CASES, ids=[c[0] for c in GROUPED_CASES])
def test_router_sigmoid_grouped_matches_oracle(name, m, E, H, k, ng, tg, scale):
    x, w, bias, _ = _case(500 + m + E, m, E, H, with_bias=True)
    for normalize in (True, False):
        ids, wt, lg, _ = _run(x, w, bias, None, m, E, H, k, q4k.ROUTE_SIGMOID_GROUPED, normalize, scale, ng, tg)
        exact = _check_grouped(x, w, bias, m, E, H, k, ng, tg, normalize, scale, ids, wt, lg)
        assert exact >= m // 2


def test_router_shared_gate_logit_and_batched_equals_per_token():
    m, E, H, k = 6, 128, 2048, 8
    x, w, _, wsg = _case(610, m, E, H, with_sg=True)
    ids, wt, lg, sg = _run(x, w, None, wsg, m, E, H, k, q4k.ROUTE_SOFTMAX)
    ref = oracle.router_logits(x, wsg[None, :], m, 1, H)[:, 0]
    beta = _beta(x, wsg[None, :], H)[:, 0]
    assert np.all(np.abs(sg - ref) <= beta)
    # a token routed alone gets the same bits as in the batch
    for t in (0, 5):
        i1, w1, l1, s1 = _run(x[t:t + 1], w, None, wsg, 1, E, H, k, q4k.ROUTE_SOFTMAX)
        assert np.array_equal(l1[0], lg[t]) and np.array_equal(i1[0], ids[t])
        assert np.array_equal(w1[0], wt[t]) and s1[0] == sg[t]
    # and every call the same bits
    again = _run(x, w, None, wsg, m, E, H, k, q4k.ROUTE_SOFTMAX)
    for a, b in zip(again, (ids, wt, lg, sg)):
        assert np.array_equal(a, b)


def test_router_ties_go_to_the_lower_id():
    """Every expert's row is the same: the logits are the same bits, so the choice is ids
    0..k-1 (groups 0..topk_group-1 first when grouped) with equal weights."""
    m, E, H, k = 3, 64, 1024, 6
    x = inputs.normal(620, "h_post", (m, H))
    row = inputs.bf16_normal(620, "w_router", (1, H), 1.0 / math.sqrt(H))
    w = np.repeat(row, E, axis=0)
    ids, wt, lg, _ = _run(x, w, None, None, m, E, H, k, q4k.ROUTE_SOFTMAX, True)
    assert (ids == np.arange(k)).all()
    np.testing.assert_allclose(wt, 1.0 / k, rtol=1e-6)
    ids, wt, lg, _ = _run(x, w, None, None, m, E, H, k, q4k.ROUTE_SIGMOID_GROUPED, True, 2.0, 8, 2)
    assert (ids == np.arange(k)).all()
    np.testing.assert_allclose(wt, 2.0 / k, rtol=1e-6)


def test_router_feeds_the_layer():
    """Router -> layer on the device against oracle routing -> oracle layer (Qwen3-like
    shapes, reduced expert width). The router's ids are checked decisive first, so the two
    layers route the same pairs."""
    m, E, H, I, k, SI = 4, 16, 1024, 256, 4, 256
    x, wr, _, wsg = _case(630, m, E, H, with_sg=True)
    h_mid = inputs.normal(630, "h_mid", (m, H))
    wg, wu, wd = (oracle_slab(630, p, E, *(I, H) if p != "down" else (H, I)) for p in ("gate", "up", "down"))
    sgs, sus, sds = (oracle_slab(631, p, 1, *(SI, H) if p != "down" else (H, SI)) for p in ("gate", "up", "down"))
    ids = torch.empty((m, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((m, k), dtype=torch.float32, device="cuda")
    sg = torch.empty((m,), dtype=torch.float32, device="cuda")
    lg = torch.empty((m, E), dtype=torch.float32, device="cuda")
    xd = dev(x)
    q4k.q4k_moe_router(xd, dev(wr.view(np.int16)), None, dev(wsg.view(np.int16)), m, E, H, k, q4k.ROUTE_SOFTMAX,
                       True, 1.0, 1, 1, ids, wt, lg, sg)
    y = torch.empty((m, H), dtype=torch.float32, device="cuda")
    nbytes = q4k.q4k_moe_layer_workspace_size(m, k, E, H, I, SI)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward(dev(wg), dev(wu), dev(wd), E, dev(sgs), dev(sus), dev(sds), SI, q4k.SHARED_SIGMOID, xd,
                              dev(h_mid), ids, wt, sg, m, k, H, I, y, ws, nbytes, f)
    got = host(y)
    assert int(host(f)[0]) == 0
    ref_lg = oracle.router_logits(x, wr, m, E, H)
    ref_ids, ref_w = oracle.route_softmax(ref_lg, k, True)
    beta = _beta(x, wr, H)
    for t in range(m):
        assert _decisive(ref_ids[t], ref_lg[t], beta[t], np.ones(E, bool), k)
    assert np.array_equal(host(ids), ref_ids)
    ref_sg = oracle.router_logits(x, wsg[None, :], m, 1, H)[:, 0]
    ref_y, bad = oracle.moe_layer(wg, wu, wd, E, (sgs, sus, sds), SI, q4k.SHARED_SIGMOID, x, h_mid,
                                  ref_ids.reshape(-1), ref_w.reshape(-1).astype(np.float32),
                                  ref_sg.astype(np.float32), m, k, H, I)
    assert bad == 0
    rows_close(got, ref_y, what="router -> layer")


# ---------------------------------------------------------------------------------------------
# RMSNorm

def _norm_tol(x):
    """fp32 sum of squares of depth <= hidden/1024 + 13, the IEEE sqrt and division, and two
    products per element: a relative error below (depth + 8) * 2^-24 (with margin x2)."""
    H = x.shape[1]
    return 2 * (H // 1024 + 13 + 8) * U


@pytest.mark.parametrize("m,H", [(1, 2048), (7, 4096), (64, 7168), (3, 260)])
def test_rms_norm_matches_oracle(m, H):
    x = inputs.normal(700 + m, "y", (m, H)) * np.float32(3.0)
    w = inputs.bf16_normal(700 + m, "w_norm", (H,), 0.1, 1.0)
    out = torch.empty((m, H), dtype=torch.float32, device="cuda")
    q4k.q4k_rms_norm(dev(x), dev(w.view(np.int16)), m, H, 1e-6, out)
    got = host(out)
    ref = oracle.rms_norm(x.astype(np.float64), w, 1e-6)
    np.testing.assert_allclose(got, ref, rtol=_norm_tol(x), atol=1e-30)
    # in place
    xd = dev(x)
    q4k.q4k_rms_norm(xd, dev(w.view(np.int16)), m, H, 1e-6, xd)
    assert np.array_equal(host(xd), got)


def test_layer_then_rms_norm_matches_oracle():
    """The chain the page appends after the combine: layer output -> next layer's input norm."""
    m, E, H, I, k = 3, 8, 512, 256, 2
    x = inputs.normal(710, "h_post", (m, H))
    h_mid = inputs.normal(710, "h_mid", (m, H))
    ids = inputs.ids_uniform_distinct(710, m, k, E)
    rw = inputs.routing_weights(710, m, k)
    wg, wu, wd = (oracle_slab(710, p, E, *(I, H) if p != "down" else (H, I)) for p in ("gate", "up", "down"))
    wn = inputs.bf16_normal(710, "w_norm", (H,), 0.1, 1.0)
    y = torch.empty((m, H), dtype=torch.float32, device="cuda")
    nbytes = q4k.q4k_moe_layer_workspace_size(m, k, E, H, I, 0)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward(dev(wg), dev(wu), dev(wd), E, None, None, None, 0, q4k.SHARED_NONE, dev(x), dev(h_mid),
                              dev(ids), dev(rw), None, m, k, H, I, y, ws, nbytes, f)
    normed = torch.empty_like(y)
    q4k.q4k_rms_norm(y, dev(wn.view(np.int16)), m, H, 1e-5, normed)
    got_y, got = host(y), host(normed)
    assert int(host(f)[0]) == 0
    ref_y, _ = oracle.moe_layer(wg, wu, wd, E, None, 0, 0, x, h_mid, ids, rw, None, m, k, H, I)
    rows_close(got_y, ref_y, what="layer")
    rows_close(got, oracle.rms_norm(ref_y, wn, 1e-5), what="layer -> rms_norm")
    # the norm of the kernel's own layer output, to the norm's own tolerance
    np.testing.assert_allclose(got, oracle.rms_norm(got_y.astype(np.float64), wn, 1e-5), rtol=_norm_tol(got_y))
