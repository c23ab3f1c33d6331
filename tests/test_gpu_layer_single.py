"""GPU: the single-launch layer (one persistent kernel for gate|up + SwiGLU, down and the
combine, routed and shared experts) against the two-launch layer and the oracle.

The single launch sums every output row in the same order as the two-launch layer (the order
all kernels share: each lane's block terms folded left to right, then the lane shuffles), so
the two agree bit for bit; against the oracle the per-row acceptance of helpers.rows_close
applies. Its CTAs hand results to each other as words tagged with the launch; a call whose
previous call on the workspace had the same shapes trusts the tags alone, any other call also
waits for tagged flags. So the tests also run it on a workspace full of garbage, on one
workspace call after call with the same shapes and with changing ones (and replayed from a
CUDA graph), after a call with ids out of range, and with a wait limit so short that the
waits give up (the error flag reports it, and the next call on a cleared workspace is right).
"""
import numpy as np
import pytest

import oracle
import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import inputs
from bit_quantized_moe_q4k_gb300.workloads import WORKLOADS, Workload

from helpers import dev, err_flag, host, oracle_slab, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Q4K_ERR_EXPERT_ID = 6
Q4K_ERR_TIMEOUT = 10


def _inputs(W, ids=None):
    seed = W.seed
    if ids is None:
        ids = inputs.make_ids(seed, W.ids, W.m, W.top_k, W.num_experts)
    used = sorted({int(e) for e in ids.tolist() if 0 <= e < W.num_experts})
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
    return dict(wg=wg, wu=wu, wd=wd, shared=shared, ids=np.asarray(ids, np.int32), x=x, hm=hm, rw=rw, gl=gl)


class Layer:
    """Device copies of one layer's inputs and a call of q4k_moe_layer_forward on them."""

    def __init__(self, W, a):
        self.W, self.a = W, a
        self.d = {k: dev(a[k]) for k in ("wg", "wu", "wd", "ids", "x", "hm", "rw", "gl")}
        self.sh = W.shared_inter if a["shared"] is not None else 0
        self.s = tuple(dev(s) for s in a["shared"]) if a["shared"] is not None else (None, None, None)
        self.y = torch.empty((W.m, W.hidden), dtype=torch.float32, device="cuda")

    def ws_bytes(self):
        W = self.W
        return q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, W.num_experts, W.hidden, W.inter, self.sh)

    def run(self, ws, flag, stream=None):
        W, d = self.W, self.d
        q4k.q4k_moe_layer_forward(d["wg"], d["wu"], d["wd"], W.num_experts, *self.s, self.sh, W.shared_mode, d["x"],
                                  d["hm"], d["ids"], d["rw"], d["gl"], W.m, W.top_k, W.hidden, W.inter, self.y, ws,
                                  ws.numel(), flag, stream)

    def oracle(self):
        W, a = self.W, self.a
        return oracle.moe_layer(a["wg"], a["wu"], a["wd"], W.num_experts, a["shared"], W.shared_inter, W.shared_mode,
                                a["x"], a["hm"], a["ids"], a["rw"], a["gl"], W.m, W.top_k, W.hidden, W.inter)


@pytest.fixture(autouse=True)
def _single_launch_on(monkeypatch):
    """By default the layer call takes the single launch only where each half fits one round of
    resident CTAs; every test here forces it on (and off for the two-launch references)."""
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "1")


def _two_launch(layer, monkeypatch):
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "0")
    ws = torch.empty(layer.ws_bytes(), dtype=torch.uint8, device="cuda")
    f = err_flag()
    layer.run(ws, f)
    y = host(layer.y).copy()
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "1")
    return y, int(host(f)[0])


CASES = [
    # (hidden, inter, experts, top_k, m, ids, shared_inter, shared_mode)
    (2048, 768, 128, 8, 1, "uniform", 768, 1),   # the Qwen3-MoE-like decode layer, full size
    (1024, 512, 128, 8, 4, "uniform", 512, 2),   # 32 pairs: the single launch's limit
    (512, 256, 4, 2, 3, "uniform", 256, 1),      # more pairs than experts: 4-token items
    (256, 512, 32, 16, 2, "uniform", 256, 1),    # top_k at its limit
    (768, 256, 4, 1, 32, "uniform", 512, 2),     # 32 tokens: a 32-pair shared expert
    (1024, 1280, 16, 4, 2, "zipf", 0, 0),        # no shared expert; ragged row tiles
    (4096, 1792, 8, 2, 1, "uniform", 0, 0),      # Mixtral-like shape at reduced inter
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "h{}_i{}_e{}_t{}_m{}_{}_s{}".format(*c[:7]))
def test_single_launch_matches_two_launch_and_oracle(case, monkeypatch):
    H, I, E, T, m, ids_kind, Is, mode = case
    W = Workload("single", H, I, E, T, m, ids_kind, Is, mode, 1200 + sum(case[:5]))
    assert q4k.q4k_moe_layer_launch_count(m, T, E, H, I, Is) == 1
    assert q4k.q4k_moe_layer_path(m, T, E, H, I, Is) in (q4k.PATH_PERSISTENT, q4k.PATH_PERSISTENT_WIDE)
    layer = Layer(W, _inputs(W))
    ref2, f2 = _two_launch(layer, monkeypatch)
    assert f2 == 0
    ws = torch.empty(layer.ws_bytes(), dtype=torch.uint8, device="cuda")
    f = err_flag()
    layer.run(ws, f)
    got = host(layer.y)
    assert int(host(f)[0]) == 0
    assert np.array_equal(got, ref2), "single launch differs from the two-launch layer"
    ref, _ = layer.oracle()
    rows_close(got, ref, what=f"single-launch layer {case}")


def test_single_launch_duplicate_and_out_of_range_ids(monkeypatch):
    """Repeated experts inside a token (buckets of several pairs) and ids outside [0, E):
    the flag is raised and those pairs contribute nothing, as in the two-launch layer."""
    W = Workload("dup", 512, 512, 16, 4, 3, "uniform", 256, 1, 1301)
    ids = np.array([[3, 3, 7, -1], [7, 3, 16, 0], [5, 5, 5, 5]], np.int32).reshape(-1)
    layer = Layer(W, _inputs(W, ids))
    ref2, f2 = _two_launch(layer, monkeypatch)
    assert f2 == Q4K_ERR_EXPERT_ID
    ws = torch.empty(layer.ws_bytes(), dtype=torch.uint8, device="cuda")
    f = err_flag()
    layer.run(ws, f)
    got = host(layer.y)
    assert int(host(f)[0]) == Q4K_ERR_EXPERT_ID
    assert np.array_equal(got, ref2)
    ref, bad = layer.oracle()
    assert bad == 2
    rows_close(got, ref, what="duplicate / out-of-range ids")


WIDE_CASES = [CASES[0],                                      # the Qwen3-like decode layer
              (1024, 512, 64, 8, 1, "uniform", 512, 2),     # k = 1024 / 512: one lane per row
              (1024, 512, 64, 4, 1, "zipf", 0, 0),          # no shared expert
              CASES[2]]                                     # 4-token items: the four-warp kernel


@pytest.mark.parametrize("case", WIDE_CASES, ids=["qwen3_m1", "k1024", "no_shared", "tb4"])
def test_wide_kernel_matches_four_warp_kernel(case, monkeypatch):
    """The 256-thread kernel (one item of each half per CTA, gate and up rows -- or the two
    halves of a down tile -- on separate warps) and the 128-thread kernel give the same bits,
    call after call on one workspace (tags trusted from the second call on) and with an id out
    of range."""
    H, I, E, T, m, ids_kind, Is, mode = case
    W = Workload("wide", H, I, E, T, m, ids_kind, Is, mode, 2100 + sum(case[:5]))
    expect = q4k.PATH_PERSISTENT if case is CASES[2] else q4k.PATH_PERSISTENT_WIDE
    assert q4k.q4k_moe_layer_path(m, T, E, H, I, Is) == expect
    monkeypatch.setenv("Q4K_LAYER_WIDE", "0")
    assert q4k.q4k_moe_layer_path(m, T, E, H, I, Is) == q4k.PATH_PERSISTENT
    monkeypatch.delenv("Q4K_LAYER_WIDE")
    ids = inputs.make_ids(W.seed, W.ids, W.m, W.top_k, W.num_experts).reshape(-1).copy()
    bad_ids = ids.copy()
    bad_ids[-1] = W.num_experts + 1
    for ids_now in (ids, bad_ids):
        layer = Layer(W, _inputs(W, ids_now))
        outs = {}
        for wide in ("1", "0"):
            monkeypatch.setenv("Q4K_LAYER_WIDE", wide)
            ws = torch.empty(layer.ws_bytes(), dtype=torch.uint8, device="cuda")
            got = []
            for _ in range(3):
                f = err_flag()
                layer.y.zero_()
                layer.run(ws, f)
                got.append((host(layer.y).copy(), int(host(f)[0])))
            outs[wide] = got
        for (a, fa), (b, fb) in zip(outs["1"], outs["0"]):
            assert fa == fb
            assert np.array_equal(a, b)
    monkeypatch.delenv("Q4K_LAYER_WIDE")


@pytest.mark.parametrize("fill", ["random", "ones", "zeros"])
def test_single_launch_any_workspace_contents(fill, monkeypatch):
    """The workspace needs no initialisation: whatever it holds, the first call is right."""
    W = Workload("garbage", 1024, 768, 32, 8, 2, "uniform", 768, 1, 1401)
    layer = Layer(W, _inputs(W))
    ref2, _ = _two_launch(layer, monkeypatch)
    nbytes = layer.ws_bytes()
    if fill == "random":
        g = torch.Generator(device="cuda")
        g.manual_seed(77)
        ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    else:
        ws = torch.full((nbytes,), 255 if fill == "ones" else 0, dtype=torch.uint8, device="cuda")
    f = err_flag()
    layer.run(ws, f)
    assert int(host(f)[0]) == 0
    assert np.array_equal(host(layer.y), ref2)


def test_single_launch_chained_calls_and_graph_replays(monkeypatch):
    """One workspace for a sequence of different layers (each call's flags must not be taken
    for the next call's), then the sequence captured once and replayed three times."""
    layers = []
    for i in range(3):
        W = Workload(f"chain{i}", 1024, 512, 64, 8, 1 + i, "uniform", 512, 1 + (i % 2), 1500 + i)
        layers.append(Layer(W, _inputs(W)))
    refs = [_two_launch(L, monkeypatch)[0] for L in layers]
    nbytes = max(L.ws_bytes() for L in layers)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    f = err_flag()
    for rep in range(2):
        for L, ref in zip(layers, refs):
            L.y.zero_()
            L.run(ws, f)
            assert np.array_equal(host(L.y), ref), f"eager pass {rep}"
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for L in layers:
                L.run(ws, f, stream)
    stream.synchronize()
    for rep in range(3):
        for L in layers:
            L.y.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        for L, ref in zip(layers, refs):
            assert np.array_equal(host(L.y), ref), f"graph replay {rep}"
    assert int(host(f)[0]) == 0


def test_single_launch_m_changes_on_one_workspace(monkeypatch):
    """Calls with different token counts share one workspace (sized for the largest)."""
    base = WORKLOADS["qwen3moe_h2048_i768_e128_t8_m1"]
    seq = [base.with_m(1), base.with_m(4), base.with_m(2), base.with_m(1)]
    layers = [Layer(W, _inputs(W)) for W in seq]
    refs = [_two_launch(L, monkeypatch)[0] for L in layers]
    ws = torch.empty(max(L.ws_bytes() for L in layers), dtype=torch.uint8, device="cuda")
    f = err_flag()
    for L, ref in zip(layers, refs):
        L.run(ws, f)
        assert np.array_equal(host(L.y), ref), f"m = {L.W.m}"
    assert int(host(f)[0]) == 0


def test_single_launch_hidden_changes_on_one_workspace(monkeypatch):
    """Layers of different hidden sizes share one workspace: the result words move with the
    shapes, so a call whose previous call had other shapes finds no stamp meant for it (it waits
    for the items' flags before reading their words, and leaves a stamp for the next call)."""
    seq = [Workload("h1", 1024, 512, 64, 8, 1, "uniform", 512, 1, 1701),
           Workload("h2", 2048, 512, 64, 8, 1, "uniform", 512, 2, 1702)]
    layers = [Layer(W, _inputs(W)) for W in seq]
    refs = [_two_launch(L, monkeypatch)[0] for L in layers]
    ws = torch.empty(max(L.ws_bytes() for L in layers), dtype=torch.uint8, device="cuda")
    f = err_flag()
    for L, ref in [(layers[i % 2], refs[i % 2]) for i in range(5)]:
        L.y.zero_()
        L.run(ws, f)
        assert np.array_equal(host(L.y), ref), L.W.name
    assert int(host(f)[0]) == 0


@pytest.mark.parametrize("wide", ["1", "0"])
def test_single_launch_wait_limit_runs_out(wide, monkeypatch):
    """A wait limit of 1 ns (Q4K_WAIT_NS) makes the waits give up: the kernel returns with
    Q4K_ERR_TIMEOUT in the device flag after its bulk copies have landed (no fault, no hang, the
    context stays usable), and the next call on a cleared workspace with the default limit is
    right. (Below a millisecond the mbarrier waits poll without suspending, so the first copy
    that has not landed yet makes its wait give up.)"""
    monkeypatch.setenv("Q4K_LAYER_WIDE", wide)
    W = WORKLOADS["qwen3moe_h2048_i768_e128_t8_m1"]
    layer = Layer(W, _inputs(W))
    ref2, _ = _two_launch(layer, monkeypatch)
    assert q4k.q4k_moe_layer_path(W.m, W.top_k, W.num_experts, W.hidden, W.inter, W.shared_inter) == \
        (q4k.PATH_PERSISTENT_WIDE if wide == "1" else q4k.PATH_PERSISTENT)
    ws = torch.zeros(layer.ws_bytes(), dtype=torch.uint8, device="cuda")
    f = err_flag()
    monkeypatch.setenv("Q4K_WAIT_NS", "1")
    layer.run(ws, f)
    assert int(host(f)[0]) == Q4K_ERR_TIMEOUT
    monkeypatch.delenv("Q4K_WAIT_NS")
    ws.zero_()
    f.zero_()
    layer.y.zero_()
    layer.run(ws, f)
    assert int(host(f)[0]) == 0
    assert np.array_equal(host(layer.y), ref2)
    # the same after a call that left its stamp: the next call trusts the words' tags, and its
    # polls of them give up
    monkeypatch.setenv("Q4K_WAIT_NS", "1")
    layer.run(ws, f)
    assert int(host(f)[0]) == Q4K_ERR_TIMEOUT
    monkeypatch.delenv("Q4K_WAIT_NS")
    ws.zero_()
    f.zero_()
    layer.y.zero_()
    layer.run(ws, f)
    assert int(host(f)[0]) == 0
    assert np.array_equal(host(layer.y), ref2)


def test_single_launch_same_shapes_trust_tags(monkeypatch):
    """Layers of one shape (different ids, weights and inputs) on one workspace that starts full
    of garbage: the first call waits for flags, every later one trusts the tags of the words the
    previous call wrote over. A call with an id out of range writes no words for that pair, so
    the call after it waits for flags again. Every call equals the two-launch layer bit for
    bit, eagerly and replayed from a CUDA graph."""
    W0 = WORKLOADS["qwen3moe_h2048_i768_e128_t8_m1"]
    layers = []
    for i in range(4):
        W = Workload(f"same{i}", W0.hidden, W0.inter, W0.num_experts, W0.top_k, 1, "uniform", W0.shared_inter,
                     W0.shared_mode, 1900 + i)
        ids = None
        if i == 2:  # slot 5 out of range
            ids = inputs.make_ids(W.seed, W.ids, W.m, W.top_k, W.num_experts).reshape(-1).copy()
            ids[5] = W.num_experts + 3
        layers.append(Layer(W, _inputs(W, ids)))
    refs = [_two_launch(L, monkeypatch) for L in layers]
    assert [r[1] for r in refs] == [0, 0, Q4K_ERR_EXPERT_ID, 0]
    g = torch.Generator(device="cuda")
    g.manual_seed(91)
    ws = torch.randint(0, 256, (layers[0].ws_bytes(),), dtype=torch.uint8, device="cuda", generator=g)
    for rep in range(3):
        for L, (ref, flag) in zip(layers, refs):
            f = err_flag()
            L.y.zero_()
            L.run(ws, f)
            assert int(host(f)[0]) == flag
            assert np.array_equal(host(L.y), ref), f"eager pass {rep}, {L.W.name}"
    clean = [layers[i] for i in (0, 1, 3)]
    f = err_flag()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for rep in range(2):
                for L in clean:
                    L.run(ws, f, stream)
    stream.synchronize()
    for rep in range(3):
        for L in clean:
            L.y.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        for L, i in zip(clean, (0, 1, 3)):
            assert np.array_equal(host(L.y), refs[i][0]), f"graph replay {rep}, {L.W.name}"
    assert int(host(f)[0]) == 0
