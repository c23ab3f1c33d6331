"""GPU parity of the tensor-core grouped GEMM (tcgen05) path against the CPU oracle.

Buckets of at least 2 pairs (the threshold these batches get: at least two pairs per expert)
run on the tensor-core path when the caller provides the workspace; without it the same
calls run on the id-GEMV kernel. Both
must meet the per-row acceptance; their results differ in rounding (fp16 activations in the
tensor-core products vs 16-bit fixed point), which shows the tensor-core path did run.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_moe_q4k_gb300 import inputs
import bit_quantized_moe_q4k_gb300 as q4k

from helpers import dev, err_flag, host, oracle_slab, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _ws(nbytes):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda"), nbytes


def _gemv(w, E, a, outer, inner, ids, m, T, n, k, workspace):
    out = torch.empty((m * T, n), dtype=torch.float32, device="cuda")
    f = err_flag()
    if workspace:
        ws, nbytes = _ws(q4k.q4k_moe_workspace_size(m, T, E, n, k))
        q4k.q4k_moe_id_gemv(dev(w), 0, E, dev(a), outer, inner, dev(ids), m, T, n, k, out, ws, nbytes, f)
    else:
        q4k.q4k_moe_id_gemv(dev(w), 0, E, dev(a), outer, inner, dev(ids), m, T, n, k, out, err_flag=f)
    got = host(out)
    assert int(host(f)[0]) == 0
    return got


@pytest.mark.parametrize("mode", ["gate_up", "down"])
# sizes give the path enough work (>= 64 items of 128 rows x 32 tokens) to be chosen
@pytest.mark.parametrize("E,n,k,m,T", [(32, 2048, 512, 48, 4),   # ~6 pairs per expert: small buckets
                                       (4, 2148, 512, 64, 2),    # ~32 pairs per expert, ragged last row tile
                                       (2, 4096, 1024, 40, 2),   # 40 pairs per expert: 2 chunks
                                       (3, 3072, 256, 70, 1),    # one block per row
                                       # 80 pairs per expert (chunks of 32, 32, 16): items of a
                                       # chunk pair, then of one chunk
                                       (2, 2048, 512, 80, 2)])
def test_tc_id_gemv_matches_oracle(mode, E, n, k, m, T):
    seed = 500 + n + k
    w = oracle_slab(seed, "tc", E, n, k)
    ids = inputs.ids_uniform_distinct(seed, m, T, E)
    if mode == "gate_up":
        a = inputs.normal(seed, "a", (m, k))
        outer, inner = k, 0
    else:
        a = inputs.normal(seed, "a", (m, T, k))
        outer, inner = T * k, k
    ref, _ = oracle.moe_id_gemv(w, E, a, outer, inner, ids, m, T, n, k)
    got_tc = _gemv(w, E, a, outer, inner, ids, m, T, n, k, workspace=True)
    got_gemv = _gemv(w, E, a, outer, inner, ids, m, T, n, k, workspace=False)
    rows_close(got_tc, ref, what="tensor-core path")
    rows_close(got_gemv, ref, what="id-gemv path")
    assert not np.array_equal(got_tc, got_gemv), "the tensor-core path did not run"


def test_tc_mixed_bucket_sizes_zipf():
    """Zipf ids: the head experts take the tensor-core path, the tail the id-GEMV kernel."""
    E, n, k, m, T = 16, 4096, 512, 48, 4
    seed = 611
    w = oracle_slab(seed, "tc", E, n, k)
    ids = inputs.ids_zipf_distinct(seed, m, T, E)
    counts = np.bincount(ids, minlength=E)
    assert counts.max() >= 16 and (counts[counts > 0] < 16).any()
    a = inputs.normal(seed, "a", (m, k))
    ref, _ = oracle.moe_id_gemv(w, E, a, k, 0, ids, m, T, n, k)
    rows_close(_gemv(w, E, a, k, 0, ids, m, T, n, k, workspace=True), ref, what="mixed")


def test_tc_ffn_fused_gate_up_matches_oracle():
    E, H, I, m, T = 4, 512, 4096, 40, 2  # gate|up on tensor cores, down (512 rows) on the id-GEMV kernel
    seed = 621
    wg, wu = oracle_slab(seed, "gate", E, I, H), oracle_slab(seed, "up", E, I, H)
    wd = oracle_slab(seed, "down", E, H, I)
    ids = inputs.ids_uniform_distinct(seed, m, T, E)
    x = inputs.normal(seed, "h_post", (m, H))
    ref, _ = oracle.expert_ffn(wg, wu, wd, E, x, ids, m, T, H, I)
    nbytes = q4k.q4k_moe_workspace_size(m, T, E, max(H, I), max(H, I))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((m * T, H), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_expert_ffn_forward(dev(wg), dev(wu), dev(wd), E, dev(x), dev(ids), m, T, H, I, out, ws, nbytes, f)
    got = host(out)
    assert int(host(f)[0]) == 0
    rows_close(got, ref, what="tc ffn")


def test_tc_ffn_fused_gate_up_chunk_pairs_match_oracle():
    """Buckets averaging two or more 32-token chunks: the gate|up GEMM runs items of chunk pairs
    (each block dequantized once for both chunks); 80 pairs per expert make a pair and a lone
    chunk of 16 tokens."""
    E, H, I, m, T = 2, 512, 2048, 80, 2
    seed = 631
    wg, wu = oracle_slab(seed, "gate", E, I, H), oracle_slab(seed, "up", E, I, H)
    wd = oracle_slab(seed, "down", E, H, I)
    ids = inputs.ids_uniform_distinct(seed, m, T, E)
    x = inputs.normal(seed, "h_post", (m, H))
    ref, _ = oracle.expert_ffn(wg, wu, wd, E, x, ids, m, T, H, I)
    nbytes = q4k.q4k_moe_workspace_size(m, T, E, max(H, I), max(H, I))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((m * T, H), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_expert_ffn_forward(dev(wg), dev(wu), dev(wd), E, dev(x), dev(ids), m, T, H, I, out, ws, nbytes, f)
    got = host(out)
    assert int(host(f)[0]) == 0
    rows_close(got, ref, what="tc ffn, chunk pairs")


def test_tc_layer_shared_expert_takes_tensor_cores():
    """m >= 16: the shared expert's bucket holds every token and runs on the tensor-core path."""
    from bit_quantized_moe_q4k_gb300.workloads import Workload
    W = Workload("tc_layer", 512, 256, 32, 2, 48, "uniform", 4096, 2, 631)
    seed = W.seed
    ids = inputs.make_ids(seed, W.ids, W.m, W.top_k, W.num_experts)
    wg = oracle_slab(seed, "gate", W.num_experts, W.inter, W.hidden)
    wu = oracle_slab(seed, "up", W.num_experts, W.inter, W.hidden)
    wd = oracle_slab(seed, "down", W.num_experts, W.hidden, W.inter)
    sh = (oracle_slab(seed, "sgate", 1, W.shared_inter, W.hidden), oracle_slab(seed, "sup", 1, W.shared_inter, W.hidden),
          oracle_slab(seed, "sdown", 1, W.hidden, W.shared_inter))
    x = inputs.normal(seed, "h_post", (W.m, W.hidden))
    hm = inputs.normal(seed, "h_mid", (W.m, W.hidden))
    rw = inputs.routing_weights(seed, W.m, W.top_k)
    ref, _ = oracle.moe_layer(wg, wu, wd, W.num_experts, sh, W.shared_inter, W.shared_mode, x, hm, ids, rw, None,
                              W.m, W.top_k, W.hidden, W.inter)
    nbytes = q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, W.num_experts, W.hidden, W.inter, W.shared_inter)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    y = torch.empty((W.m, W.hidden), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_moe_layer_forward(dev(wg), dev(wu), dev(wd), W.num_experts, dev(sh[0]), dev(sh[1]), dev(sh[2]),
                              W.shared_inter, W.shared_mode, dev(x), dev(hm), dev(ids), dev(rw), None, W.m, W.top_k,
                              W.hidden, W.inter, y, ws, nbytes, f)
    got = host(y)
    assert int(host(f)[0]) == 0
    rows_close(got, ref, what="tc layer")


def test_tc_side_stream_in_graph_matches_eager():
    """The tensor-core kernels of a launch run on a second stream beside the id-GEMV kernel (a
    fork and join on events). Layers with tensor-core buckets and one-pair buckets, called
    eagerly and then captured in one CUDA graph (two layers, twice each) and replayed three
    times: the same bits every time, and no error."""
    from bit_quantized_moe_q4k_gb300.workloads import Workload
    layers = []
    for i, (E, T, m, ids_kind) in enumerate([(32, 4, 24, "zipf"), (64, 8, 16, "zipf")]):
        W = Workload(f"side{i}", 512, 512, E, T, m, ids_kind, 512, 1, 700 + i)
        seed = W.seed
        ids = inputs.make_ids(seed, W.ids, W.m, W.top_k, W.num_experts)
        d = dict(wg=dev(oracle_slab(seed, "gate", E, W.inter, W.hidden)),
                 wu=dev(oracle_slab(seed, "up", E, W.inter, W.hidden)),
                 wd=dev(oracle_slab(seed, "down", E, W.hidden, W.inter)),
                 sg=dev(oracle_slab(seed, "sgate", 1, W.shared_inter, W.hidden)),
                 su=dev(oracle_slab(seed, "sup", 1, W.shared_inter, W.hidden)),
                 sd=dev(oracle_slab(seed, "sdown", 1, W.hidden, W.shared_inter)),
                 x=dev(inputs.normal(seed, "h_post", (W.m, W.hidden))), hm=dev(inputs.normal(seed, "h_mid", (W.m, W.hidden))),
                 ids=dev(ids), rw=dev(inputs.routing_weights(seed, W.m, W.top_k)),
                 gl=dev(inputs.normal(seed, "shared_gate", (W.m,))))
        nbytes = q4k.q4k_moe_layer_workspace_size(W.m, W.top_k, E, W.hidden, W.inter, W.shared_inter)
        d["ws"], d["nb"] = torch.empty(nbytes, dtype=torch.uint8, device="cuda"), nbytes
        d["y"] = torch.empty((W.m, W.hidden), dtype=torch.float32, device="cuda")
        assert q4k.q4k_moe_layer_launch_count(W.m, W.top_k, E, W.hidden, W.inter, W.shared_inter) > 3
        layers.append((W, d))
    f = err_flag()

    def run(W, d, stream=None):
        q4k.q4k_moe_layer_forward(d["wg"], d["wu"], d["wd"], W.num_experts, d["sg"], d["su"], d["sd"], W.shared_inter,
                                  W.shared_mode, d["x"], d["hm"], d["ids"], d["rw"], d["gl"], W.m, W.top_k, W.hidden,
                                  W.inter, d["y"], d["ws"], d["nb"], f, stream)

    refs = []
    for W, d in layers:
        run(W, d)
        refs.append(host(d["y"]).copy())
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for _ in range(2):
                for W, d in layers:
                    run(W, d, stream)
    stream.synchronize()
    for rep in range(3):
        for _, d in layers:
            d["y"].zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        for (W, d), ref in zip(layers, refs):
            assert np.array_equal(host(d["y"]), ref), f"replay {rep}, {W.name}"
    assert int(host(f)[0]) == 0


def test_tc_wait_limit_runs_out(monkeypatch):
    """A wait limit of 1 ns (Q4K_WAIT_NS) makes the tensor-core kernel's pipeline waits give up:
    the roles leave together (abort word), the MMAs already issued and the copies in flight
    finish before tensor memory is freed, Q4K_ERR_TIMEOUT is in the device flag, and the next
    call with the default limit on the same workspace is right (the GPU context stays usable)."""
    E, n, k, m, T = 4, 2148, 512, 64, 2
    seed = 733
    w = oracle_slab(seed, "tc", E, n, k)
    ids = inputs.ids_uniform_distinct(seed, m, T, E)
    a = inputs.normal(seed, "a", (m, k))
    ref, _ = oracle.moe_id_gemv(w, E, a, k, 0, ids, m, T, n, k)
    ws, nbytes = _ws(q4k.q4k_moe_workspace_size(m, T, E, n, k))
    dw, da, dids = dev(w), dev(a), dev(ids)
    out = torch.empty((m * T, n), dtype=torch.float32, device="cuda")
    f = err_flag()
    monkeypatch.setenv("Q4K_WAIT_NS", "1")
    q4k.q4k_moe_id_gemv(dw, 0, E, da, k, 0, dids, m, T, n, k, out, ws, nbytes, f)
    assert int(host(f)[0]) == 10  # Q4K_ERR_TIMEOUT
    monkeypatch.delenv("Q4K_WAIT_NS")
    f.zero_()
    q4k.q4k_moe_id_gemv(dw, 0, E, da, k, 0, dids, m, T, n, k, out, ws, nbytes, f)
    got = host(out)
    assert int(host(f)[0]) == 0
    rows_close(got, ref, what="tensor-core path after a timed-out call")
