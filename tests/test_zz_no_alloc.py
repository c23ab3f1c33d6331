"""q4k_expert_ffn_forward_noalloc: the FFN entry point that allocates nothing.

It exists for callers that may not call cudaMalloc when they run the layer (a plugin in an
application that owns all device memory, a latency-critical loop, a process with its device
memory reserved up front). Its scratch is the library's static device array, shared by every
call. The tests run calls in a row -- a larger one first, so a later, smaller call would
expose anything the earlier one left behind -- and require each to equal the workspace
entry point bit for bit (the two run the same id-GEMV launches on the same inputs) and to
meet the oracle's per-row acceptance; one case fills the array exactly, the largest size
accepted. The file is named to be collected last.
"""
import numpy as np
import pytest

import oracle
import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import inputs

from helpers import dev, err_flag, host, oracle_slab, rows_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _case(seed, E, H, I, m, T):
    a = {"wg": oracle_slab(seed, "gate", E, I, H), "wu": oracle_slab(seed, "up", E, I, H),
         "wd": oracle_slab(seed, "down", E, H, I), "ids": inputs.ids_uniform_distinct(seed, m, T, E),
         "x": inputs.normal(seed, "h_post", (m, H))}
    return a, [dev(a[k]) for k in ("wg", "wu", "wd", "ids", "x")]


def _with_workspace(args, E, H, I, m, T):
    wg, wu, wd, ids, x = args
    nbytes = q4k.q4k_moe_workspace_size(m, T, E, max(H, I), max(H, I))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((m * T, H), dtype=torch.float32, device="cuda")
    q4k.q4k_expert_ffn_forward(wg, wu, wd, E, x, ids, m, T, H, I, out, ws, nbytes)
    return host(out)


def _no_alloc(args, E, H, I, m, T):
    wg, wu, wd, ids, x = args
    out = torch.full((m * T, H), float("nan"), dtype=torch.float32, device="cuda")
    f = err_flag()
    q4k.q4k_expert_ffn_forward_noalloc(wg, wu, wd, E, x, ids, m, T, H, I, out, f)
    got = host(out)
    assert int(host(f)[0]) == 0
    return got


def _oracle(a, E, H, I, m, T):
    out, bad = oracle.expert_ffn(a["wg"], a["wu"], a["wd"], E, a["x"], a["ids"], m, T, H, I)
    assert bad == 0
    return out


def test_no_alloc_matches_workspace_entry_point_and_oracle_call_after_call():
    # the first call fills 86 KB of the array, the second only 10 KB of it, the third 86 KB again
    shapes = [(16, 1024, 768, 7, 4), (8, 512, 256, 5, 2), (16, 1024, 768, 7, 4)]
    for i, (E, H, I, m, T) in enumerate(shapes):
        a, args = _case(700 + i, E, H, I, m, T)
        got = _no_alloc(args, E, H, I, m, T)
        ref = _with_workspace(args, E, H, I, m, T)
        assert np.array_equal(got, ref), f"no-alloc call {i + 1} differs from the workspace entry point"
        rows_close(got, _oracle(a, E, H, I, m, T), what=f"no-alloc call {i + 1} vs oracle")


def test_no_alloc_fills_the_array_exactly():
    """m*top_k*inter*4 equal to the array's size: the call reaches its last bytes."""
    cap = q4k.q4k_expert_ffn_noalloc_max_scratch_bytes()
    E, H, I, T = 4, 256, 4096, 2
    m = cap // (T * I * 4)
    assert m * T * I * 4 == cap
    a, args = _case(733, E, H, I, m, T)
    got = _no_alloc(args, E, H, I, m, T)
    rows_close(got, _oracle(a, E, H, I, m, T), what="no-alloc call at the array's size")
    # a smaller call right after it still gets its own result
    a2, args2 = _case(734, E, H, 512, 3, T)
    got2 = _no_alloc(args2, E, H, 512, 3, T)
    assert np.array_equal(got2, _with_workspace(args2, E, H, 512, 3, T))


def test_no_alloc_rejects_sizes_beyond_the_static_scratch():
    cap = q4k.q4k_expert_ffn_noalloc_max_scratch_bytes()
    assert cap == 4 << 20
    E, H, I, T = 4, 256, 4096, 2
    m = cap // (T * I * 4) + 1  # one token too many
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(q4k.Q4KError) as ei:
        q4k.q4k_expert_ffn_forward_noalloc(z, z, z, E, out, torch.zeros(1, dtype=torch.int32, device="cuda"), m, T,
                                           H, I, out)
    assert ei.value.status == 9  # Q4K_ERR_LIMIT
