"""Host-side checks of the C ABI (no GPU): the library builds for sm_103a, loads, exports
every entry point include/q4kmoe.h declares, and rejects invalid arguments with the
documented status before anything is enqueued."""
import ctypes
import os
import re

import pytest

import bit_quantized_moe_q4k_gb300 as q4k
from bit_quantized_moe_q4k_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4kmoe.h")

A16 = 1 << 20          # a fake 16-byte-aligned address; never dereferenced by these calls
MISALIGNED = A16 + 4


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b((?:q4k|moe)_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_pages_calls():
    names = declared_functions()
    for required in ("q4k_moe_id_gemv", "q4k_expert_ffn_forward", "moe_combine_residual"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = q4k.load()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_lib.SIGNATURES) >= set(declared_functions())


def _st(fn, *args):
    lib = q4k.load()
    return getattr(lib, fn)(*args)


def gemv(**kw):
    a = dict(w=A16, off=0, E=4, a=A16, outer=256, inner=0, ids=A16, m=3, T=2, n=64, k=256, out=A16, ws=None,
             wsb=0, flag=None, stream=None)
    a.update(kw)
    return _st("q4k_moe_id_gemv", a["w"], a["off"], a["E"], a["a"], a["outer"], a["inner"], a["ids"], a["m"],
               a["T"], a["n"], a["k"], a["out"], a["ws"], a["wsb"], a["flag"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(k=100), 2), (dict(k=0), 2), (dict(n=6), 2), (dict(n=0), 2), (dict(m=-1), 2), (dict(E=0), 2),
    (dict(T=0), 3), (dict(T=17), 3), (dict(E=5000), 9), (dict(k=65536 + 256), 9),
    (dict(w=None), 1), (dict(a=None), 1), (dict(ids=None), 1), (dict(out=None), 1),
    (dict(w=MISALIGNED), 7), (dict(off=8), 7), (dict(a=MISALIGNED), 7), (dict(outer=255), 7), (dict(inner=2), 7),
])
def test_id_gemv_rejects(kw, status):
    assert gemv(**kw) == status
    assert q4k.load().q4k_last_error_string()  # a message is recorded


def test_empty_batch_is_a_no_op_without_device_work():
    assert gemv(m=0) == 0
    assert gemv(off=144 * 16, m=0) == 0


def test_ffn_and_layer_workspace_checks():
    lib = q4k.load()
    need = lib.q4k_moe_workspace_size(3, 2, 4, 512, 512)
    assert need >= 3 * 2 * 512 * 4 and need % 256 == 0
    args = [A16, A16, A16, 4, A16, A16, 3, 2, 512, 512, A16]  # hidden = inter: need is exact
    assert lib.q4k_expert_ffn_forward(*args, None, 0, None, None) == 4
    assert lib.q4k_expert_ffn_forward(*args, A16, need - 1, None, None) == 4
    assert lib.q4k_expert_ffn_forward(*args, A16 + 16, need, None, None) == 4  # not 256-byte aligned
    lw = lib.q4k_moe_layer_workspace_size(1, 8, 128, 2048, 768, 768)
    assert lw >= (8 * 768 + 768 + 8 * 2048 + 2048) * 4
    assert lib.q4k_moe_layer_workspace_size(1, 0, 128, 2048, 768, 768) == 0


def test_layer_rejects_bad_mode_and_missing_shared():
    lib = q4k.load()
    base = [A16, A16, A16, 8]
    tail_args = [A16, A16, A16, A16, A16, 1, 2, 256, 256, A16, None, 0, None, None]
    assert lib.q4k_moe_layer_forward(*base, None, None, None, 256, 3, *tail_args) == 8
    assert lib.q4k_moe_layer_forward(*base, None, None, None, 256, 1, *tail_args) == 1
    assert lib.q4k_moe_layer_forward(*base, A16, A16, A16, 256, 1, A16, A16, A16, A16, None, 1, 2, 256, 256, A16,
                                     None, 0, None, None) == 1  # sigmoid gate without logits


def test_combine_rejects():
    lib = q4k.load()
    ok = [A16, A16, A16, A16, A16]
    assert lib.moe_combine_residual(*ok, 3, 2, 2, 256, A16, None) == 8
    assert lib.moe_combine_residual(*ok, 1, 2, 0, 256, A16, None) == 3
    assert lib.moe_combine_residual(*ok, 1, 2, 2, 258, A16, None) == 2
    assert lib.moe_combine_residual(A16, A16, A16, None, None, 2, 2, 2, 256, A16, None) == 1
    assert lib.moe_combine_residual(*ok, 0, 0, 2, 256, A16, None) == 0  # m == 0


def test_bucket_and_quantize_reject():
    lib = q4k.load()
    assert lib.q4k_moe_bucket(A16, -1, 4, A16, A16, A16, None, None) == 2
    assert lib.q4k_moe_bucket(A16, 4, 0, A16, A16, A16, None, None) == 2
    assert lib.q4k_moe_bucket(A16, 4, 4097, A16, A16, A16, None, None) == 9
    assert lib.q4k_moe_bucket(None, 4, 4, A16, A16, A16, None, None) == 1
    assert lib.q4k_quantize_rows(A16, 4, 300, A16, None) == 2
    assert lib.q4k_quantize_rows(MISALIGNED, 4, 256, A16, None) == 7
    assert lib.q4k_quantize_rows(A16, 0, 256, A16, None) == 0


def fmt4(**kw):
    a = dict(fmt=1, w=A16, w2=None, off=0, stride=1 << 20, so=0, bo=0, gs=64, E=4, a=A16, outer=256, inner=0, ids=A16,
             m=3, T=2, n=64, k=256, out=A16, flag=None)
    a.update(kw)
    return q4k.load().q4k_moe_id_gemv_fmt(a["fmt"], a["w"], a["w2"], a["off"], a["stride"], a["so"], a["bo"], a["gs"],
                                          a["E"], a["a"], a["outer"], a["inner"], a["ids"], a["m"], a["T"], a["n"],
                                          a["k"], a["out"], a["flag"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=0), 8), (dict(fmt=3), 8), (dict(gs=48), 2), (dict(gs=256), 2), (dict(so=2), 7), (dict(bo=6), 7),
    (dict(stride=1000), 2), (dict(stride=16), 2), (dict(fmt=2, stride=64 * 128 + 256 + 64 * 5 - 16), 2),
    (dict(k=100), 2), (dict(n=6), 2), (dict(T=17), 3), (dict(E=5000), 9),
    (dict(w=None), 1), (dict(a=None), 1), (dict(ids=None), 1), (dict(out=None), 1),
    (dict(w=MISALIGNED), 7), (dict(off=8), 7), (dict(w2=MISALIGNED), 7), (dict(a=MISALIGNED), 7), (dict(outer=255), 7),
])
def test_fmt4_id_gemv_rejects(kw, status):
    assert fmt4(**kw) == status
    assert q4k.load().q4k_last_error_string()


def test_fmt4_empty_batch():
    assert fmt4(m=0) == 0
    assert fmt4(m=0, fmt=2, stride=64 * 128 + 256 + 64 * 5 + 16 - (64 * 128 + 256 + 64 * 5) % 16) == 0


def router(**kw):
    a = dict(x=A16, w=A16, bias=None, wsg=None, m=3, E=128, H=2048, k=8, scoring=0, norm=1, scale=1.0, ng=1, tg=1,
             ids=A16, wt=A16, logits=A16, sg=None)
    a.update(kw)
    return q4k.load().q4k_moe_router(a["x"], a["w"], a["bias"], a["wsg"], a["m"], a["E"], a["H"], a["k"], a["scoring"],
                                     a["norm"], a["scale"], a["ng"], a["tg"], a["ids"], a["wt"], a["logits"], a["sg"],
                                     None)


@pytest.mark.parametrize("kw,status", [
    (dict(m=-1), 2), (dict(E=0), 2), (dict(E=4097), 9), (dict(k=0), 3), (dict(k=17), 3), (dict(E=4, k=5), 3),
    (dict(H=12), 2), (dict(H=0), 2), (dict(H=16384 + 8), 9), (dict(scoring=2), 8),
    (dict(scoring=1, ng=3), 2), (dict(scoring=1, ng=64, E=128), 2), (dict(scoring=1, ng=8, tg=9), 2),
    (dict(scoring=1, ng=8, tg=0), 2), (dict(scoring=1, E=16, ng=8, tg=2, k=6), 2),
    (dict(x=None), 1), (dict(w=None), 1), (dict(ids=None), 1), (dict(wt=None), 1), (dict(wsg=A16), 1),
    (dict(logits=None), 1),
    (dict(x=MISALIGNED), 7), (dict(w=MISALIGNED), 7), (dict(wsg=MISALIGNED, sg=A16), 7),
])
def test_router_rejects(kw, status):
    assert router(**kw) == status
    assert q4k.load().q4k_last_error_string()


def test_router_and_norm_empty_batch():
    assert router(m=0) == 0
    assert router(m=0, scoring=1, ng=8, tg=4, E=256, H=7168) == 0
    lib = q4k.load()
    assert lib.q4k_rms_norm(A16, A16, 0, 2048, 1e-6, A16, None) == 0


def test_rms_norm_rejects():
    lib = q4k.load()
    assert lib.q4k_rms_norm(A16, A16, -1, 2048, 1e-6, A16, None) == 2
    assert lib.q4k_rms_norm(A16, A16, 2, 2050, 1e-6, A16, None) == 2
    assert lib.q4k_rms_norm(None, A16, 2, 2048, 1e-6, A16, None) == 1
    assert lib.q4k_rms_norm(MISALIGNED, A16, 2, 2048, 1e-6, A16, None) == 7
    assert lib.q4k_rms_norm(A16, A16 + 2, 2, 2048, 1e-6, A16, None) == 7


def test_binding_raises_with_status_name():
    with pytest.raises(q4k.Q4KError) as ei:
        _lib._check(2)
    assert "Q4K_ERR_SHAPE" in str(ei.value)


def test_layer_launch_count_single_launch_rule(monkeypatch):
    """Q4K_SINGLE_LAUNCH=1: layers with at most 32 routed pairs and no tensor-core bucket run as
    one persistent launch; =0: every layer as gate|up + down (+ tensor-core kernels). Unset: the
    single launch for layers each of whose halves fits one round of resident CTAs (a property of
    the device; a layer of thousands of row tiles never qualifies). The flag words widen the
    workspace wherever the single launch can apply, whatever the switch."""
    lib = q4k.load()
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "1")
    assert lib.q4k_moe_layer_launch_count(1, 8, 128, 2048, 768, 768) == 1   # Qwen3-like decode
    assert lib.q4k_moe_layer_launch_count(4, 8, 128, 2048, 768, 768) == 1   # 32 pairs
    assert lib.q4k_moe_layer_launch_count(5, 8, 128, 2048, 768, 768) == 3   # 40 pairs (+ the combine)
    assert lib.q4k_moe_layer_launch_count(1, 2, 8, 4096, 14336, 0) == 1     # Mixtral-like decode
    assert lib.q4k_moe_layer_launch_count(16, 2, 8, 4096, 14336, 0) == 8    # tensor-core buckets, pre-staged
                                                                             # down rows, combine
    assert lib.q4k_moe_layer_launch_count(4, 2, 8, 4096, 14336, 0) == 1     # one pair per expert: no TC bucket
    assert lib.q4k_moe_layer_launch_count(33, 1, 4, 256, 256, 256) == 3     # a 33-pair shared expert
    with_flags = lib.q4k_moe_layer_workspace_size(1, 8, 128, 2048, 768, 768)
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "0")
    assert lib.q4k_moe_layer_launch_count(1, 8, 128, 2048, 768, 768) == 2
    # the size does not depend on the switch (a workspace stays valid for both paths)
    assert lib.q4k_moe_layer_workspace_size(1, 8, 128, 2048, 768, 768) == with_flags
    monkeypatch.delenv("Q4K_SINGLE_LAUNCH", raising=False)
    assert lib.q4k_moe_layer_launch_count(1, 8, 128, 2048, 768, 768) in (1, 2)
    assert lib.q4k_moe_layer_launch_count(1, 2, 8, 4096, 14336, 0) == 3     # 3584 gate|up row tiles:
                                                                             # gate|up, pre-staging, down
    # the activations and expert outputs, plus the generation word and 1024 start tags
    assert with_flags >= (8 * 768 + 768 + 8 * 2048 + 2048) * 4 + 8 * (1 + 1024)


def test_layer_path_query(monkeypatch):
    """q4k_moe_layer_path names the kernels a layer call runs: the persistent single launch for a
    decode layer, two launches otherwise or when switched off; -1 for invalid sizes."""
    lib = q4k.load()
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "1")
    assert lib.q4k_moe_layer_path(1, 8, 128, 2048, 768, 768) in (q4k.PATH_PERSISTENT, q4k.PATH_PERSISTENT_WIDE)
    assert lib.q4k_moe_layer_path(5, 8, 128, 2048, 768, 768) == q4k.PATH_TWO_LAUNCH  # 40 pairs
    monkeypatch.setenv("Q4K_SINGLE_LAUNCH", "0")
    assert lib.q4k_moe_layer_path(1, 8, 128, 2048, 768, 768) == q4k.PATH_TWO_LAUNCH
    assert lib.q4k_moe_layer_path(0, 8, 128, 2048, 768, 768) == -1
    assert lib.q4k_moe_layer_path(1, 17, 128, 2048, 768, 768) == -1


def test_bench_traffic_record_keys_on_code_lines():
    """The committed DRAM traffic of a kernel is matched to its source by a hash of the code
    lines: whole-line comments and blank lines do not change it, code does."""
    import bench
    src = "int a = 1;  // keep\n\n// a comment\n    // another\nint b = 2;\n"
    assert bench.code_text(src) == bench.code_text("// new header\n" + src + "\n\n")
    assert bench.code_text(src) != bench.code_text(src.replace("int b = 2;", "int b = 3;"))
    assert bench.code_text(src) != bench.code_text(src.replace("// keep", "// changed"))  # code line
    sha = bench.source_sha("layer_kernel")
    assert len(sha) == 16 and sha == bench.source_sha("layer_kernel", read=lambda p: open(
        os.path.join(ROOT, p)).read())


def test_bench_reports_a_raised_flag_of_a_secondary_record():
    """A secondary measurement whose device error flag is raised records the flag's meaning
    instead of stopping the run; a clear flag records nothing."""
    import bench

    class Flag:
        def __init__(self, v):
            self.v = v

        def item(self):
            return self.v

    assert bench.flag_error(Flag(0)) is None
    assert "timeout" in bench.flag_error(Flag(10)) and "10" in bench.flag_error(Flag(10))
    assert "expert id" in bench.flag_error(Flag(6))
    assert "see q4kmoe.h" in bench.flag_error(Flag(42))
