"""Host-side pieces of the benchmark that need no GPU: the key of the ncu traffic table (the kernel
sources with comments removed) and the lookup of a workload's entry."""
import importlib.util
import os
import shutil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join("routed_expert_layer_moe_gb300", "csrc")


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def copy_sources(dst):
    os.makedirs(os.path.join(dst, CSRC))
    for n in ("gemm_tc.cu", "common.cuh"):
        shutil.copy(os.path.join(ROOT, CSRC, n), os.path.join(dst, CSRC, n))
    return os.path.join(dst, CSRC, "gemm_tc.cu")


def test_source_hash_ignores_comments_but_not_code(tmp_path):
    bench = load_bench()
    ref = bench.src_hash("gemm_tc.cu", "common.cuh")
    bench.ROOT = str(tmp_path / "a")
    g = copy_sources(bench.ROOT)
    assert bench.src_hash("gemm_tc.cu", "common.cuh") == ref
    src = open(g).read()
    open(g, "w").write("// a new comment line\n/* and a block\n   comment */\n" + src.replace("\n", "\n\n", 3))
    assert bench.src_hash("gemm_tc.cu", "common.cuh") == ref
    bench.ROOT = str(tmp_path / "b")
    g = copy_sources(bench.ROOT)
    src = open(g).read()
    i = src.index("constexpr int BM = 128;")
    open(g, "w").write(src[:i] + "constexpr int BM = 64;" + src[i + len("constexpr int BM = 128;"):])
    assert bench.src_hash("gemm_tc.cu", "common.cuh") != ref


def test_traffic_entries_are_keyed_by_workload_form_and_hash():
    bench = load_bench()
    for key, value in bench.TRAFFIC.items():
        workload, form, h = key.split(":")
        assert workload in bench.mi.CONFIGS and form in ("split", "ffn") and len(h) == 16
        assert isinstance(value, int) and value > 0
