"""Host logic of bench.py that the measurement relies on (CPU only): the
kernel-source hash that keeps a committed ncu traffic figure tied to the
kernel it was taken on, and how workload lines pick that figure up."""
import bench


def test_code_only_drops_comments_and_blank_lines_but_not_strings():
    src = 'int a = 1;  // note\n// whole line\n\n  asm("x // y");  // z\nint b;\n'
    assert bench._code_only(src) == 'int a = 1;\n  asm("x // y");\nint b;'


def test_comment_edit_keeps_the_hash_code_edit_changes_it():
    name = "fp4tc_gemv.cuh"
    with open(bench.os.path.join(bench.CSRC, name), encoding="utf-8") as f:
        text = f.read()
    base = bench._code_only(text)
    assert bench._code_only(text.replace("#pragma once", "// an added comment\n#pragma once", 1)) == base
    assert bench._code_only(text.replace("#pragma once", "#pragma once\nint added;", 1)) != base


def test_traffic_table_names_known_workloads_and_captures():
    rows = [ln.split() for ln in open(bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert rows
    for w, h, b, capture in rows:
        assert w in bench.TRAFFIC_SOURCES and len(h) == 12 and int(b) > 0
        assert bench.os.path.exists(bench.os.path.join(bench.ROOT, "profiles", capture)), capture


def test_tensor_core_lines_take_their_workload_figure(monkeypatch):
    figures = {"nvfp4_experts_64of64_2048x4096": 123}
    monkeypatch.setattr(bench, "profiled_traffic", lambda name: figures.get(name))
    out = bench.with_traffic({"nvfp4_experts_64of64_2048x4096_tensor_core": {},
                              "nvfp4_experts_64of64_2048x4096_cuda_core": {}})
    assert out["nvfp4_experts_64of64_2048x4096_tensor_core"] == {"ncu_dram_bytes_per_launch": 123}
    assert out["nvfp4_experts_64of64_2048x4096_cuda_core"] == {}
