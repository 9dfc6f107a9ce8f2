"""The kernel-source hash that decides whether recorded DRAM counters are current:
comments and whitespace do not change it, code does."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    bench = _bench()
    src = tmp_path / "k.cuh"
    src.write_text("int f(int x) {\n  return x + 1;  // one\n}\n/* block */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ("k.cuh",))
    h0 = bench.kernel_sources_hash()
    src.write_text("// header comment\nint f(int x) {\n    return x + 1;  // changed comment\n}\n")
    assert bench.kernel_sources_hash() == h0
    src.write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.kernel_sources_hash() != h0


def test_recorded_traffic_is_used_only_for_the_code_it_was_taken_on(tmp_path, monkeypatch):
    # A DRAM record counts only while the kernel code it was captured on is the
    # current code; otherwise the bench line reports traffic as null.
    import json
    bench = _bench()
    src = tmp_path / "k.cuh"
    src.write_text("int f() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ("k.cuh",))
    (tmp_path / "profiles").mkdir()
    rec = {"attn_fwd_kernel": {"long128k": {"sources_sha256_16": bench.kernel_sources_hash(),
                                            "dram_bytes_per_launch": 123.0}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench._recorded_traffic("long128k") == 123.0
    assert bench._recorded_traffic("self8k") is None
    src.write_text("int f() { return 2; }\n")
    assert bench._recorded_traffic("long128k") is None
