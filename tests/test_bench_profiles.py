"""bench.py's roofline `traffic` comes from the committed ncu summaries only
while they describe the current kernel: the digest ignores comments and blank
lines and changes with any code edit, and a summary whose digest differs
gives no traffic figure."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_digest_ignores_comments_not_code(tmp_path):
    b = _bench()
    base = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    p = tmp_path / "k.cu"
    p.write_text(base)
    d0 = b.kernel_source_digest(str(p))
    p.write_text("// a header comment\n\nint f(int x) {\n  return x + 1;  // reworded\n}\n")
    assert b.kernel_source_digest(str(p)) == d0
    p.write_text(base.replace("x + 1", "x + 2"))
    assert b.kernel_source_digest(str(p)) != d0


def test_stale_summary_gives_no_traffic(tmp_path, monkeypatch):
    b = _bench()
    root = tmp_path
    (root / "quantized_kv_cache_store_gb300" / "csrc").mkdir(parents=True)
    (root / "profiles").mkdir()
    src = root / "quantized_kv_cache_store_gb300" / "csrc" / "verify_tc.cu"
    src.write_text("int k() { return 1; }\n")
    digest = b.kernel_source_digest(str(src))
    summary = root / "profiles" / "stage1_poc_k8v4_ncu.txt"
    summary.write_text(f"# a capture\nkernel_source_digest = {digest}\ndram_bytes_per_launch = 123\n")
    monkeypatch.setattr(b, "ROOT", str(root))
    assert b.ncu_traffic("stage1", "poc_k8v4") == 123.0
    src.write_text("int k() { return 2; }\n")
    assert b.ncu_traffic("stage1", "poc_k8v4") is None


def test_committed_summaries_parse():
    """Every committed stage-1 summary carries a digest and per-launch DRAM bytes
    close to the algorithmic bytes (each cache byte read once)."""
    b = _bench()
    for wl, alg in (("poc_k8v4", 25690112), ("poc_k3v4_nc", 15728640)):
        path = os.path.join(ROOT, "profiles", f"stage1_{wl}_ncu.txt")
        vals = {}
        for line in open(path):
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
        assert len(vals["kernel_source_digest"]) == 16
        assert 1.0 <= float(vals["dram_bytes_per_launch"]) / alg < 1.05
    assert b.kernel_source_digest(os.path.join(ROOT, "quantized_kv_cache_store_gb300", "csrc", "verify_tc.cu"))
