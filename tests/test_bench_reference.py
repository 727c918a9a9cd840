"""bench.py's reference arm on the host: `--impl reference` times the fp64 oracle on the CPU cores
and prints one JSON line with the contract's keys (run here on the tiny workload, which needs no
GPU and a few seconds)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_its_json_line_on_the_host():
    sys.path.insert(0, ROOT)
    import oracle
    oracle.build()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, check=True).stdout
    line = json.loads([ln for ln in out.splitlines() if ln.startswith("{")][-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["dtype"] == "f64" and line["data"] == "synthetic"
    assert "tiny" in line["config"]["workload"] and "f32 inputs" in line["config"]["workload"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_source_hash_follows_code_not_comments(tmp_path, monkeypatch):
    """The key that ties an ncu figure to its kernel: unchanged by edits to comments or layout,
    changed by any edit to the code."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int *p) { p[0] = 1; }  // store\n/* block\n note */\n")
    h0 = bench.src_hash("k.cu")
    src.write_text("// a longer header\n// over two lines\n__global__ void k(int *p) {\n"
                   "    p[0] = 1;\n}\n")
    assert bench.src_hash("k.cu") == h0
    src.write_text("__global__ void k(int *p) { p[0] = 2; }\n")
    assert bench.src_hash("k.cu") != h0
