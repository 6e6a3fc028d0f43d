"""The benchmark's JSON line and its bookkeeping, checked on the CPU.

`bench.py --impl reference` times the float64 oracle on the host cores and
prints the same JSON line as the GPU arm, so its keys can be checked here.
The source hash that keys the recorded DRAM traffic must ignore comments
and whitespace and change with the code."""
import json
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_step_bookkeeping():
    import bench
    ce = bench.CE
    tiles = (ce["V"] + 127) // 128
    assert bench.CE_TILES == tiles
    assert bench.CE_CORE_BYTES_PER_TOKEN == 4 * ce["V"] + 4 * tiles + 12
    mlp = bench.MLP
    assert bench.MLP_FLOPS == 6 * 2.0 * mlp["T"] * mlp["d"] * mlp["F"]
    assert bench.CE_GEMM_FLOPS == 2 * 2.0 * ce["T"] * ce["d"] * ce["V"]


def test_source_hash_ignores_comments(tmp_path):
    import bench
    csrc = os.path.join(ROOT, "backward_tcgen05_tma_gemms_gb300", "csrc")
    copy = tmp_path / "backward_tcgen05_tma_gemms_gb300" / "csrc"
    shutil.copytree(csrc, copy)
    names = bench.GEMM_SOURCES
    root = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        h0 = bench.kernel_source_hash(names)
        f = copy / names[0]
        src = f.read_text()
        f.write_text("// a comment\n" + src.replace("\n", "\n\n", 3) + "\n/* another */\n")
        assert bench.kernel_source_hash(names) == h0
        f.write_text(src + "\nstatic int tps_extra_symbol = 1;\n")
        assert bench.kernel_source_hash(names) != h0
    finally:
        bench.ROOT = root
