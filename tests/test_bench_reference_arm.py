"""bench.py's reference arm (the fp64 oracle on the host cores) runs without a
GPU and prints one JSON line with the fields the benchmark contract names."""
import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parent.parent


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                        "--workload", "tiny_broadcast", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny_broadcast"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_stored_traffic_matches_the_current_kernel_sources():
    # bench.py reports roofline.traffic only while the stored ncu counters were
    # taken from the sources that are built now; every entry must name a kernel
    # of this library and carry the hash of its current source file and headers
    import bench
    src = {"jfa_fwd_kernel": "fwd.cu", "jfa_fwd2_kernel": "fwd2.cu", "jfa_bwd_kernel": "bwd.cu"}
    assert bench.NCU_TRAFFIC
    for key, entry in bench.NCU_TRAFFIC.items():
        kernel, workload = key.split(":")[:2]
        assert kernel in src and workload in bench.workloads.WORKLOADS, key
        assert entry["bytes"] > 0
        assert entry["src_hash"] == bench.src_hash(src[kernel]), (
            f"{key}: counters taken from other sources; re-capture them (profiles/ gives the command)")


def test_source_hash_follows_code_not_comments():
    # a comment or a re-wrap leaves the code text (and so the hash) unchanged;
    # any change to code, string literals included, changes it
    import bench
    src = 'int a = 1;  // one\n/* two\n   lines */ asm("add.s32 %0, %1; // kept");\n'
    same = 'int a = 1;\n// another comment\nasm("add.s32 %0, %1; // kept"); /* x */\n'
    assert bench.code_text(src) == bench.code_text(same)
    assert bench.code_text(src) != bench.code_text(src.replace("a = 1", "a = 2"))
    assert bench.code_text(src) != bench.code_text(src.replace("// kept", "// gone"))
