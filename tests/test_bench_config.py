"""bench.py's description of what it times (CPU): the L2 note that the timing rules rest on,
the kernel family, ceiling and launch count it reports for each dtype and head dimension,
the kernel-source hash that gates recorded DRAM traffic, the input description, and the
reference (CPU oracle) arm's JSON line."""
import os

import bench
from bwd_xfa_fwd_gb300 import inputs
from bwd_xfa_fwd_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_l2_note_follows_the_total_of_the_streamed_inputs():
    # workload 5: Q, K, V, dO of 64 MiB each, 256 MiB per step against a 129 MB L2
    assert "larger than L2" in bench.workload_config(inputs.WORKLOADS[5])["l2"]
    assert "larger than L2" in bench.workload_config(inputs.WORKLOADS[4])["l2"]
    for wid in (1, 2, 3):   # 0.02 / 1 / 12 MiB each: fit, timed warm
        assert "fit in L2" in bench.workload_config(inputs.WORKLOADS[wid])["l2"]


def test_family_resolution_matches_the_library_dispatch():
    w5, w2, w1 = inputs.WORKLOADS[5], inputs.WORKLOADS[2], inputs.WORKLOADS[1]
    assert bench.resolved_family(w5, "auto") == "tc"
    assert bench.resolved_family(w5, "tcgen05_det") == "tc_det"
    assert bench.resolved_family(w2, "auto") == "tf32x3"      # fp32, hd 64
    assert bench.resolved_family(w1, "tcgen05") == "tf32x3"   # fp32, hd 32
    assert bench.resolved_family(w5, "simt") == "simt"
    hd128 = inputs.Workload("f32_hd128", 1, 1, 256, 128, "f32", 0.1, seed=0)
    assert bench.resolved_family(hd128, "auto") == "simt"    # fp32 hd 128 stays on FFMA


def test_ceilings_and_launch_counts():
    pk = {"bf16_tflops": 1892.5}
    peak, _ = bench.tensor_peak(pk, "measured", "tc")
    assert peak == 1892.5
    peak, _ = bench.tensor_peak(pk, "measured", "tf32x3")
    assert abs(peak - 1892.5 * 1.1 / 2.25 / 3.0) < 1e-9
    peak, _ = bench.tensor_peak(pk, "measured", "simt")
    assert abs(peak - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
    w5, w2 = inputs.WORKLOADS[5], inputs.WORKLOADS[2]
    assert bench.kernel_labels(w5, "tc")[2] == 4        # fwd, prep, bwd, dQ conversion
    assert bench.kernel_labels(w2, "tf32x3")[2] == 4    # fwd, prep, key-tile and query-tile kernels
    assert bench.kernel_labels(w2, "simt")[2] == 3      # fwd, prep, bwd (dQ summed in place)


def test_source_hash_ignores_comments_only():
    import os
    import tempfile
    src = "int f(int x)\n{\n    return x + 1;   // one\n}\n"
    with tempfile.TemporaryDirectory() as d:
        paths = []
        for i, text in enumerate((src, src.replace("// one", "// two"), src.replace("x + 1", "x + 2"))):
            p = os.path.join(d, f"k{i}.cu")
            with open(p, "w") as f:
                f.write(text)
            paths.append(p)
        saved = dict(bench.KERNEL_SOURCES)
        try:
            hashes = []
            for p in paths:
                bench.KERNEL_SOURCES["probe"] = (os.path.relpath(p, bench.ROOT),)
                hashes.append(bench.source_hash("probe"))
        finally:
            bench.KERNEL_SOURCES.clear()
            bench.KERNEL_SOURCES.update(saved)
    assert hashes[0] == hashes[1] and hashes[0] != hashes[2]


def test_data_note_states_each_workloads_distribution():
    notes = {i: bench.data_note(WORKLOADS[i]) for i in WORKLOADS}
    assert "dO ~ N(0,0.1^2)" in notes[2] and "bf16" not in notes[2]
    assert "Q, K ~ N(0,2^2)" in notes[4] and "rounded to bf16" in notes[4]
    assert notes[5].startswith("synthetic, seed 5: Q, K, V, dO ~ N(0,1), rounded to bf16")


def test_reference_arm_line_on_the_smallest_workload():
    """`bench.py --impl reference` times the CPU oracle and prints one JSON line with the
    contract's keys (run on workload 1, which takes well under a second)."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == WORKLOADS[1].name
    # the same config object as the repo arm's line (no family or other run options in it)
    assert d["config"] == bench.workload_config(WORKLOADS[1])
