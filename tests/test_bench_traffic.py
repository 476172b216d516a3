"""bench.py --traffic-json on a synthetic ncu CSV (no GPU): the last 14 bf16_tc_gemm launches
of the capture are one step's 7 forward GEMMs then its 7 dX GEMMs, in projection order; the
record averages their DRAM bytes per kind and is keyed to the GEMM source's SHA-256."""

import hashlib
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _csv(path):
    hdr = '"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n'
    lines = [hdr]
    # two other kernels and 16 GEMM launches: the first two belong to an earlier step
    lines.append('"0","adapter_tc(AdapterLaunch)","gpu__time_duration.sum","ns","1,000"\n')
    for i in range(16):
        gid = 1 + i
        kind_bytes = 1_000_000 * (i + 1)
        for name, unit, val in (("dram__bytes_read.sum", "byte", kind_bytes),
                                ("dram__bytes_write.sum", "Kbyte", 5),
                                ("gpu__time_duration.sum", "us", 10 + i)):
            lines.append(f'"{gid}","bf16_tc_gemm(GemmLaunch)","{name}","{unit}","{val:,}"\n')
    lines.append('"99","finish_partials(FinishJobs)","gpu__time_duration.sum","ns","500"\n')
    with open(path, "w") as f:
        f.writelines(["==PROF== noise line\n"] + lines)


def test_traffic_record_from_synthetic_csv(tmp_path):
    path = tmp_path / "gemm.csv"
    _csv(path)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--traffic-json", str(path)],
                         capture_output=True, text=True, cwd=ROOT, timeout=120)
    assert out.returncode == 0, out.stderr
    rec = json.loads(out.stdout)
    fwd, dx = rec["launches"]["fwd_gemm"], rec["launches"]["dx_gemm"]
    assert [x["projection"] for x in fwd] == ["q", "k", "v", "o", "gate", "up", "down"]
    assert [x["projection"] for x in dx] == ["q", "k", "v", "o", "gate", "up", "down"]
    # launches 3..9 (1-based IDs) are the forward ones, 10..16 the dX ones
    assert [x["dram_bytes"] for x in fwd] == [1_000_000 * k + 5_000 for k in range(3, 10)]
    assert [x["dram_bytes"] for x in dx] == [1_000_000 * k + 5_000 for k in range(10, 17)]
    assert fwd[0]["duration_ns"] == 12_000
    assert rec["per_launch_bytes"]["fwd_gemm"] == sum(x["dram_bytes"] for x in fwd) // 7
    src = os.path.join(ROOT, "bit_nf4_quantized_gb300", "csrc", "linear_tc.cu")
    assert rec["source_sha256"] == hashlib.sha256(open(src, "rb").read()).hexdigest()
