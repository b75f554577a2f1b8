"""Host-side logic of bench.py (CPU): the source hash that ties stored ncu
counters to a build, the per-path launch counts, and the counted work."""
import os
import shutil

import bench
import gated_delta_rule_30_gb300 as kda


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "gated_delta_rule_30_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "gated_delta_rule_30_gb300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("*.o", "*.so"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash("decode")
    f = csrc / "kda_decode.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n\n", "\n   \n", 1) + "/* trailing */\n")
    assert bench.kernel_source_hash("decode") == h0
    f.write_text(text.replace("kDecThreads = kDim", "kDecThreads = 2 * kDim", 1))
    assert bench.kernel_source_hash("decode") != h0
    # a shared header counts for every kernel
    hdr = csrc / "kda_internal.h"
    hdr.write_text(hdr.read_text() + "\nconstexpr int kExtra = 1;\n")
    f.write_text(text)
    assert bench.kernel_source_hash("decode") != h0


def test_every_path_has_a_launch_count_and_sources():
    for path in kda.PATHS.values():
        assert bench.LAUNCHES[path] >= 1, path
    for path in ("sliced", "transposed", "segmented"):
        assert "recurrence/" + path in bench.KERNEL_SOURCES
    for kernel, files in bench.KERNEL_SOURCES.items():
        for name in files:
            assert os.path.exists(os.path.join(bench.ROOT, "gated_delta_rule_30_gb300", "csrc",
                                               name)), (kernel, name)


def test_counted_work_single_token_step():
    """T = 1: 1282 B per head-token plus the fp32 state read and written once."""
    import torch
    p = {"H": 32, "B": 1024, "T": 1, "N": 1024, "cu_seqlens": None,
         "state_dtype": torch.float32}
    head_tokens, flops, nbytes = bench.counted_work(p)
    assert head_tokens == 1024 * 32
    assert nbytes == 1024 * 32 * 1282 + 2 * 1024 * 32 * 128 * 128 * 4
    assert flops > 0


def test_backward_reference_arm_line():
    """bench.py --pass bwd --impl reference (the fp64 reverse-mode oracle on the host
    cores) prints one JSON line with the contract's keys, on the small workload."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--pass", "bwd",
                          "--impl", "reference", "--workload", "ref_small", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC_BWD
    assert line["value"] > 0 and line["unit"] == bench.UNIT and line["dtype"] == "f64"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["head_tokens_per_step"] == 512


def test_backward_counted_work_constants():
    """Counted bytes per head-token of the backward pass: q, k, v, g, dout (bf16)
    and beta read, dq, dk, dv, dg (fp32) and dbeta written; counted operations:
    11 D^2 (3 of a forward token step, 8 of a reverse one)."""
    D = 128
    assert bench.BWD_BYTES_PER_HEAD_TOKEN == 5 * 2 * D + 2 + 4 * 4 * D + 4
    assert bench.BWD_OPS_PER_HEAD_TOKEN == 11 * D * D
    assert abs(bench.FP32_LANE_PEAK_GOPS - 152 * 128 * 2.07) < 1e-9
