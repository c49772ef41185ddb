"""bench.py's host logic, without a GPU: the reference arm's JSON line (the
CPU oracle timed on a bounded sample), the GPU arm failing loudly when there
is no GPU (no CPU fallback), and the DRAM-traffic record keyed by a digest of
the dominant kernel's own sources."""
import json
import os
import shutil
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _last_json(out):
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert lines, out[-2000:]
    return json.loads(lines[-1])


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = _last_json(r.stdout)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] in ("GB/s", "TFLOP/s") and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "decode_block32" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_fails_loudly_without_a_gpu():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0
    assert not any(ln.startswith("{") and '"value"' in ln for ln in r.stdout.splitlines())


def test_traffic_record_keyed_by_source_digest(tmp_path, monkeypatch):
    f = tmp_path / "dram_traffic.txt"
    digest = bench.kernel_source_digest("decode_block32")
    f.write_text(f"# comment\ndecode_block32  {digest}  12345  note\nprefill_block128  {digest}  999\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("decode_block32") == 12345
    # prefill_block128 hashes every source: another digest, so no figure
    assert bench.measured_traffic("prefill_block128") is None
    f.write_text(f"decode_block32  {'0' * 16}  12345\n")
    assert bench.measured_traffic("decode_block32") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.txt"))
    assert bench.measured_traffic("decode_block32") is None


def test_digest_follows_the_listed_sources_only(tmp_path, monkeypatch):
    root = tmp_path / "r"
    shutil.copytree(os.path.join(ROOT, "fp8_block_scaled_sgq_gb300", "csrc"),
                    root / "fp8_block_scaled_sgq_gb300" / "csrc")
    shutil.copytree(os.path.join(ROOT, "include"), root / "include")
    monkeypatch.setattr(bench, "ROOT", str(root))
    d0 = bench.kernel_source_digest("decode_block32")
    assert d0 == bench.kernel_source_digest("decode_block32")
    csrc = root / "fp8_block_scaled_sgq_gb300" / "csrc"
    with open(csrc / "gemm_dual.cuh", "a") as fh:   # not a source of the decode kernel
        fh.write("\n// edit\n")
    assert bench.kernel_source_digest("decode_block32") == d0
    with open(csrc / "gemm_kernel.cuh", "a") as fh:  # a source of it
        fh.write("\n// edit\n")
    d1 = bench.kernel_source_digest("decode_block32")
    assert d1 != d0
    with open(root / "include" / "sgq.h", "a") as fh:
        fh.write("\n/* edit */\n")
    assert bench.kernel_source_digest("decode_block32") != d1
