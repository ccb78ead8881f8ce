"""The bench's output contract on CPU: `bench.py --impl reference` prints one JSON line with the
keys the driver reads (the GPU arm's line is checked on the GPU machine by running it)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["warmup"] >= 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_figures_survive_comment_edits_and_retire_on_code_edits(tmp_path, monkeypatch):
    """A DRAM-traffic figure is reported only while its kernel source's code is the one it was
    captured on: the hash leaves out comments and blank space, and sees any change to the code."""
    bench = _bench()
    csrc = tmp_path / "video_audio_gen_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    code = "__global__ void k(float* x) {\n  x[threadIdx.x] *= 2.f;\n}\n"
    (csrc / "k.cu").write_text(code)
    h0 = bench.source_hash("k.cu")
    (csrc / "k.cu").write_text("// doubled\n/* one\n   element per thread */\n" + code.replace("  x", "    x") + "\n\n")
    assert bench.source_hash("k.cu") == h0
    (csrc / "k.cu").write_text(code.replace("*= 2.f", "*= 3.f"))
    assert bench.source_hash("k.cu") != h0


def test_traffic_kinds_map_to_their_kernel_sources():
    bench = _bench()
    bf16, fp32 = {"dtype": "bf16"}, {"dtype": "fp32"}
    assert bench.traffic_src("attention", bf16) == "attention.cu"
    assert all(bench.traffic_src(k, bf16) == "gemm.cu" for k in ("gemm_qkv", "gemm_out", "gemm_ffn_up", "gemm_ffn_down"))
    assert bench.traffic_src("norm_modulate", bf16) == "elementwise.cu"
    assert bench.traffic_src("attention", fp32) == bench.traffic_src("gemm_qkv", fp32) == "fp32.cu"
    for (kind, workload), entry in bench.TRAFFIC.items():
        assert entry["bytes"] > 0 and len(entry["src_sha"]) == 16
        src = bench.traffic_src(kind, fp32 if "fp32" in workload else bf16)
        assert os.path.exists(os.path.join(ROOT, "video_audio_gen_gb300", "csrc", src))
