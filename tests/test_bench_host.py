"""Host-side pieces of bench.py that need no GPU: the algorithmic byte and
FLOP counts the roofline divides by, and the rule that a profile's DRAM
traffic is reported only for the kernel source it was measured on."""
import os

import numpy as np

import bench
import synth


def test_algorithmic_counts_dec1():
    w = synth.WORKLOADS["dec1"]
    ids = np.arange(8, dtype=np.int32).reshape(1, 8)  # one token, 8 distinct experts
    work = bench.algorithmic(w, [ids])
    per_expert = 3 * w.I * w.H * 34 / 32  # gate, up, down Q8_0 rows, 34 bytes per 32 weights
    assert work["U"] == [8]
    assert abs(work["gu_bytes"] + work["d_bytes"] - (8 * per_expert + 2 * w.H * 2 + 2 * 8 * w.I * 4)) < 1
    assert work["flops"] == 8 * 3 * 2 * w.H * w.I


def test_algorithmic_counts_repeated_expert():
    w = synth.WORKLOADS["dec16"]
    ids = np.tile(np.arange(8, dtype=np.int32), (16, 1))  # 16 tokens, all on experts 0..7
    work = bench.algorithmic(w, [ids])
    assert work["U"] == [8]  # each touched expert's weights count once per call
    assert work["flops"] == 16 * 8 * 3 * 2 * w.H * w.I


def test_measured_traffic_requires_matching_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = tmp_path / "quantized_sparse_moe_router_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["decode_experts"]:
        (src / f).write_text("// " + f + "\nint x_" + f.replace(".", "_") + " = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.kernel_source_hash("decode_experts")
    (prof / "decode_experts_dec1.md").write_text(
        f"# summary\n\ntraffic_bytes_per_launch: 40203008\nsource_sha256: {digest}\n")
    assert bench.measured_traffic("decode_experts", "dec1") == 40203008.0
    # comments and blank lines do not change the measured code
    (src / "decode.cu").write_text("/* new\n   comment */\n\nint x_decode_cu = 1;   // same code\n")
    assert bench.measured_traffic("decode_experts", "dec1") == 40203008.0
    (src / "decode.cu").write_text("int x_decode_cu = 2;\n")  # kernel edited after the capture
    assert bench.measured_traffic("decode_experts", "dec1") is None
    assert bench.measured_traffic("decode_experts", "dec16") is None  # no summary for that workload


def test_whole_job_rate_is_aggregate():
    assert bench.whole_job_rate(100.0, 2.0, 4) == 200.0


def test_gemm_roofline_takes_the_binding_bound():
    # a weight-streaming GEMM (few FLOPs a byte) is HBM-bound, a token-heavy one tensor-bound;
    # achieved and frac follow from the work and the time, and the other bound is reported beside
    import bench
    hbm, bf16 = 6789.0, 1905.7
    r = bench.gemm_roofline(fl=1.08e12, gb=8.2e9, k_us=1700.0, hbm=hbm, bf16=bf16, peak_src="measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 8.2e9 / 1700e-6 / 1e9) < 0.1 and abs(r["frac"] - r["achieved"] / hbm) < 1e-4
    assert r["tensor"]["unit"] == "TFLOP/s" and abs(r["tensor"]["achieved"] - 1.08e12 / 1700e-6 / 1e12) < 0.1
    r = bench.gemm_roofline(fl=2.06e11, gb=0.5e9, k_us=305.0, hbm=hbm, bf16=bf16, peak_src="measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["hbm"]["unit"] == "GB/s"
    assert abs(r["frac"] - 2.06e11 / 305e-6 / 1e12 / bf16) < 1e-4
