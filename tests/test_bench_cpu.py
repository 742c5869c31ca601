"""Host-side bookkeeping of bench.py: the algorithmic bytes each roofline
divides by, the unit each workload reports in, and the gate that keeps a DRAM
traffic figure from being reported once the kernels have changed."""
import argparse
import os

import bench
import oracle


def _args(**kw):
    a = dict(workload="decode", path="auto", fused=False, api="gemm", m=1, k=3584, n=3584,
             variant="w4a8")
    a.update(kw)
    return argparse.Namespace(**a)


def test_algorithmic_bytes_match_the_formats():
    """Counted from the formats, not from the formula: the packed weight is
    what the packer sizes it to, activations one int8 code per element plus an
    fp32 scale per token and an int32 sum per token and group, outputs bf16."""
    M, N, K = 16, 512, 3584
    G = K // 128
    packed = oracle.packed_w4_bytes(N, K)
    assert packed == 8512 * (N // 128) * G
    assert bench.w4a8_bytes(M, N, K) == packed + M * K + 4 * M + 4 * M * G + 2 * M * N
    assert bench.w4a16_bytes(M, N, K) == packed + 2 * M * K + 2 * M * N
    assert bench.w8a16_bytes(M, N, K) == N * K + 2 * N + 2 * M * K + 2 * M * N
    assert bench.w8a8_bytes(M, N, K) == N * K + 2 * N + M * K + 4 * M + 2 * M * N
    # quantization reads bf16 x, writes codes, scales and group sums
    assert bench.quant_bytes(M, K) == 2 * M * K + M * K + 4 * M + 4 * M * G


def test_units_follow_token_count():
    assert not bench.ops_unit(_args())                              # decode: GB/s
    assert bench.ops_unit(_args(workload="prefill"))                # prefill: TOPS
    assert bench.ops_unit(_args(workload="model", m=4096))
    assert not bench.ops_unit(_args(workload="model", m=64))
    assert bench.ops_unit(_args(workload="linear", m=65))
    assert not bench.ops_unit(_args(workload="linear", m=64))


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    """A capture keyed to the current kernel sources is read back; the same
    capture under any other sources hash is not (reported as null)."""
    key = bench.config_key(_args())
    good = tmp_path / "good"
    (good / "profiles").mkdir(parents=True)
    (good / "profiles" / "dram_traffic.txt").write_text(
        f"sources_sha256={bench.kernel_sources_hash()}\n"
        f"config={key}\tkernel=gemv_w4_kernel (W4A8)\tbytes_per_launch=1234\tlaunches=5\n")
    monkeypatch.setattr(bench, "ROOT", str(good))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: open(
        os.path.join(str(good), "profiles", "dram_traffic.txt")).readline().split("=")[1].strip())
    assert bench.measured_traffic(_args(), "gemv_w4_kernel (W4A8)") == 1234.0
    assert bench.measured_traffic(_args(), "tc_gemm_kernel (W4A8)") is None
    assert bench.measured_traffic(_args(workload="prefill"), "gemv_w4_kernel (W4A8)") is None
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "0" * 64)
    assert bench.measured_traffic(_args(), "gemv_w4_kernel (W4A8)") is None
