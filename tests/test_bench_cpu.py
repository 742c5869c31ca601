"""Host-side bookkeeping of bench.py: the algorithmic bytes each roofline
divides by, the plan of a step (which library calls, with which work), the unit
each workload reports in, the bound a roofline names, and the gate that keeps a
DRAM traffic figure from being reported once the kernels have changed."""
import argparse
import os

import bench
import oracle


def _args(**kw):
    a = dict(workload="sweep", path="auto", fused=False, api="grouped", m=1, k=3584, n=3584,
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
    # quantization reads bf16 x, writes codes, scales and group sums; the
    # operand form for the tensor cores (2 bytes a code) is counted apart
    assert bench.quant_bytes(M, K) == 2 * M * K + M * K + 4 * M + 4 * M * G
    assert bench.quant_actual_bytes(M, K) == bench.quant_bytes(M, K) + 2 * M * K
    assert bench.quant_actual_bytes(M, K, with_tc=False) == bench.quant_bytes(M, K)
    # the operand form alone (the int8 codes left out where no GEMV reads them)
    assert bench.quant_actual_bytes(M, K, with_codes=False) == 2 * M * K + 2 * M * K + 4 * M + 4 * M * G


def test_sweep_covers_m_1_to_4096_with_every_linear():
    cells = [c for p in bench.part_names(_args()) for c in bench.plan_part(_args(), p)]
    ms = sorted({c.M for c in cells})
    assert ms == [1, 4, 16, 512, 2048, 4096]
    gemms = [c for c in cells if c.kind == "w4a8"]
    # decode: q|k|v, o, gate|up, down at three M; prefill: the same + the head
    assert len(gemms) == 3 * 4 + 3 * 5
    names = {n for c in gemms for n in c.names}
    assert names == {"q", "k", "v", "o", "gate", "up", "down", "head"}
    # the same integer work however the siblings are launched
    ops = lambda a: sum(c.ops for p in bench.part_names(a) for c in bench.plan_part(a, p))
    assert ops(_args()) == ops(_args(api="gemm")) == ops(_args(api="linear"))
    per_m = {M: sum(c.ops for c in gemms if c.M == M) for M in ms}
    kn = sum(K * N for (_, K, N) in bench.SHAPES_7B)
    assert per_m[1] == 2 * kn and per_m[4096] == 2 * 4096 * (kn + 3584 * 152064)
    # one quantization per linear input and M (attn, o, mlp, down; + head)
    assert sum(c.kind == "quant" for c in cells) == 3 * 4 + 3 * 5


def test_units_follow_token_count():
    assert bench.ops_unit(_args())                                  # sweep: TOPS
    assert not bench.ops_unit(_args(workload="decode"))             # decode: GB/s
    assert bench.ops_unit(_args(workload="prefill"))                # prefill: TOPS
    assert bench.ops_unit(_args(workload="model", m=4096))
    assert not bench.ops_unit(_args(workload="model", m=64))
    assert bench.ops_unit(_args(workload="linear", m=65))
    assert not bench.ops_unit(_args(workload="linear", m=64))


def test_roofline_bound_follows_the_ridge():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops_sustained": 1500.0, "source": "measured"}
    # decode-sized: 64 ops a byte, below the 250 ops/B ridge -> HBM
    r = bench._roofline("k", 1.0, 10 ** 9, 64 * 10 ** 9, 10, peaks, None, None)
    assert r["bound"] == "hbm" and abs(r["achieved"] - 1000.0) < 1e-6
    # prefill-sized: far above the ridge -> tensor, with the int8 multiple
    r = bench._roofline("k", 1.0, 10 ** 9, 2000 * 10 ** 9, 10, peaks, {"tops": 100.0}, 5.0)
    assert r["bound"] == "tensor" and abs(r["frac"] - 2000.0 / 1500.0) < 1e-4
    assert abs(r["frac_of_int8_peak"] - 20.0) < 1e-4 and r["traffic"] == 5.0


def test_both_arms_print_the_same_config():
    a = _args()
    assert bench.workload_config(a) == bench.workload_config(_args())
    cfg = bench.workload_config(a)
    assert cfg["parts"] == ["decode", "prefill"]
    assert cfg["int_ops_per_step"] > 10 ** 13


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    """A capture keyed to the current kernel sources is read back per call
    shape and averaged per launch; the same capture under any other sources
    hash is not (null)."""
    good = tmp_path / "good"
    (good / "profiles").mkdir(parents=True)
    lab = "tc_gemm_kernel (W4A8, fp16 tiles)"
    (good / "profiles" / "dram_traffic.txt").write_text(
        f"sources_sha256=abc\n"
        f"kernel={lab}\tM=512\tN=3584\tK=3584\tbytes=1000\n"
        f"kernel={lab}\tM=2048\tN=3584\tK=3584\tbytes=3000\n")
    monkeypatch.setattr(bench, "ROOT", str(good))
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "abc")
    table = bench.traffic_table()
    mk = lambda M: bench.Cell("x", "w4a8", M, 3584, 3584, "o", ("o",), 0, 0)
    assert bench.measured_traffic(table, lab, [mk(512), mk(2048)], [1, 1]) == 2000.0
    # a call of two launches (a split second launch): bytes per launch
    assert bench.measured_traffic(table, lab, [mk(512), mk(2048)], [1, 2]) == 4000.0 / 3
    assert bench.measured_traffic(table, lab, [mk(512), mk(4096)], [1, 1]) is None
    assert bench.measured_traffic(table, "gemv_w4_kernel (W4A8)", [mk(512)], [1]) is None
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda: "0" * 64)
    assert bench.traffic_table() == {}
    assert os.path.exists(str(good / "profiles" / "dram_traffic.txt"))


def test_sources_hash_ignores_comments_only():
    """A comment or blank-line edit keeps the measured traffic valid; a code
    edit does not."""
    code = "int a = 1;  // the first\n/* a block\n   comment */\nint b = 2;\n"
    assert bench._code_only(code) == bench._code_only(
        "int a = 1;\n\n// another note\nint b = 2;  /* trailing */\n")
    assert bench._code_only(code) != bench._code_only("int a = 1;\nint b = 3;\n")


def test_launch_accounting_counts_split_tails():
    """gpu_launches counts every kernel launch of the step's calls: the
    quantizations, one GEMM launch a call, and the second launch the library
    reports for a long-K grid's split tail (the down projection at 2048 and
    4096 tokens). Host-only queries of the library (its SM count falls back
    to 148 without a device; these shapes split on 148 and 152 alike)."""
    import w4a8_quantized_gemm_gb300 as eg
    from w4a8_quantized_gemm_gb300 import builder
    builder.build()
    eg.load()
    cells = bench.plan_part(_args(workload="prefill"), "prefill")
    launches = [bench.call_launches(eg, c, eg.PATH_AUTO) for c in cells]
    tails = [c for c in cells if c.kind == "w4a8" and
             bench.kernel_launches(eg, c, eg.PATH_AUTO) == 2]
    assert sorted((c.M, c.N, c.K) for c in tails) == [(2048, 3584, 18944), (4096, 3584, 18944)]
    assert sum(launches) == len(cells) + 2 == 32
