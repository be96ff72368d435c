"""Host-side arithmetic of bench.py, checked without a GPU: the algorithmic
bytes of one product, the whole-job aggregate over replicas, the roofline of
the dominant kernel, and the DRAM-traffic lookup keyed on the kernel source
(a capture counts only while the source it was taken from is unchanged)."""
import os

import pytest

import bench


def test_algorithmic_bytes_of_one_product():
    # W8A16: fp16 X read (2MK), E4M3 W read (NK), fp16 Y written (2MN),
    # one fp32 scale per channel (4N)
    assert bench.w8a16_bytes(1, 16, 32) == 2 * 32 + 16 * 32 + 2 * 16 + 4 * 16
    # the launch the committed M=16 capture was taken on
    assert bench.w8a16_bytes(16, 22016, 4096) == 91101184
    # W8A8: codes of A and W, the output, the weight scale(s), the activation scale
    assert bench.w8a8_bytes(16, 32, 64, 2, True) == 16 * 64 + 32 * 64 + 16 * 32 * 2 + 4 * 32 + 4
    assert bench.w8a8_bytes(16, 32, 64, 1, False) == 16 * 64 + 32 * 64 + 16 * 32 + 4 + 4


def test_aggregate_is_the_work_of_all_replicas_over_the_slowest_step():
    # 610 MB per step in 0.1 ms: 6100 GB/s on one GPU, 4x on four replicas
    assert bench.aggregate(610e6, 0.1, 1, "GB/s") == pytest.approx(6100.0)
    assert bench.aggregate(610e6, 0.1, 4, "GB/s") == pytest.approx(24400.0)
    # 2e11 flops in 0.1 ms: 2000 TFLOP/s
    assert bench.aggregate(2e11, 0.1, 1, "TFLOP/s") == pytest.approx(2000.0)


PEAKS = {"hbm_gbs": 6807.9, "bf16_tflops": 1906.3, "source": "measured"}


def test_roofline_of_the_dominant_kernel_uses_its_share_of_the_step():
    per_kind = {
        "quant_dynamic": {"ms": 1.0, "units_per_step": 12e6, "unit": "bytes",
                          "launches_per_step": 2},
        "scaled_mm_tcgen05": {"ms": 3.0, "units_per_step": 1.2e11, "unit": "flops",
                              "launches_per_step": 2},
    }
    rf, kinds = bench.roofline(per_kind, PEAKS, ms_per_step=0.08)
    assert rf["kernel"] == "scaled_mm_tcgen05"
    assert rf["share"] == 0.75
    # 1.2e11 flops in 0.08 ms x 0.75 = 60 us: 2000 TFLOP/s against 2 x 1906.3
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert rf["achieved"] == pytest.approx(2000.0, abs=0.01)
    assert rf["peak"] == pytest.approx(3812.6)
    assert rf["frac"] == pytest.approx(2000.0 / 3812.6, abs=1e-4)
    assert kinds["quant_dynamic"]["share"] == 0.25


def test_roofline_of_a_bandwidth_bound_step():
    per_kind = {"w8a16_skinny": {"ms": 5.0, "units_per_step": 610e6, "unit": "bytes",
                                 "launches_per_step": 12}}
    rf, _ = bench.roofline(per_kind, PEAKS, ms_per_step=0.1265)
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["share"] == 1.0
    assert rf["achieved"] == pytest.approx(610e6 / 0.1265e-3 / 1e9, abs=0.1)
    assert rf["peak"] == pytest.approx(6807.9)
    assert rf["launches_per_step"] == 12


def _fake_tree(root, skinny_src):
    csrc = os.path.join(root, "fp8_quantized_linear_gb300", "csrc")
    os.makedirs(csrc)
    os.makedirs(os.path.join(root, "profiles"))
    with open(os.path.join(csrc, "skinny.cu"), "w") as f:
        f.write(skinny_src)
    with open(os.path.join(csrc, "gemm_tcgen05.cu"), "w") as f:
        f.write("// another kernel\n")
    with open(os.path.join(csrc, "common.cuh"), "w") as f:
        f.write("// shared header\n")


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    # the hash covers the kernel's file and the library headers it includes
    root = str(tmp_path)
    _fake_tree(root, '#include "common.cuh"\n// kernel v1\n')
    monkeypatch.setattr(bench, "ROOT", root)
    h = bench.kernel_source_hash("skinny.cu")
    with open(os.path.join(root, "profiles", "traffic.md"), "w") as f:
        f.write("| kind | hash | bytes | algorithmic | launch |\n|---|---|---|---|---|\n")
        f.write(f"| w8a16_skinny | {h} | 93158144 | 91101184 | M=16 N=22016 K=4096 |\n")
    got = bench.traffic_from_profile("w8a16_skinny")
    assert got == {"bytes": 93158144, "algorithmic_bytes": 91101184,
                   "launch": "M=16 N=22016 K=4096"}
    # a kind without a row has no figure
    assert bench.traffic_from_profile("scaled_mm_tcgen05") is None
    # a changed kernel source (or shared header) voids the capture
    with open(os.path.join(root, "fp8_quantized_linear_gb300", "csrc", "skinny.cu"), "a") as f:
        f.write("// edited\n")
    assert bench.traffic_from_profile("w8a16_skinny") is None
    with open(os.path.join(root, "fp8_quantized_linear_gb300", "csrc", "skinny.cu"), "w") as f:
        f.write('#include "common.cuh"\n// kernel v1\n')
    assert bench.traffic_from_profile("w8a16_skinny") is not None
    with open(os.path.join(root, "fp8_quantized_linear_gb300", "csrc", "common.cuh"), "a") as f:
        f.write("// edited\n")
    assert bench.traffic_from_profile("w8a16_skinny") is None


def test_reference_arm_prints_one_line_on_rank_0_only(monkeypatch, capsys):
    # the oracle timed on the host: rank 0 prints the line, other ranks
    # return without work
    import json
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3",
                             "--workload", "tiny_w8a8"])
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(args)
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["config"]["workload"] == "tiny_w8a8"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_per_shape_roofline_is_the_lower_of_tensor_peak_and_bandwidth():
    # M = 64, N = K = 8192 E4M3 with E4M3 output and per-channel scales:
    # AI = 2MNK / bytes ~ 124 flop/B, so 6807.9 GB/s allows ~845 TFLOP/s,
    # below the 3812.6 TFLOP/s peak: bound by HBM
    M, N, K = 64, 8192, 8192
    nbytes = bench.w8a8_bytes(M, N, K, 1, True)
    flops = 2 * M * N * K
    r = bench.shape_roofline(flops, nbytes, 30e-6, 3812.6, 6807.9)
    mem_roof = 6807.9 * flops / nbytes / 1e3
    assert r["bound"] == "hbm"
    assert r["roof_TFLOP/s"] == pytest.approx(mem_roof, abs=0.05)
    assert r["frac"] == pytest.approx(flops / 30e-6 / 1e12 / mem_roof, abs=1e-4)
    assert r["hbm_frac"] == pytest.approx(nbytes / 30e-6 / 1e9 / 6807.9, abs=1e-4)
    # M = 4096: compute-bound, the roofline is the tensor peak
    M = 4096
    nbytes = bench.w8a8_bytes(M, N, K, 1, True)
    r = bench.shape_roofline(2 * M * N * K, nbytes, 200e-6, 3812.6, 6807.9)
    assert r["bound"] == "tensor" and r["roof_TFLOP/s"] == 3812.6
    assert r["frac"] == pytest.approx(2 * M * N * K / 200e-6 / 1e12 / 3812.6, abs=1e-4)


def test_small_m_summary_splits_at_the_target():
    rows = [{"M": 1, "N": 16, "K": 16, "hbm_frac": 0.71},
            {"M": 16, "N": 32, "K": 16, "hbm_frac": 0.69},
            {"M": 64, "N": 32, "K": 16, "hbm_frac": 0.10}]
    s = bench.small_m_summary([("w", rows)])
    assert s["target_hbm_frac"] == 0.70
    assert s["at_or_above"] == ["w M=1 N=16 K=16: 0.71"]
    assert s["below"] == ["w M=16 N=32 K=16: 0.69"]


def test_default_workload_is_the_largest():
    args = bench.parse_args([])
    assert args.workload == "llama70b_static_fp8out"
    import synthetic
    flops = {n: sum(2 * m * n_ * k for (m, n_, k) in w.shapes)
             for n, w in synthetic.WORKLOADS.items()}
    assert max(flops, key=flops.get) == args.workload


def test_long_timed_regions_use_the_sustained_tensor_peak():
    peaks = {"hbm_gbs": 6807.9, "bf16_tflops": 1951.8, "bf16_tflops_sustained": 1690.5,
             "source": "measured"}
    per_kind = {"scaled_mm_tcgen05": {"ms": 1.0, "units_per_step": 3e12, "unit": "flops",
                                      "launches_per_step": 12}}
    burst, _ = bench.roofline(per_kind, peaks, ms_per_step=1.0)
    sust, _ = bench.roofline(per_kind, peaks, ms_per_step=1.0, sustained=True)
    assert burst["peak"] == pytest.approx(3903.6) and sust["peak"] == pytest.approx(3381.0)
    assert burst["frac"] == burst["frac_of_burst"] == pytest.approx(3000 / 3903.6, abs=1e-4)
    assert sust["frac"] == pytest.approx(3000 / 3381.0, abs=1e-4)
    assert sust["frac_of_burst"] == burst["frac"]
    assert "sustained" in sust["peak_source"] and "burst" in burst["peak_source"]


def _two_machine_makespan(order, first, second):
    t1 = t2 = 0
    for i in order:
        t1 += first[i]
        t2 = max(t2, t1) + second[i]
    return t2


def test_johnson_order_minimizes_the_two_machine_makespan():
    # brute force over every order of small random instances (ties included)
    import itertools
    import random
    rng = random.Random(5)
    for _ in range(200):
        n = rng.randint(1, 6)
        first = [rng.randint(0, 9) for _ in range(n)]
        second = [rng.randint(0, 9) for _ in range(n)]
        order = bench.johnson_order(first, second)
        assert sorted(order) == list(range(n))
        best = min(_two_machine_makespan(p, first, second) for p in itertools.permutations(range(n)))
        assert _two_machine_makespan(order, first, second) == best


def test_johnson_order_of_the_headline_copies():
    # a product with a small input and a large output goes early, one with
    # a large input and a small output late
    order = bench.johnson_order([67, 235, 1, 17], [235, 34, 4, 59])
    assert order == [2, 3, 0, 1]
