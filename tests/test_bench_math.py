"""The bench line's roofline arithmetic, recomputed on the CPU from closed
forms: which measured peak a fraction takes (burst for a timed region under
a second, sustained beyond), the routed experts' FLOPs, the whole layer's
expert FLOPs and the decode workloads' weight bytes.  Every fraction on the
line must recompute from its other fields."""
import importlib.util
import math
import os

from expert_ffn_layer_affinity_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

PK = dict(hbm=6500.0, bf16=1800.0, bf16_sust=1400.0, src="measured")


def test_peak_follows_the_timed_region():
    assert bench.tensor_peak(PK, 0.2)[0] == 1800.0
    assert bench.tensor_peak(PK, bench.SUSTAINED_AFTER_S - 1e-6)[0] == 1800.0
    assert bench.tensor_peak(PK, bench.SUSTAINED_AFTER_S)[0] == 1400.0
    assert bench.tensor_peak(PK, 5.0)[0] == 1400.0
    # E4M3 takes twice the bf16 figure (the nominal dense ratio)
    assert bench.tensor_peak(PK, 0.2, fp8=True)[0] == 3600.0
    assert bench.tensor_peak(PK, 5.0, fp8=True)[0] == 2800.0


def test_v3_routed_flops_and_roofline_entry():
    cfg = synth.CONFIGS["v3"]
    R = cfg.T * cfg.K
    flops = 6.0 * 7168 * 2048 * 65536            # GEMM1 (w1, w3) + GEMM2 over R rows
    assert R == 65536
    assert bench.algorithmic(cfg, 256)["routed"]["flops"] == flops
    ms = flops / 1e12                             # 1000 TFLOP/s by construction
    res = dict(per={"routed": ms, "shared": 0.5}, touched=256, ms=20 * 7.0)
    r = bench.roofline_entry(cfg, res, 20, PK)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["achieved"], 1000.0, rel_tol=1e-6)
    assert r["peak"] == 1800.0                    # 0.14 s timed: burst
    assert math.isclose(r["frac"], 1000.0 / 1800.0, abs_tol=1e-4)
    assert math.isclose(r["frac_of_sustained"], 1000.0 / 1400.0, abs_tol=1e-4)
    assert math.isclose(r["traffic"], bench.GEMM_TRAFFIC_PER_EXPERT * 256, rel_tol=1e-12)
    # a seconds-long timed region takes the sustained peak
    res_long = dict(res, ms=2000.0)
    assert bench.roofline_entry(cfg, res_long, 200, PK)["peak"] == 1400.0


def test_layer_fraction_counts_routed_and_shared_experts():
    cfg = synth.CONFIGS["v3"]
    flops = 6.0 * 7168 * 2048 * 8192 * (8 + 1)
    assert cfg.expert_flops() == flops
    ms_step = flops / 1e12 / 0.9                  # 900 TFLOP/s by construction
    lf = bench.layer_fraction(cfg, ms_step, 0.2, PK)
    assert math.isclose(lf["expert_tflops"], 900.0, abs_tol=0.05)
    assert math.isclose(lf["frac"], 0.5, abs_tol=1e-4)
    assert math.isclose(lf["frac_of_sustained"], 900.0 / 1400.0, abs_tol=1e-4)


def test_decode_fraction_is_weight_streaming_against_hbm():
    cfg = synth.CONFIGS["v3_decode"].with_T(64)
    touched = 200
    wbytes = 3.0 * (touched + 1) * 2048 * 7168 * 2    # w1, w3, w2 of touched + shared experts
    ms = wbytes / 6.5e12 * 1e3                        # 6500 GB/s by construction
    res = dict(per={"routed": ms * 0.9, "shared": ms * 0.1}, touched=touched, ms=20 * 3.0)
    r = bench.roofline_entry(cfg, res, 20, PK)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["weight_bytes_per_step"] == wbytes
    assert math.isclose(r["achieved"], 6500.0, abs_tol=0.1)
    assert math.isclose(r["frac"], 1.0, abs_tol=1e-4)


def test_tiny_layer_reports_no_fraction():
    cfg = synth.CONFIGS["tiny"]
    res = dict(per={"routed": 0.02, "shared": 0.01}, touched=16, ms=50 * 0.1)
    r = bench.roofline_entry(cfg, res, 50, PK)
    assert r["frac"] is None and r["achieved"] is None
