"""Host-side checks of the benchmark's bookkeeping (no GPU): the roofline record
states the bound the arithmetic intensity gives, and both arms report one config."""
import math

import bench
from expert_grouped_gemm_gb300.inputs import WORKLOADS

PEAKS = {"hbm_gbs": 6780.0, "bf16_tflops": 1942.5}


def test_bound_follows_the_ridge_point():
    q = WORKLOADS["qwen3_t4096_full"]
    r = bench.gemm_roofline(q, q.P, q.E, q.E, 1.0, PEAKS, "test")
    # 9.3e11 flop over 5.1e9 B: about 185 flop/B, below the ridge 1942.5e12 / 6780e9 = 286.5
    assert r["flop_per_byte"] < r["ridge_flop_per_byte"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm_gbs"]
    assert math.isclose(r["frac"], r["achieved"] / r["peak"])
    assert math.isclose(r["tensor_frac"], r["gemm_flops_per_step"] / 1e-3 / 1e12 / PEAKS["bf16_tflops"])
    # the byte floor dominates, so the roofline fraction is the HBM fraction
    assert math.isclose(r["frac_roofline"], r["hbm_frac"])
    g = WORKLOADS["glm45_t8192_full"]
    r = bench.gemm_roofline(g, g.P, g.E - 4, g.E - 4, 5.0, PEAKS, "test")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["frac_roofline"], r["tensor_frac"])


def test_both_arms_report_the_same_config():
    for w in WORKLOADS.values():
        c = bench.bench_config(w, 1)
        assert c == bench.bench_config(w, 1)
        assert c["workload"] == w.name
        # nothing measured on the GPU is part of the config
        assert not any(k.startswith(("R_", "expert_load", "zero_load")) for k in c)
