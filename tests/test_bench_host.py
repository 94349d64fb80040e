"""Host-side arithmetic of bench.py (no GPU): the method bytes and flops the
rooflines divide by, the choice of the binding roof, the launch count, and
the digest that closes the JSON line."""
import math

import pytest

import bench


def test_layer_costs_dsv4_m4096():
    c = bench.layer_costs(4096, 4096, 256, 2048, 8)
    touched = 256 * (1 - (1 - 8 / 256) ** 4096)
    assert math.isclose(touched, 256.0, rel_tol=1e-12)        # every expert touched
    w13 = 256 * 2 * 2048 * 4096 * 2
    assert c["gate_up"]["method"] == pytest.approx(w13 + 4096 * 4096 * 2 + 4096 * 8 * 8)
    assert c["gate_up"]["impl"] == 4096 * 8 * 4096 * 2 + 4096 * 8 * 2048 * 2   # gathered rows, act
    assert c["gate_up"]["flops"] == 2.0 * 4096 * 8 * 2 * 2048 * 4096
    assert c["down"]["method"] == pytest.approx(256 * 4096 * 2048 * 2 + 4096 * 4096 * 2)
    assert c["down"]["impl"] == 4096 * 8 * 2048 * 2 + 4096 * 8 * 4096 * 4     # act, contributions
    # the step adds the router's weight and scores once
    assert c["step"]["method"] == pytest.approx(256 * 4096 * 4 + 4096 * 256 * 4 + 4096 * 4096 * 2 + w13
                                                + 256 * 4096 * 2048 * 2 + 4096 * 4096 * 2 + 4096 * 8 * 8)


def test_layer_costs_decode_touches_k_experts():
    c = bench.layer_costs(1, 2048, 128, 768, 8)
    assert c["gate_up"]["method"] == pytest.approx(8 * 2 * 768 * 2048 * 2 + 2048 * 2 + 64)
    # the gathered copy is workspace, not method bytes; the in-GEMM feed has none
    assert bench.layer_costs(1, 2048, 128, 768, 8, "gemm")["gate_up"]["impl"] == 8 * 768 * 2


def test_roofline_entry_picks_the_binding_roof():
    hbm, tc = 6767.7, 1929.6
    # HBM-bound: 8.6 GB take 1.27 ms at the copy bandwidth, 1.1 TFLOP 0.57 ms at the bf16 peak
    c = {"method": 8.6e9, "impl": 0.4e9, "flops": 1.1e12}
    r = bench.roofline_entry("k", c, 1.5, hbm, tc, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(8.6e9 / 1.5e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / hbm)
    assert r["implementation_bytes"] == 0.4e9 and r["traffic"] is None
    # tensor-bound: 0.1 GB take 15 us, 1 PFLOP 0.52 s
    c = {"method": 1e8, "impl": 0, "flops": 1e15}
    r = bench.roofline_entry("k", c, 1.0, hbm, tc, "measured", traffic=123)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(1e15 / 1e-3 / 1e12 / tc)
    assert r["traffic"] == 123


def test_launches_per_step():
    # router + top-k, three-launch permutation, gather, gate/up, down, combine
    assert bench.launches_per_step(4096, 256) == 9
    # one-CTA permutation up to 1024 tokens when its shared memory fits
    assert bench.launches_per_step(1024, 128) == 7
    assert bench.launches_per_step(1024, 1024) == 9          # E=1024 does not fit
    assert bench.launches_per_step(4096, 256, "gemm") == 8   # no gather launch


def test_summary_digest_keys():
    rl = {"bound": "hbm", "frac": 0.88, "achieved": 5950.0, "unit": "GB/s", "ms_per_launch": 1.45,
          "tensor_frac_of_burst": 0.39}
    extras = {
        "router_us_vs_M": {"fp32_fma_peak_tflops_measured": 77.7,
                           "1": {"warm_us": 3.7, "warm_fp32_frac": 0.007, "fused_router_topk_warm_us": 8.7,
                                 "chained_router_topk_warm_us": 8.7,
                                 "cublas_fp32_rows_changed_vs_M4096": 1}},
        "moe_layer_us_vs_M": {"workload": "w", "1": {"cold_us": 100.0, "cold_hbm_frac": 0.5}},
    }
    s = bench.summarize(extras, rl, rl, rl)
    assert s["rooflines"]["gate_up"]["frac"] == 0.88
    assert s["router_dsv4_warm_us_fp32frac"] == {"1": [3.7, 0.007]}
    assert s["cublas_fp32_rows_changed_vs_M4096"] == {"1": 1}
    assert s["layer_cold_us_hbmfrac"]["1"] == [100.0, 0.5]


def test_code_digest_ignores_comments_not_code():
    src = 'int f(int a) {  // add one\n  /* block\n comment */ return a + 1;\n}\nconst char *s = "// kept";\n'
    same = 'int f(int a) {\n return a + 1; }   // other words\nconst char *s = "// kept";'
    assert bench.code_digest(src) == bench.code_digest(same)
    assert bench.code_digest(src) != bench.code_digest(src.replace("a + 1", "a + 2"))
    assert bench.code_digest(src) != bench.code_digest(src.replace('"// kept"', '"// gone"'))

