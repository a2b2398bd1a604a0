"""Host logic of bench.py that the JSON line's claims rest on, checked without a GPU."""
import bench


def test_launches_per_step_match_the_ncu_launch_lists():
    # counts seen in the ncu launch lists of the same workloads (profiles/launches_*.md,
    # profiles/dram_traffic_per_launch.md): decode layer 5 (quantize only in front of down),
    # prefill 8 (prep with the quantizer inside + main per GEMM; 12 with a quantize kernel per
    # GEMM), M = 4 mix 10 (a quantize per activation)
    assert bench.launches_per_step(bench.CONFIGS[1]) == 5
    assert bench.launches_per_step(bench.CONFIGS[4]) == 8
    assert bench.launches_per_step(bench.CONFIGS[5]) == 8
    assert bench.launches_per_step(bench.CONFIGS[4], "unfused") == 12
    assert bench.launches_per_step(bench.CONFIGS[4], "batched") == 8
    assert bench.launches_per_step(bench.CONFIGS[3]) == 10
    assert bench.launches_per_step(bench.CONFIGS[2]) == 1
    assert bench.launches_per_step(bench.CONFIGS[6]) == 7
    assert bench.launches_per_step(bench.CONFIGS[1], "unfused") == 8     # 4 activations + 4 GEMVs
    assert bench.launches_per_step(bench.CONFIGS[1], "fused") == 4
    assert bench.launches_per_step(bench.CONFIGS[1], "batched") == 5     # one quantize for all + 4 GEMVs
    assert bench.launches_per_step(bench.CONFIGS[3], "batched") == 6


def test_recorded_traffic_is_keyed_to_existing_kernel_families():
    for (cfg_id, kernel), t in bench.TRAFFIC.items():
        assert cfg_id in bench.CONFIGS
        assert kernel.split("_")[0] in bench.KERNEL_SOURCES
        assert len(t["digest"]) == 16 and t["bytes_per_launch"] > 0
        # a figure is reported only while its kernel family's sources are unchanged
        assert (bench.recorded_traffic(cfg_id, kernel) is not None) == (t["digest"] == bench.kernel_sources_digest(kernel))


def test_weight_bytes_of_the_headline_workloads():
    # Llama-3-8B decode layer in Q4_K: (6144 + 4096 + 28672) x 4096 + 4096 x 14336 weights at 144 B / 256
    assert bench.weight_bytes(bench.CONFIGS[1]) == 122683392
    # Qwen2-7B prefill: 2 M sum(N K) integer ops
    assert bench.int_ops(bench.CONFIGS[4]) == 954556481536


def test_mmq_roofline_counts_the_mmas_of_the_kernel_that_ran():
    # Q4_K: A_hi and A_lo against the exact sc*q operand, plus the min term's 3 MMAs per 64
    # products; Q6_K: three hi/lo products. The f32-input entry points run the same kernels.
    dk = {"calls_per_step": 4, "ms_per_step": 1.0, "ops": 1e12, "avg_us": 250.0}
    peaks = {"tcgen05_f16_tflops": 2000.0}
    for key, per in (("mmq_q4k", 2.0 + 3.0 / 64.0), ("mmq_q4k_f32", 2.0 + 3.0 / 64.0),
                     ("mmq_q6k", 3.0), ("mmq_q6k_f32", 3.0)):
        r = bench.roofline(bench.CONFIGS[4], 4, key, dk, peaks)
        assert r["f16_mma_per_integer_product"] == per
        assert abs(r["issued_mma_utilisation"] - 1000.0 * per / 2000.0) < 1e-9


def test_prefill_traffic_is_recorded_for_the_default_front_end():
    # the bench's default prefill line runs the f32-input MMQ; its DRAM figure must be the one
    # the ncu launch list of that kernel pair measured
    fused = all(bench.gemm_fused("auto", bench.CONFIGS[4], g) for g in bench.CONFIGS[4]["gemms"])
    assert fused
    assert (4, "mmq_q4k_f32") in bench.TRAFFIC
