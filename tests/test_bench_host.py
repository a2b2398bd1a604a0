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
