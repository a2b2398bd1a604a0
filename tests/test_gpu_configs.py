"""Full-size parity at every benchmark configuration, in the launch
configuration bench.py times (programmatic dependent launch, one stream,
the same Workload buffers), on sampled output rows that the oracle computes
one by one."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def sample_rows(N, n=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, 1, N // 3, N // 2, N - 2, N - 1}
    rows.update(int(v) for v in rng.integers(0, N, n))
    return sorted(r for r in rows if 0 <= r < N)


@pytest.mark.parametrize("cfg_id,front_end", [(0, "fused"), (1, "fused"), (2, "fused"), (3, "fused"), (1, "unfused"),
                                              (3, "unfused"), (1, "auto"), (0, "batched"), (1, "batched"),
                                              (2, "batched"), (3, "batched"), (4, "auto"), (5, "auto"), (7, "auto"),
                                              (8, "auto"), (9, "auto"), (10, "auto")])
def test_config_full_size(cfg_id, front_end):
    import bench
    wl = bench.Workload(cfg_id, seed=0, copies=1)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        wl.step(0, pdl=True, stream=stream, front_end=front_end)
        wl.step(0, pdl=True, stream=stream, front_end=front_end)  # twice: PDL chaining across steps
    torch.cuda.synchronize()
    cfg = wl.cfg
    q8 = {}
    quantized = {g[5] for g in cfg["gemms"] if not bench.gemm_fused(front_end, cfg, g)}
    for s, x in wl.host_x.items():
        c, d, sref = oracle.quantize_q8_1(x)
        if s in quantized:
            codes, scales = wl.q8[s]
            sc = scales.cpu().numpy().view(np.uint16)
            assert np.array_equal(codes.cpu().numpy(), c), s
            assert np.array_equal(sc[:, :, 0], d) and np.array_equal(sc[:, :, 1], sref), s
        q8[s] = (c, d)
    for (name, q, N, K, res, s) in cfg["gemms"]:
        y = wl.y[name].cpu().numpy()
        c, d = q8[s]
        r = wl.host_r.get(name)
        qt = {"q4k": oracle.Q4_K, "q5k": oracle.Q5_K, "q6k": oracle.Q6_K, "q80": oracle.Q8_0,
              "q2k": oracle.Q2_K, "q3k": oracle.Q3_K}[q]
        for n in sample_rows(N, seed=N):
            y_ref, ab = oracle.gemm(qt, wl.host_w[name], N, K, c, d, residual=r, rows=(n, n + 1))
            tol = 1e-4 * ab[:, 0] + (0 if r is None else 2.0 ** -22 * np.abs(r[:, n]))
            err = np.abs(y[:, n].astype(np.float64) - y_ref[:, 0])
            assert np.all(err <= tol), f"config {cfg_id} {name} row {n}: max err/tol {np.max(err / tol):.3g}"


def test_decode_chain_with_producers_full_size():
    """The decode layer chained through the fused producers (bench config 6): every stage
    against the oracle applied to the previous stage's device output, at full size."""
    import bench
    import quantized_q8_activation_gb300 as qk
    wl = bench.Workload(6, seed=0, copies=1)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        wl.step(0, pdl=True, stream=stream)
        wl.step(0, pdl=True, stream=stream)
    torch.cuda.synchronize()
    cfg = wl.cfg
    gm = {g[0]: g for g in cfg["gemms"]}
    eps = bench.NORM_EPS

    def check_norm(x_dev, g_host, slot):
        # the producer's codes are the q8_1 of its binary32 output; rerun it with the output kept
        K = x_dev.shape[1]
        y = torch.empty_like(x_dev)
        qk.rmsnorm_q8_1(x_dev, wl.g[g_host], eps, y=y)
        torch.cuda.synchronize()
        y_np = y.cpu().numpy()
        y_ref, _ = oracle.rmsnorm(x_dev.cpu().numpy(), wl.host_g[g_host], eps)
        assert np.all(np.abs(y_np - y_ref) <= (K / 2 + 8) * 2.0 ** -24 * np.abs(y_ref) + 2.0 ** -126)
        c, d, s = oracle.quantize_q8_1(y_np)
        codes, scales = wl.q8[slot]
        sc = scales.cpu().numpy().view(np.uint16)
        assert np.array_equal(codes.cpu().numpy(), c) and np.array_equal(sc[:, :, 0], d)
        assert np.array_equal(sc[:, :, 1], s)

    def check_gemm(name, codes_np, d_np, residual):
        _, q, N, K, _, _ = gm[name]
        y = wl.y[name].cpu().numpy()
        for n in sample_rows(N, seed=N):
            y_ref, ab = oracle.gemm(oracle.Q4_K, wl.host_w[name], N, K, codes_np, d_np, residual=residual,
                                    rows=(n, n + 1))
            tol = 1e-4 * ab[:, 0] + (0 if residual is None else 2.0 ** -22 * np.abs(residual[:, n]))
            assert np.all(np.abs(y[:, n].astype(np.float64) - y_ref[:, 0]) <= tol), f"{name} row {n}"

    def q8_host(slot):
        codes, scales = wl.q8[slot]
        return codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)[:, :, 0].copy()

    check_norm(wl.x["x_attn_in"], "attn", "x_attn_in")
    check_gemm("qkv", *q8_host("x_attn_in"), None)
    c, d, _ = oracle.quantize_q8_1(wl.host_x["x_attn_out"])
    check_gemm("attn_out", c, d, wl.host_r["attn_out"])
    check_norm(wl.y["attn_out"], "ffn", "x_ffn_in")
    check_gemm("gate_up", *q8_host("x_ffn_in"), None)
    F = gm["gate_up"][2] // 2
    h = torch.empty((1, F), dtype=torch.float32, device="cuda")
    qk.swiglu_q8_1(wl.y["gate_up"], F, h=h)
    torch.cuda.synchronize()
    c, d, s = oracle.quantize_q8_1(h.cpu().numpy())
    codes, scales = wl.q8["x_ffn_mid"]
    assert np.array_equal(codes.cpu().numpy(), c)
    check_gemm("down", *q8_host("x_ffn_mid"), wl.y["attn_out"].cpu().numpy())
