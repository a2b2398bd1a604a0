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
                                              (3, "unfused"), (1, "auto"), (4, "auto"), (5, "auto")])
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
        qt = oracle.Q4_K if q == "q4k" else oracle.Q6_K
        for n in sample_rows(N, seed=N):
            y_ref, ab = oracle.gemm(qt, wl.host_w[name], N, K, c, d, residual=r, rows=(n, n + 1))
            tol = 1e-4 * ab[:, 0] + (0 if r is None else 2.0 ** -22 * np.abs(r[:, n]))
            err = np.abs(y[:, n].astype(np.float64) - y_ref[:, 0])
            assert np.all(err <= tol), f"config {cfg_id} {name} row {n}: max err/tol {np.max(err / tol):.3g}"
