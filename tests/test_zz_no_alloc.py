"""qk_mmq_q4k_noalloc (static workspace) against qk_mmq_q4k (caller workspace).

Collected last on purpose: it must pass alone and after every other GPU test
(which leave the library loaded and its static array holding old data)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_q8_activation_gb300 as m
    m.build()
    m.lib()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_matches_workspace_entry_point_twice_in_a_row(qk):
    cases = [(300, 200, 1024, True), (2048, 128, 3584, False)]   # the second fills most of the static array
    for (M, N, K, res) in cases:
        w = qk.repack(qk.Q4_K, dev(synth.weights("q4k", N, K, seed=M + N)), N, K)
        codes, scales = qk.quantize_q8_1(dev(synth.activations(M, K, seed=K)))
        r = dev(synth.residual(M, N, seed=N)) if res else None
        y_ref = qk.mmq_q4k(w, codes, scales, N, K, residual=r)
        y1 = qk.mmq_q4k_noalloc(w, codes, scales, N, K, residual=r)
        y2 = qk.mmq_q4k_noalloc(w, codes, scales, N, K, residual=r, pdl=True)   # second call in a row
        torch.cuda.synchronize()
        assert torch.equal(y1, y_ref), (M, N, K)
        assert torch.equal(y2, y_ref), (M, N, K)


def test_noalloc_rejects_oversize(qk):
    M, N, K = 2048, 256, 18944
    assert qk.mmq_workspace_bytes(M, N, K) > qk.STATIC_WS_BYTES
    codes, scales = qk.empty_q8_1(M, K)
    w = torch.empty(qk.repacked_bytes(qk.Q4_K, N, K), dtype=torch.uint8, device="cuda")
    with pytest.raises(qk.QKError) as e:
        qk.mmq_q4k_noalloc(w, codes, scales, N, K)
    assert e.value.status == -6
