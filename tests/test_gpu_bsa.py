"""GPU parity of the BSA flat selection (the single-level baseline of the paper's
selection-speed figure) against the oracle, through the C ABI, on the same seeded inputs."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import hierarchical_top_block_gb300 as pisa
    from hierarchical_top_block_gb300.build import build as _build

    _build()
    import gpu_helpers as H


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(o, w, K_sel, causal=True, sample=None, seed=0):
    Q, K, V = W.prefill_inputs(w, "cuda")
    P = pisa.pisa_build_pyramid(K)
    idx = pisa.pisa_select_bsa(Q, P, K_sel, causal=causal)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    idx = idx.cpu().numpy()
    B, N = w.B, w.N
    if sample is None:
        rows = np.array([(b, g, t) for b in range(B) for g in range(w.H_kv) for t in range(N)], np.int64)
    else:
        rng = np.random.default_rng(seed)
        rows = np.stack([rng.integers(0, B, sample), rng.integers(0, w.H_kv, sample), rng.integers(0, N, sample)], 1)
        rows[:4, 2] = [0, N - 1, min(N - 1, 127), min(N - 1, 128)]
        rows = rows.astype(np.int64)
    Qb = H.to_np_bits(Q)
    Pb = H.to_np_bits(P)
    gi = idx[rows[:, 0], rows[:, 1], rows[:, 2]]
    return H.check_bsa(o, Qb, Pb, K_sel, rows, gi, causal=causal)


@pytest.mark.parametrize("K_sel", [1, 4, 8, 16])
def test_bsa_tiny_all_rows(oracle_impl, K_sel):
    rep = _run(oracle_impl, W.WORKLOADS["tiny"], K_sel)
    assert rep["rows"] == 1024


@pytest.mark.parametrize("N,GQ,H_kv,d,K_sel,causal", [
    (1, 4, 1, 64, 4, True), (63, 2, 2, 128, 3, True), (129, 8, 1, 128, 5, True), (64 * 130 + 7, 16, 1, 128, 16, True),
    (64 * 70 + 1, 1, 2, 64, 16, True), (300, 4, 1, 64, 4, False), (64 * 200 + 5, 16, 1, 128, 8, False),
    (64 * 300 + 9, 16, 1, 128, 32, True), (64 * 90, 4, 2, 64, 20, False),
])
def test_bsa_ragged_shapes(oracle_impl, N, GQ, H_kv, d, K_sel, causal):
    w = W.WORKLOADS["prefill_4k"].with_(B=2, N=N, H_q=GQ * H_kv, H_kv=H_kv, d=d, K=K_sel, needles=0)
    rows = w.B * w.H_kv * w.N
    _run(oracle_impl, w, K_sel, causal=causal, sample=None if rows <= 4096 else 1500, seed=N)


def test_bsa_prefill_4k_sampled(oracle_impl):
    _run(oracle_impl, W.WORKLOADS["prefill_4k"], 16, sample=1024, seed=1)


@pytest.mark.parametrize("K_sel", [8, 16])
def test_bsa_prefill_32k_sampled(oracle_impl, K_sel):
    _run(oracle_impl, W.WORKLOADS["prefill_32k"], K_sel, sample=1024, seed=K_sel)


def test_bsa_prefill_256k_sampled(oracle_impl):
    """The full-size selection-speed workload at the pages' K = 8: sampled rows, every one of
    which ranks up to 4095 blocks."""
    _run(oracle_impl, W.WORKLOADS["prefill_256k"], 8, sample=512, seed=3)
