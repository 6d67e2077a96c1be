"""GPU parity of the attention backward (dQ, dK, dV over the selected blocks) against the
CPU oracle on the same seeded inputs and the GPU's own selection.

Tolerance: relative L2 <= 1e-2 per gradient and max-abs <= 2e-2 x max(1, max |oracle|):
the kernels round P and dS to bf16 for the tensor-core products and take D from the
forward's bf16 O, the oracle stays in fp64 throughout."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import workloads as W

pisa = pytest.importorskip("hierarchical_top_block_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _close(name, got, ref):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref).max()
    assert err <= 2e-2 * max(1.0, np.abs(ref).max()), f"{name}: max-abs {err} (max |ref| {np.abs(ref).max()})"
    assert H.rel_l2(got, ref) <= 1e-2, f"{name}: relative L2 {H.rel_l2(got, ref)}"


def _check(oracle_impl, w, K_sel, causal=True, seed=0):
    Q, K, V = W.prefill_inputs(w, "cuda")
    gen = torch.Generator(device="cpu").manual_seed(1234 + seed)
    dO = (torch.randn(Q.shape, generator=gen) * 0.5).to(torch.bfloat16).to("cuda")
    P = pisa.pisa_build_pyramid(K)
    idx = pisa.pisa_select_prefill(Q, K, P, K_sel, causal=causal)
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx, causal=causal)
    dQ, dK, dV = pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, causal=causal)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    rQ, rK, rV = oracle_impl.sparse_attention_backward(H.to_np_bits(Q), H.to_np_bits(K), H.to_np_bits(V),
                                                       idx.cpu().numpy(), H.to_np_bits(dO), causal=causal)
    _close("dQ", dQ.cpu().numpy(), rQ)
    _close("dK", dK.cpu().numpy(), rK)
    _close("dV", dV.cpu().numpy(), rV)


def test_backward_tiny(oracle_impl):
    _check(oracle_impl, W.WORKLOADS["tiny"], 4)


def test_backward_ragged_gq16_d128(oracle_impl):
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=2048 + 33, H_q=32, H_kv=2, K=8)
    _check(oracle_impl, w, 8, seed=1)


def test_backward_non_causal(oracle_impl):
    w = W.WORKLOADS["tiny"].with_(N=64 * 9 + 5, H_q=8, H_kv=2, d=128)
    _check(oracle_impl, w, 3, causal=False, seed=2)


def _planted_selection(N, K_sel, seed):
    """Every query keeps its own block, blocks 0 and 1 (when eligible) and random other eligible
    blocks up to K: blocks 0 and 1 are then selected by every query, more than the 256 queries
    of one dK/dV chunk, so their gradients are summed over many chunks."""
    rng = np.random.default_rng(seed)
    idx = np.full((1, 1, N, K_sel), -1, np.int32)
    for t in range(N):
        own = t // 64
        s = {own} | {b for b in (0, 1) if b <= own}
        others = [int(b) for b in rng.permutation(own + 1) if b not in s]
        s |= set(others[:K_sel - len(s)])
        v = sorted(s)
        idx[0, 0, t, :len(v)] = v
    return idx


def test_backward_multi_chunk_blocks(oracle_impl):
    """G_Q = 16, d = 128, K = 16 (the benchmark's shape) on a selection where 26 blocks are each
    selected by more queries than one dK/dV chunk holds (up to all 2085 queries): the chunked
    accumulation of dK and dV, and dQ over the same blocks, against the oracle in full."""
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=2048 + 37, K=16)
    Q, K, V = W.prefill_inputs(w, "cuda")
    idx_np = _planted_selection(w.N, 16, seed=0)
    assert (np.bincount(idx_np[idx_np >= 0].ravel()) > 256).sum() >= 20
    idx = torch.from_numpy(idx_np).to("cuda")
    gen = torch.Generator(device="cpu").manual_seed(77)
    dO = (torch.randn(Q.shape, generator=gen) * 0.5).to(torch.bfloat16).to("cuda")
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx)
    dQ, dK, dV = pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    rQ, rK, rV = oracle_impl.sparse_attention_backward(H.to_np_bits(Q), H.to_np_bits(K), H.to_np_bits(V), idx_np,
                                                       H.to_np_bits(dO))
    _close("dQ", dQ.cpu().numpy(), rQ)
    _close("dK", dK.cpu().numpy(), rK)
    _close("dV", dV.cpu().numpy(), rV)


def test_backward_k32(oracle_impl):
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=64 * 40 + 9, H_q=16, H_kv=1, K=32)
    _check(oracle_impl, w, 32, seed=3)
