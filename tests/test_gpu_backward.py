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


def _check(oracle_impl, w, K_sel, causal=True, seed=0, least_ws=False):
    Q, K, V = W.prefill_inputs(w, "cuda")
    gen = torch.Generator(device="cpu").manual_seed(1234 + seed)
    dO = (torch.randn(Q.shape, generator=gen) * 0.5).to(torch.bfloat16).to("cuda")
    P = pisa.pisa_build_pyramid(K)
    idx = pisa.pisa_select_prefill(Q, K, P, K_sel, causal=causal)
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx, causal=causal)
    ws = None
    if least_ws:  # the least scratch: no dS rows, the dQ kernel forms S and dP again
        shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d, w.N)
        params = pisa.make_params(K_sel, causal)
        least = pisa.pisa_attn_backward_min_workspace_bytes(shape, params)
        assert 0 < least < pisa.pisa_attn_backward_workspace_bytes(shape, params)
        ws = torch.empty(least, dtype=torch.uint8, device="cuda")
    dQ, dK, dV = pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO, causal=causal, ws=ws)
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


def test_backward_ragged_gq16_d128_least_workspace(oracle_impl):
    """The same shape with only the least scratch: dK/dV on tcgen05 without writing dS, and dQ
    forming S and dP itself."""
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=2048 + 33, H_q=32, H_kv=2, K=8)
    _check(oracle_impl, w, 8, seed=1, least_ws=True)


@pytest.mark.parametrize("N,K_sel", [(37, 1), (64 * 3 + 1, 2)])
def test_backward_short_sequences_gq16_d128(oracle_impl, N, K_sel):
    """The tcgen05 path on sequences of one partial block and of a single key past three full
    blocks: K and V rows past N read as zero, partial tiles of a chunk."""
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=N, H_q=16, H_kv=1, K=K_sel)
    _check(oracle_impl, w, K_sel, seed=N)


def test_backward_non_causal(oracle_impl):
    w = W.WORKLOADS["tiny"].with_(N=64 * 9 + 5, H_q=8, H_kv=2, d=128)
    _check(oracle_impl, w, 3, causal=False, seed=2)


def test_backward_non_causal_gq16(oracle_impl):
    # the tensor-core dK/dV path (G_Q = 16, d = 128) without the causal mask, ragged N
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=64 * 12 + 17, H_q=16, H_kv=1, K=5)
    _check(oracle_impl, w, 5, causal=False, seed=4)


def test_backward_gq8_two_sequences(oracle_impl):
    # G_Q = 8 (16 queries a tile on the tensor-core path), two sequences, two KV heads
    w = W.WORKLOADS["prefill_4k"].with_(B=2, N=64 * 20 + 3, H_q=16, H_kv=2, K=7)
    _check(oracle_impl, w, 7, seed=5)


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


def _pick_blocks(idx_np, M1, rng, per_bg, cap_rows):
    """Key blocks to check, per (sequence, KV head): the first and the last block and random
    selected ones across the range of selection counts, while the queries selecting the chosen
    blocks stay within cap_rows in total (the oracle recomputes each of them)."""
    B, H_kv = idx_np.shape[:2]
    out, rows = [], 0
    for bg in range(B * H_kv):
        sel = idx_np.reshape(B * H_kv, -1)[bg]
        cnt = np.bincount(sel[sel >= 0], minlength=M1)
        chosen = [j for j in (0, M1 - 1) if cnt[j] > 0]
        order = np.argsort(cnt, kind="stable")
        picked = [int(j) for j in order[cnt[order] > 0]]
        # spread over the count distribution: quantiles of the selected blocks
        for qn in np.linspace(0.05, 0.95, per_bg):
            chosen.append(picked[int(qn * (len(picked) - 1))])
        chosen += [int(j) for j in rng.choice(picked, size=2, replace=False)]
        for j in dict.fromkeys(chosen):
            if cnt[j] <= cap_rows // 4 and rows + cnt[j] <= cap_rows:
                out.append(bg * M1 + j)
                rows += int(cnt[j])
    return np.array(out, np.int64), rows


def _check_sampled(oracle_impl, w, n_rows, per_bg, cap_rows, seed):
    Q, K, V = W.prefill_inputs(w, "cuda")
    gen = torch.Generator(device="cpu").manual_seed(4321 + seed)
    dO = (torch.randn(Q.shape, generator=gen) * 0.5).to(torch.bfloat16).to("cuda")
    P = pisa.pisa_build_pyramid(K)
    idx = pisa.pisa_select_prefill(Q, K, P, w.K)
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx)
    dQ, dK, dV = pisa.pisa_sparse_attn_backward(Q, K, V, idx, O, LSE, dO)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    N, M1 = w.N, (w.N + 63) // 64
    idx_np = idx.cpu().numpy()
    rng = np.random.default_rng(seed)
    t = np.unique(np.concatenate([rng.choice(N, n_rows, replace=False), [0, 1, 63, 64, 65, N - 64, N - 1]]))
    rows = np.concatenate([b * N + t for b in range(w.B)]).astype(np.int64)
    blocks, nsel = _pick_blocks(idx_np, M1, rng, per_bg, cap_rows)
    assert len(blocks) >= 4 and nsel > 0
    rQ, rK, rV = oracle_impl.sparse_attention_backward_sampled(H.to_np_bits(Q), H.to_np_bits(K), H.to_np_bits(V),
                                                               idx_np, H.to_np_bits(dO), rows, blocks)
    gQ = dQ.reshape(w.B * N, w.H_q, w.d)[torch.from_numpy(rows).to("cuda")].cpu().numpy()
    _close("dQ (sampled positions)", gQ, rQ)
    bg, j = blocks // M1, blocks % M1
    keys = (j[:, None] * 64 + np.arange(64)[None, :])
    valid = keys < N
    gK = dK.reshape(w.B * w.H_kv, N, w.d).cpu().numpy()
    gV = dV.reshape(w.B * w.H_kv, N, w.d).cpu().numpy()
    kk = np.minimum(keys, N - 1)
    _close("dK (sampled blocks)", gK[bg[:, None], kk][valid], rK[valid])
    _close("dV (sampled blocks)", gV[bg[:, None], kk][valid], rV[valid])


def test_backward_32k_sampled(oracle_impl):
    """The benchmark's 32K shape (B = 1, N = 32768, H_q = 32, H_kv = 2, d = 128, K = 16) on the
    GPU's own selection, through the full-size chunked path: dQ on about 1000 sampled positions
    (every head) and dK, dV of key blocks across the range of selection counts (the first and
    last block included), against the oracle's sampled backward."""
    _check_sampled(oracle_impl, W.WORKLOADS["prefill_32k"], n_rows=1000, per_bg=5, cap_rows=4000, seed=5)


def test_backward_256k_sampled(oracle_impl):
    """The bench's 256K shape (B = 1, N = 262144, H_q = 16, H_kv = 1, d = 128, K = 16): dQ on
    about 500 sampled positions and dK, dV of a few key blocks, as above."""
    _check_sampled(oracle_impl, W.WORKLOADS["prefill_256k"], n_rows=500, per_bg=5, cap_rows=12000, seed=6)
