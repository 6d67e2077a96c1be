"""GPU parity: the CUDA path through the C ABI against the oracle on the same seeded inputs."""
import math

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


def _inputs(w, device="cuda"):
    return W.prefill_inputs(w, device)


@pytest.fixture(scope="module", autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_generator_identical_on_gpu():
    w = W.WORKLOADS["prefill_4k"].with_(B=2, N=777, H_kv=2, H_q=8)
    for (a, b) in zip(W.prefill_inputs(w, "cuda"), W.prefill_inputs(w, "cpu")):
        assert torch.equal(a.cpu().view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("K_sel", [4, 8, 16])
def test_tiny_all_rows(oracle_impl, K_sel):
    w = W.WORKLOADS["tiny"].with_(K=K_sel)
    Q, K, V = _inputs(w)
    rep = H.full_prefill_check(oracle_impl, Q, K, V, K_sel)
    assert rep["rows"] == w.N


@pytest.mark.parametrize("N,GQ,H_kv,d,K_sel", [
    (1, 4, 1, 64, 4), (63, 4, 1, 64, 4), (64, 2, 2, 128, 2), (65, 8, 1, 128, 3), (130, 1, 2, 64, 1),
    (64 * 37 + 11, 16, 1, 128, 5), (64 * 70 + 1, 8, 2, 64, 16), (2048 + 64 * 9 + 33, 16, 1, 128, 16),
])
def test_ragged_shapes_all_rows(oracle_impl, N, GQ, H_kv, d, K_sel):
    w = W.WORKLOADS["prefill_4k"].with_(B=2, N=N, H_q=GQ * H_kv, H_kv=H_kv, d=d, K=K_sel, needles=min(3, max(0, N // 200)))
    Q, K, V = _inputs(w)
    rows = w.B * w.H_kv * w.N
    H.full_prefill_check(oracle_impl, Q, K, V, K_sel, sample=None if rows <= 4096 else 1500, seed=N)


@pytest.mark.parametrize("d,GQ", [(64, 4), (128, 16), (128, 4)])
def test_non_causal(oracle_impl, d, GQ):
    w = W.WORKLOADS["tiny"].with_(N=64 * 20 + 7, d=d, H_q=GQ, H_kv=1)
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, 4, causal=False)


def test_prefill_4k_sampled(oracle_impl):
    w = W.WORKLOADS["prefill_4k"]
    Q, K, V = _inputs(w)
    rep = H.full_prefill_check(oracle_impl, Q, K, V, w.K, sample=768, seed=2)
    assert rep["rows"] == 768


def test_dense_when_K_covers_all_leaves(oracle_impl):
    """K >= ceil(N/C): every eligible leaf is selected, so the output is dense causal attention."""
    w = W.WORKLOADS["tiny"].with_(N=64 * 12 + 5, K=13)
    Q, K, V = _inputs(w)
    res = H.run_gpu_prefill(Q, K, V, 13)
    N = w.N
    for t in (0, 63, 64, 300, N - 1):
        sel = [x for x in res["idx"][0, 0, t] if x >= 0]
        assert sel == list(range(t // 64 + 1))
    Qf, Kf, Vf = Q[0].double().cpu().numpy(), K[0, 0].double().cpu().numpy(), V[0, 0].double().cpu().numpy()
    O = res["O"][0].float().cpu().numpy()
    for t in (0, 100, N - 1):
        for h in range(w.H_q):
            z = Qf[t, h] @ Kf[: t + 1].T / math.sqrt(w.d)
            p = np.exp(z - z.max())
            ref = (p / p.sum()) @ Vf[: t + 1]
            assert np.abs(O[t, h] - ref).max() <= H.ATTN_MAX_ABS


def test_bad_index_is_reported_not_faulted():
    w = W.WORKLOADS["tiny"]
    Q, K, V = _inputs(w)
    idx = torch.full((1, 1, w.N, 4), -1, dtype=torch.int32, device="cuda")
    idx[..., 0] = torch.arange(w.N, device="cuda", dtype=torch.int32) // 64
    idx[0, 0, 100, 1] = 10_000  # out of range
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 5
    assert pisa.pisa_get_last_device_error() == 0  # cleared by the read
    assert torch.isfinite(LSE).all()


def test_bounded_wait_times_out_and_the_device_stays_usable(oracle_impl):
    """The timeout path of the bounded waits: a CTA holding tensor memory waits on an mbarrier that
    nothing completes, with a 1 ms limit; it gives up, frees the tensor memory and returns, the
    error word reads PISA_ERR_TIMEOUT (cleared by the read), and the library's kernels still run
    and match the oracle afterwards."""
    import time

    assert pisa.pisa_get_last_device_error() == 0
    t0 = time.perf_counter()
    pisa.pisa_check_wait_timeout(1_000_000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert pisa.pisa_get_last_device_error() == 4
    assert pisa.pisa_get_last_device_error() == 0
    w = W.WORKLOADS["tiny"]
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, w.K, sample=128, seed=5)


def test_argument_errors_are_synchronous():
    w = W.WORKLOADS["tiny"]
    Q, K, V = _inputs(w)
    with pytest.raises(pisa.PisaError):
        pisa.pisa_select_prefill(Q, K, pisa.pisa_build_pyramid(K), 33)  # K > 32 unsupported
    assert pisa.pisa_get_last_device_error() == 0


@pytest.mark.parametrize("K_sel", [16, 8])
def test_prefill_32k_sampled(oracle_impl, K_sel):
    """The long-prefill workload at its own K and at K = 8 (both timed by the benchmark)."""
    w = W.WORKLOADS["prefill_32k"]
    Q, K, V = _inputs(w)
    rep = H.full_prefill_check(oracle_impl, Q, K, V, K_sel, sample=192, seed=3 + K_sel)
    assert rep["rows"] == 192


@pytest.mark.parametrize("K_sel", [16, 8])
def test_prefill_256k_sampled(oracle_impl, K_sel):
    """Full selection-scale size, the launch configuration the benchmark times (at the
    workload's K and at K = 8); the oracle computes sampled rows one by one.  Q is generated on
    the GPU and, for the sampled rows only, on the CPU; K and V are generated on both and
    compared bit for bit."""
    w = W.WORKLOADS["prefill_256k"]
    Q = W.make_q(w, "cuda")
    K = W.make_kv(w, "K", "cuda")
    V = W.make_kv(w, "V", "cuda")
    res = H.run_gpu_prefill(Q, K, V, K_sel)
    Kc, Vc = W.make_kv(w, "K", "cpu"), W.make_kv(w, "V", "cpu")
    assert torch.equal(K.cpu().view(torch.int16), Kc.view(torch.int16))
    assert torch.equal(V.cpu().view(torch.int16), Vc.view(torch.int16))
    Kb, Vb = W.bits(Kc), W.bits(Vc)
    Pb = oracle_impl.build_pyramid(Kb)
    assert np.array_equal(W.bits(res["P"]), Pb)
    rng = np.random.default_rng(4)
    # selection on 256 rows, attention on 2048 (the selection rows among them)
    ts = np.concatenate([[0, 63, 64, w.N - 1, w.N - 65], rng.integers(0, w.N, 251)]).astype(np.int64)
    ta = np.unique(np.concatenate([ts, rng.integers(0, w.N, 2048 - ts.size)])).astype(np.int64)
    Qb = np.zeros((1, w.N, w.H_q, w.d), np.uint16)
    qrows = W.q_rows(w, 0, ta)
    Qb[0, ta] = W.bits(qrows)
    assert torch.equal(Q[0, torch.as_tensor(ta, device="cuda")].cpu().view(torch.int16), qrows.view(torch.int16))
    rows = np.stack([np.zeros_like(ts), np.zeros_like(ts), ts], 1)
    H.check_selection(oracle_impl, Qb, Kb, Pb, K_sel, rows, res["idx"][0, 0, ts], res["s2"][0, 0, ts],
                      res["score"][0, 0, ts])
    bt = np.stack([np.zeros_like(ta), ta], 1)
    assert len(bt) >= 2000
    O = res["O"][0, torch.as_tensor(bt[:, 1], device="cuda")].float().cpu().numpy()
    LSE = res["LSE"][0][:, bt[:, 1]].T
    H.check_attention(oracle_impl, Qb, Kb, Vb, res["idx"], bt, O, LSE)


def _decode_check(o, w, N0, steps, N_cap, pairs=None, scoring=0):
    """Runs the GPU decode for `steps` steps from N0 cached tokens and checks every step on
    the (sequence, KV head) pairs given: the pyramid cache (bit-exact), idx (gap rule) and
    o / lse.  The oracle runs each pair as its own one-sequence, one-KV-head problem."""
    B, H_q, H_kv, d, K_sel = w.B, w.H_q, w.H_kv, w.d, w.K
    G = H_q // H_kv
    wk = w.with_(N=N0)
    Kc = torch.zeros(B, H_kv, N_cap, d, dtype=torch.bfloat16, device="cuda")
    Vc = torch.zeros_like(Kc)
    for b in range(B):
        for g in range(H_kv):
            Kc[b, g, :N0] = W.kv_slice(wk, "K", b, g, device="cuda")
            Vc[b, g, :N0] = W.kv_slice(wk, "V", b, g, device="cuda")
    Pc = pisa.pisa_build_pyramid(Kc, N=N0)
    seq = torch.full((B,), N0, dtype=torch.int32, device="cuda")
    pairs = [(b, g) for b in range(B) for g in range(H_kv)] if pairs is None else pairs
    ref = {}
    for b, g in pairs:
        kc = np.zeros((1, 1, N_cap, d), np.uint16)
        vc = np.zeros((1, 1, N_cap, d), np.uint16)
        kc[0, 0, :N0] = W.bits(W.kv_slice(wk, "K", b, g))
        vc[0, 0, :N0] = W.bits(W.kv_slice(wk, "V", b, g))
        pc = o.build_pyramid(kc, N=N0)
        assert H.pyramid_equal(W.bits(Pc[b, g]), pc[0, 0], N0, N_cap), "initial pyramid cache differs"
        ref[(b, g)] = [kc, vc, pc, np.array([N0], np.int32)]
    for s in range(steps):
        q, k, v = W.decode_step_inputs(w, s, "cuda")
        out = torch.empty(B, H_q, d, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, H_q, dtype=torch.float32, device="cuda")
        idx = torch.empty(B, H_kv, K_sel, dtype=torch.int32, device="cuda")
        pisa.pisa_decode_step(q, k, v, Kc, Vc, Pc, seq, K_sel, o=out, lse=lse, idx_out=idx, scoring=scoring)
        torch.cuda.synchronize()
        assert pisa.pisa_get_last_device_error() == 0
        qn, kn, vn = W.bits(q), W.bits(k), W.bits(v)
        for (b, g), (kc, vc, pc, sl) in ref.items():
            T = int(sl[0])
            ro, rl, ri = o.decode_step(qn[b:b + 1, g * G:(g + 1) * G].copy(), kn[b:b + 1, g:g + 1].copy(),
                                       vn[b:b + 1, g:g + 1].copy(), kc, vc, pc, sl, K_sel, scoring=scoring)
            assert H.pyramid_equal(W.bits(Pc[b, g]), pc[0, 0], T + 1, N_cap), f"pyramid cache differs at step {s}, pair {(b, g)}"
            gi = idx[b, g].cpu().numpy()
            if not np.array_equal(gi, ri[0, 0]):
                n = T + 1
                Qp = np.zeros((1, n, G, d), np.uint16)
                Qp[0, T] = qn[b, g * G:(g + 1) * G]
                Kp = kc[:, :, :n].copy()
                H.check_selection(o, Qp, Kp, o.build_pyramid(Kp), K_sel, np.array([(0, 0, T)], np.int64), gi[None],
                                  scoring=scoring)
            go = out[b, g * G:(g + 1) * G].float().cpu().numpy()
            assert np.abs(go - ro[0]).max() <= H.ATTN_MAX_ABS, (s, b, g, np.abs(go - ro[0]).max())
            assert H.rel_l2(go, ro[0]) <= H.ATTN_REL_L2
            assert np.abs(lse[b, g * G:(g + 1) * G].cpu().numpy() - rl[0]).max() <= H.ATTN_MAX_ABS
    assert torch.equal(seq.cpu(), torch.full((B,), N0 + steps, dtype=torch.int32))


def test_decode_small_all_sequences(oracle_impl):
    # 2040 cached tokens: the steps cross a leaf boundary (2048) and a level change (M_1 32 -> 33)
    w = W.WORKLOADS["decode_128k"].with_(B=3, H_q=8, H_kv=2, K=6)
    _decode_check(oracle_impl, w, N0=2040, steps=24, N_cap=2304)


def test_decode_gq16_d64(oracle_impl):
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=16, H_kv=1, d=64, K=16)
    _decode_check(oracle_impl, w, N0=64 * 9 + 60, steps=10, N_cap=1024)


def test_decode_fullsize_sampled(oracle_impl):
    """The batched decode workload at full size (64 x 131072 cached tokens), two steps,
    compared on 16 (sequence, KV head) pairs spread over the batch and every KV head."""
    w = W.WORKLOADS["decode_128k"]
    pairs = [(4 * i + (i % 3), i % w.H_kv) for i in range(16)]
    _decode_check(oracle_impl, w, N0=w.N, steps=2, N_cap=w.N + w.decode_steps, pairs=pairs)


def test_decode_gq16_d128(oracle_impl):
    # both head tiles of the level walk (G_Q = 16) at d = 128, crossing a leaf boundary
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=16, H_kv=1, d=128, K=16)
    _decode_check(oracle_impl, w, N0=64 * 37 + 61, steps=6, N_cap=4096)


def test_decode_full_cache_is_refused():
    """A sequence whose cache is full is reported and left untouched; the others step."""
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=8, H_kv=2, K=4)
    N0, N_cap = 300, 320
    Kc = torch.zeros(w.B, w.H_kv, N_cap, w.d, dtype=torch.bfloat16, device="cuda")
    wk = w.with_(N=N_cap)
    for b in range(w.B):
        for g in range(w.H_kv):
            Kc[b, g] = W.kv_slice(wk, "K", b, g, device="cuda")
    Vc = Kc.clone()
    Pc = pisa.pisa_build_pyramid(Kc, N=N_cap)
    seq = torch.tensor([N_cap, N0], dtype=torch.int32, device="cuda")
    K0, V0, P0 = Kc.clone(), Vc.clone(), Pc.clone()
    q, k, v = W.decode_step_inputs(w, 0, "cuda")
    pisa.pisa_decode_step(q, k, v, Kc, Vc, Pc, seq, w.K)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 5
    assert torch.equal(Kc[0], K0[0]) and torch.equal(Vc[0], V0[0]) and torch.equal(Pc[0], P0[0])
    assert torch.equal(Kc[1, :, N0], k[1].to(Kc.dtype)) and not torch.equal(Kc[1], K0[1])
    assert seq.tolist() == [N_cap, N0 + 1]


# ---- the ablation scorings: PISA-1 (log m + mean) and PISA-2 (+ variance / 2) ----------------
@pytest.mark.parametrize("scoring", [1, 2])
def test_scoring_variants_tiny_all_rows(oracle_impl, scoring):
    w = W.WORKLOADS["tiny"]
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, 8, scoring=scoring)


@pytest.mark.parametrize("scoring", [1, 2])
def test_scoring_variants_prefill_4k_sampled(oracle_impl, scoring):
    w = W.WORKLOADS["prefill_4k"]
    Q, K, V = _inputs(w)
    rep = H.full_prefill_check(oracle_impl, Q, K, V, w.K, sample=512, seed=5 + scoring, scoring=scoring)
    assert rep["rows"] == 512


def test_scoring_variant_ragged_d128(oracle_impl):
    N, GQ, H_kv, d, K_sel = 64 * 37 + 11, 8, 2, 128, 5
    w = W.WORKLOADS["tiny"].with_(N=N, H_q=GQ * H_kv, H_kv=H_kv, d=d, K=K_sel)
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, K_sel, sample=1200, seed=N, scoring=2)


@pytest.mark.parametrize("scoring", [1, 2])
def test_decode_scoring_variants(oracle_impl, scoring):
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=8, H_kv=2, K=6)
    _decode_check(oracle_impl, w, N0=2040, steps=12, N_cap=2304, scoring=scoring)


@pytest.mark.parametrize("case", ["4k_b2", "35000_b2_chunked", "35000_noncausal_pisa2_chunked", "20000_d64_k4_chunked",
                                  "35000_k32_chunked"])
def test_prefill_host_matches_the_device_path(case):
    """The whole prefill from pinned host buffers (the end-to-end entry point) returns exactly
    what the device-resident calls return on the same inputs.  The 35000-token cases run as six
    query chunks (4096, 8192, 5184, 5240, 8192, 4096) with two sequences per batch, so the
    chunked copies of Q, O, LSE and the selection rows are all strided; the last one also
    selects without the causal mask (every block of the sequence is a candidate for every
    chunk) and with the PISA-2 block score.  The device scratch starts as all-ones bytes (NaN
    in bf16 and fp32): in causal mode V arrives in the same chunks as Q, and a V row read
    before its chunk's copy would put NaN into O."""
    causal, scoring = True, 0
    if case == "4k_b2":
        w = W.WORKLOADS["prefill_4k"].with_(B=2)
    elif case == "20000_d64_k4_chunked":  # d = 64, G_Q = 4, K = 4: chunks 4096, 3904, 3968, 3936, 4096
        w = W.WORKLOADS["tiny"].with_(N=20000)
    else:
        w = W.WORKLOADS["prefill_32k"].with_(B=2, N=35000, H_q=8, H_kv=2)
        if case == "35000_noncausal_pisa2_chunked":
            causal, scoring = False, 2
        if case == "35000_k32_chunked":  # two candidates per lane in every chunk
            w = w.with_(K=32)
    Q, K, V = _inputs(w)
    P = pisa.pisa_build_pyramid(K)
    idx = pisa.pisa_select_prefill(Q, K, P, w.K, causal=causal, scoring=scoring)
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx, causal=causal)
    torch.cuda.synchronize()
    Qh, Kh, Vh = (x.cpu().pin_memory() for x in (Q, K, V))
    Oh = torch.empty(Q.shape, dtype=torch.bfloat16).pin_memory()
    Lh = torch.empty(LSE.shape, dtype=torch.float32).pin_memory()
    Ih = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
    shape = pisa.make_shape(w.B, w.N, w.H_q, w.H_kv, w.d, w.N)
    params = pisa.make_params(w.K, causal, 0.0, scoring=scoring)
    ws = torch.full((pisa.pisa_prefill_host_workspace_bytes(shape, params),), 0xFF, dtype=torch.uint8, device="cuda")
    pisa.pisa_prefill_host(Qh, Kh, Vh, w.K, causal=causal, dev_ws=ws, O_host=Oh, LSE_host=Lh, idx_host=Ih,
                           scoring=scoring)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    assert torch.equal(Ih, idx.cpu())
    assert torch.equal(Oh, O.cpu())
    assert torch.equal(Lh, LSE.cpu())


# ---- K up to 32 (the pages' continued-pretraining setting): 2K candidates, two per lane -----
@pytest.mark.parametrize("N,GQ,H_kv,d,K_sel", [
    (16384 + 37, 16, 1, 128, 32),    # levels with 64 candidates are scored (walk, top-K, attention)
    (64 * 200 + 5, 8, 2, 64, 24),
    (64 * 150, 4, 1, 128, 17),
])
def test_k_up_to_32_sampled(oracle_impl, N, GQ, H_kv, d, K_sel):
    w = W.WORKLOADS["prefill_4k"].with_(B=1, N=N, H_q=GQ * H_kv, H_kv=H_kv, d=d, K=K_sel, needles=4)
    Q, K, V = _inputs(w)
    rep = H.full_prefill_check(oracle_impl, Q, K, V, K_sel, sample=768, seed=K_sel)
    assert rep["rows"] == 768


def test_k32_tiny_all_rows_dense(oracle_impl):
    """K = 32 >= M_1 = 16: every eligible leaf is selected (dense causal attention)."""
    w = W.WORKLOADS["tiny"].with_(K=32)
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, 32)


@pytest.mark.parametrize("N,d,K_sel", [(64 * 40 + 3, 64, 32), (64 * 150 + 17, 128, 20)])
def test_k_up_to_32_non_causal(oracle_impl, N, d, K_sel):
    """Without the mask every leaf is a candidate; 64-candidate levels at N > 64 * 128."""
    w = W.WORKLOADS["tiny"].with_(N=N, d=d, H_q=8, H_kv=2)
    Q, K, V = _inputs(w)
    H.full_prefill_check(oracle_impl, Q, K, V, K_sel, causal=False, sample=600, seed=N)


def test_decode_k32_d64_gq16(oracle_impl):
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=16, H_kv=1, d=64, K=32)
    _decode_check(oracle_impl, w, N0=64 * 140 + 60, steps=5, N_cap=16384)


def test_decode_k32(oracle_impl):
    # 64 candidates at the scored levels of the walk and 64 leaf slots
    w = W.WORKLOADS["decode_128k"].with_(B=2, H_q=8, H_kv=2, K=32)
    _decode_check(oracle_impl, w, N0=64 * 160 + 50, steps=4, N_cap=16384)


@pytest.mark.parametrize("H_q,H_kv,d,K_sel,N0", [(8, 2, 128, 6, 2040), (16, 1, 128, 16, 64 * 37 + 61),
                                                 (16, 1, 64, 32, 64 * 40 + 5), (4, 4, 128, 16, 3000)])
def test_decode_kept_logits_equal_recomputed(H_q, H_kv, d, K_sel, N0):
    """The decode step that keeps the leaf scoring's logits for the attention (pisa_decode_step_ws)
    gives the same o, lse, idx, caches and lengths, bit for bit, as the one that reads the
    selected blocks' K rows again (G_Q 4, 16 and 1; d 128 and 64; K up to 32; leaf boundaries
    crossed)."""
    w = W.WORKLOADS["decode_128k"].with_(B=3, H_q=H_q, H_kv=H_kv, d=d, K=K_sel)
    N_cap = N0 + 128
    wk = w.with_(N=N0)
    Kc = torch.zeros(w.B, H_kv, N_cap, d, dtype=torch.bfloat16, device="cuda")
    Vc = torch.zeros_like(Kc)
    for b in range(w.B):
        for g in range(H_kv):
            Kc[b, g, :N0] = W.kv_slice(wk, "K", b, g, device="cuda")
            Vc[b, g, :N0] = W.kv_slice(wk, "V", b, g, device="cuda")
    Pc = pisa.pisa_build_pyramid(Kc, N=N0)
    seq = torch.full((w.B,), N0, dtype=torch.int32, device="cuda")
    state = {kept: [Kc.clone(), Vc.clone(), Pc.clone(), seq.clone()] for kept in (False, True)}
    for s in range(70):  # crosses the leaf boundaries after N0
        q, k, v = W.decode_step_inputs(w, s, "cuda")
        outs = {}
        for kept, (kc, vc, pc, sl) in state.items():
            o = torch.empty(w.B, H_q, d, dtype=torch.bfloat16, device="cuda")
            lse = torch.empty(w.B, H_q, dtype=torch.float32, device="cuda")
            idx = torch.empty(w.B, H_kv, K_sel, dtype=torch.int32, device="cuda")
            pisa.pisa_decode_step(q, k, v, kc, vc, pc, sl, K_sel, o=o, lse=lse, idx_out=idx, keep_logits=kept)
            outs[kept] = (o, lse, idx)
        torch.cuda.synchronize()
        assert pisa.pisa_get_last_device_error() == 0
        for a, b in zip(outs[False], outs[True]):
            assert torch.equal(a, b), s
    for a, b in zip(state[False], state[True]):
        assert torch.equal(a, b)
