"""The keys a causal chunk's selection reads (CPU, with the oracle).

The host-buffer prefill copies K in per-chunk slices and builds the pyramid over each slice as
it arrives, so the selection of queries t < T must not depend on keys at or past a prefix x(T):
the level walk reads the child summaries of a candidate only at levels where more than K
candidates can be eligible (summary page of "Block Sparse Attention with Log-Linear
Complexity", section "Method step details", step 2: a level is scored when more than K nodes
remain), those candidates start at or before t, and Stage 2 reads the keys of level-2 nodes
that start at or before t.  Here the keys at and past x(T) are replaced by large values, which
changes every pyramid node over them (the root included), and the oracle's selection of the
chunk's queries must stay the same; a shorter cut must change some of them, so the test can
fail.
"""
import numpy as np
import pytest
import torch

import workloads as W


def key_prefix(T: int, K: int, N: int) -> int:
    """End of the keys the causal selection of queries t < T reads (the rule the host pipeline
    uses): the end of the last eligible node at the highest level l >= 2 with more than K
    eligible nodes (2^(l+5) keys a node), or of the last eligible level-2 node."""
    m, L = (N + 63) // 64, 1
    while m > 1:
        m, L = (m + 1) // 2, L + 1
    x = (((T - 1) >> 7) + 1) << 7
    for l in range(2, L):  # the levels the walk may score
        cnt = ((T - 1) >> (l + 5)) + 1
        if cnt > K:
            x = max(x, cnt << (l + 5))
    return min(x, N)


def _rows(T, n, rng):
    t = np.unique(np.concatenate([np.arange(max(0, T - 8), T), rng.integers(0, T, n)]))
    return np.stack([np.zeros_like(t), np.zeros_like(t), t], axis=1).astype(np.int64)


def _garbled(Kb, x, rng):
    # every key from x on is one large vector of random signs: a node mean over any of them is
    # pulled far along it, so the scores of the nodes that hold them change for every query
    K2 = Kb.copy()
    if x < K2.shape[2]:
        sign = np.where(rng.random(K2.shape[-1]) < 0.5, -60.0, 60.0).astype(np.float32)
        big = np.broadcast_to(sign, K2[:, :, x:].shape).copy()
        K2[:, :, x:] = W.bits(torch.from_numpy(big).to(torch.bfloat16))
    return K2


@pytest.mark.parametrize("K_sel", [1, 2, 4, 16])
def test_selection_ignores_keys_past_the_prefix(oracle_impl, K_sel):
    o = oracle_impl
    w = W.WORKLOADS["tiny"].with_(N=20000, K=K_sel)
    Q, K, _ = W.prefill_inputs(w)
    Qb, Kb = W.bits(Q), W.bits(K)
    P = o.build_pyramid(Kb)
    rng = np.random.default_rng(K_sel)
    shorter_changed = False
    for T in (1000, 4096, 8000, 12345):
        x = key_prefix(T, K_sel, w.N)
        assert T <= x <= w.N
        rows = _rows(T, 40, rng)
        ref = o.select(Qb, Kb, P, K_sel, rows)["idx"]
        K2 = _garbled(Kb, x, rng)
        got = o.select(Qb, K2, o.build_pyramid(K2), K_sel, rows)["idx"]
        assert np.array_equal(got, ref), (T, x)
        # the keys past T that the rule keeps are read: cut at the last level-2 node instead
        x2 = min(w.N, (((T - 1) >> 7) + 1) << 7)
        if x2 < x:
            K3 = _garbled(Kb, x2, rng)
            alt = o.select(Qb, K3, o.build_pyramid(K3), K_sel, rows)["idx"]
            shorter_changed |= not np.array_equal(alt, ref)
    # levels above the leaf pairs are scored for these chunks; at K = 1 the causal selection is
    # the own block alone whatever the scores, so no cut can change it
    if 2 <= K_sel <= 4:
        assert shorter_changed


def test_prefix_is_monotone_and_reaches_n():
    for N in (4096, 20000, 35000, 262144):
        for K_sel in (1, 4, 16, 32):
            prev = 0
            for T in range(64, N + 1, max(64, N // 97)):
                x = key_prefix(T, K_sel, N)
                assert prev <= x <= N and x >= min(N, T)
                prev = x
            assert key_prefix(N, K_sel, N) == N
