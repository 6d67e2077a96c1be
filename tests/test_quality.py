"""The selection-quality measurement against the oracle, on the CPU: its exact reference
block sets are the oracle's selection whenever no level prunes (then the method itself is
exact), so Recall@K of the oracle's own selection is 1 there; the kept mass of a selection
that covers every eligible block is 1 (the dense softmax sums to one)."""
import numpy as np
import torch

from hierarchical_top_block_gb300 import quality
import pins


def _as_tensors(Q, K):
    f = lambda x: torch.from_numpy(pins.b2f(x).astype(np.float32))  # noqa: E731
    return f(Q), f(K)


def test_reference_sets_match_the_exact_selection(oracle_impl):
    o = oracle_impl
    Q, K, V = pins._tiny_inputs(seed=31, N=64 * 6, H_q=4, H_kv=2)
    P = o.build_pyramid(K)
    Qt, Kt = _as_tensors(Q, K)
    K_sel = 4                       # g K = 8 >= 6 leaves: no level prunes
    for t in (5, 100, 200, 300, 383):
        for h in range(2):
            ref = o.select(Q, K, P, K_sel, np.array([[0, h, t]]))["idx"][0]
            got = quality.exact_topk_blocks(Qt, Kt, 0, t, K_sel)[h].numpy()
            assert np.array_equal(ref, got), (t, h, ref, got)


def test_recall_and_mass_of_exact_and_dense_selections(oracle_impl):
    o = oracle_impl
    Q, K, V = pins._tiny_inputs(seed=33, N=64 * 6)
    P = o.build_pyramid(K)
    Qt, Kt = _as_tensors(Q, K)
    N = Q.shape[1]
    rows = [(0, t) for t in range(0, N, 41)]
    idx = np.full((1, 1, N, 4), -1, np.int32)
    sel = o.select(Q, K, P, 4, np.array([[0, 0, t] for _, t in rows]))["idx"]
    for (b, t), s in zip(rows, sel):
        idx[0, 0, t] = s
    rep = quality.selection_quality(Qt, Kt, torch.from_numpy(idx), 4, rows)
    assert rep["recall_at_k"] == 1.0
    # K >= the number of leaves: every eligible block is kept, so the kept mass is 1
    idx6 = np.full((1, 1, N, 6), -1, np.int32)
    sel6 = o.select(Q, K, P, 6, np.array([[0, 0, t] for _, t in rows]))["idx"]
    for (b, t), s in zip(rows, sel6):
        idx6[0, 0, t] = s
    rep6 = quality.selection_quality(Qt, Kt, torch.from_numpy(idx6), 6, rows)
    assert abs(rep6["kept_mass"] - 1.0) < 1e-12
    assert rep["kept_mass"] < 1.0
