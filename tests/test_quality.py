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


def test_needle_hit_rate_counts_rows():
    """Hand-built selections: a row hits when its set holds the needle key's block."""
    idx = torch.full((2, 1, 300, 3), -1, dtype=torch.int32)
    idx[0, 0, 200] = torch.tensor([0, 2, 3], dtype=torch.int32)      # holds block 2 (key 130)
    idx[0, 0, 250] = torch.tensor([1, 3, -1], dtype=torch.int32)     # does not
    idx[1, 0, 299] = torch.tensor([2, 4, -1], dtype=torch.int32)     # holds block 2 (key 191)
    targets = [(0, 0, 130, 200), (0, 0, 130, 250), (1, 0, 191, 299), (1, 0, 192, 299)]
    assert quality.needle_hit_rate(idx, targets) == {"rows": 4, "hit_rate": 0.5}
    assert quality.needle_hit_rate(idx, []) == {"rows": 0, "hit_rate": None}


def test_needle_hit_rate_equals_the_exact_reference_without_pruning(oracle_impl):
    """On the small needle workload with g K >= M_1 nothing is pruned, so the oracle's needle
    hits are those of the exact top-K reference, which holds every planted needle there."""
    import workloads as W
    o = oracle_impl
    w = W.WORKLOADS["tiny"]                       # 16 leaves, 2 needles x 8 aimed rows
    Q, K, V = W.prefill_inputs(w, "cpu")
    Qb, Kb = (x.contiguous().view(torch.int16).numpy().view(np.uint16) for x in (Q, K))
    nl = W.needles(w)
    targets = [(n.b, n.g, n.pos, t) for n in nl for (t, _h) in n.rows]
    rows = np.array([(b, g, t) for (b, g, _p, t) in targets], np.int64)
    K_sel = 8
    sel = o.select(Qb, Kb, o.build_pyramid(Kb), K_sel, rows)["idx"]
    idx = torch.full((w.B, w.H_kv, w.N, K_sel), -1, dtype=torch.int32)
    idx[rows[:, 0], rows[:, 1], rows[:, 2]] = torch.from_numpy(sel)
    ref = torch.full_like(idx, -1)
    for b, g, t in rows:
        ref[b, g, t] = quality.exact_topk_blocks(Q, K, int(b), int(t), K_sel)[g].to(torch.int32)
    assert torch.equal(idx, ref)
    assert quality.needle_hit_rate(idx, targets) == quality.needle_hit_rate(ref, targets) == {"rows": 16, "hit_rate": 1.0}
