"""Needle-hit rate of the GPU selection against the oracle's, on the query rows each planted
needle was aimed at (4K and 32K needle workloads; K = 16, and K = 8 at 32K).  Both selections
are checked row by row with the parity rule (identical where every level's K-th gap is at
least 1e-3, an admissible top-K elsewhere), so the two rates may differ only by the share of
rows where the sets differ.  The rate itself is a statistic, not a pin: coarse levels can
prune a needle whose block the exact top-K holds."""
import numpy as np
import pytest
import torch

import gpu_helpers as H
import workloads as W
from hierarchical_top_block_gb300 import quality


def needle_rows(w):
    targets = [(n.b, n.g, n.pos, t) for n in W.needles(w) for (t, _h) in n.rows]
    return targets, np.array([(b, g, t) for (b, g, _p, t) in targets], np.int64)


@pytest.mark.gpu
@pytest.mark.parametrize("name,K_sel", [("prefill_4k", 16), ("prefill_32k", 16), ("prefill_32k", 8)])
def test_needle_hit_rate_matches_the_oracle(oracle_impl, name, K_sel):
    w = W.WORKLOADS[name]
    Q, K, V = W.prefill_inputs(w, "cuda")
    res = H.run_gpu_prefill(Q, K, V, K_sel)
    targets, rows = needle_rows(w)
    Qb, Kb = H.to_np_bits(Q), H.to_np_bits(K)
    Pb = oracle_impl.build_pyramid(Kb)
    sl = (rows[:, 0], rows[:, 1], rows[:, 2])
    rep = H.check_selection(oracle_impl, Qb, Kb, Pb, K_sel, rows, res["idx"][sl], res["s2"][sl], res["score"][sl])
    ref = np.full_like(res["idx"], -1)
    ref[sl] = oracle_impl.select(Qb, Kb, Pb, K_sel, rows)["idx"]
    r_gpu = quality.needle_hit_rate(torch.from_numpy(res["idx"]), targets)["hit_rate"]
    r_ref = quality.needle_hit_rate(torch.from_numpy(ref), targets)["hit_rate"]
    assert abs(r_gpu - r_ref) <= rep["ambiguous"] / len(rows) + 1e-12, (r_gpu, r_ref, rep)
    print(f"{name} K={K_sel}: needle-hit rate GPU {r_gpu:.4f}, oracle {r_ref:.4f} over {len(rows)} rows "
          f"({rep['ambiguous']} rows differ at near-ties)")
