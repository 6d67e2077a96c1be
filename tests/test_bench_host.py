"""Host-side logic of bench.py's secondary sections, on the CPU: the device calls are replaced
by stand-ins (the oracle's selection for the selection-quality section, a counter for the
decode loop), so what is checked is the bookkeeping around them: which rows and steps are
measured and which fields the JSON line gets."""
import numpy as np
import torch

import bench
import hierarchical_top_block_gb300 as pisa
import workloads as W


class _Event:
    def __init__(self, enable_timing=False):
        pass

    def record(self, *args):
        pass

    def elapsed_time(self, other):
        return 0.125


def _no_device(monkeypatch):
    monkeypatch.setattr(torch.cuda, "Event", _Event)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "empty_cache", lambda *a: None)


def test_selection_quality_section_reports_needle_hits(monkeypatch, oracle_impl):
    o = oracle_impl
    bits = W.bits
    monkeypatch.setattr(pisa, "pisa_build_pyramid", lambda K: o.build_pyramid(bits(K)))

    def select(Q, K, P, K_sel, scoring="lse"):
        B, N, H_q, d = Q.shape
        H_kv = K.shape[1]
        rows = np.array([(b, g, t) for b in range(B) for g in range(H_kv) for t in range(N)], np.int64)
        sc = pisa.SCORING[scoring] if isinstance(scoring, str) else scoring
        return torch.from_numpy(o.select(bits(Q), bits(K), P, K_sel, rows, scoring=sc)["idx"].reshape(B, H_kv, N, K_sel))

    monkeypatch.setattr(pisa, "pisa_select_prefill", select)
    _no_device(monkeypatch)
    w = W.WORKLOADS["tiny"]                       # K = 4; 2 needles x 8 aimed rows
    res = bench.selection_quality_section(w, "cpu", samples=8)
    assert res["needle_rows"] == 16
    for K_sel in (4, 8):
        for name in ("lse", "pisa1", "pisa2"):
            rep = res[f"K{K_sel}_{name}"]
            assert 0.0 <= rep["needle_hit_rate"] <= 1.0 and rep["queries"] == 8
    assert res["K8_lse"]["needle_hit_rate"] == 1.0      # g K >= M_1: nothing pruned, every needle kept
    assert res["K8_lse"]["recall_at_k"] == 1.0


def test_secondary_decode_times_every_step(monkeypatch):
    seen = []

    def decode(q, k, v, Kc, Vc, Pc, seq, K_sel, o=None, lse=None, ws=None):
        # the logits scratch is allocated once, at the size the library asks for
        assert ws is not None and ws.numel() == pisa.pisa_decode_workspace_bytes(
            pisa.make_shape(w.B, 0, w.H_q, w.H_kv, w.d, Kc.shape[2]), pisa.make_params(w.K)) > 0
        seen.append((int(seq[0]), Kc.shape[2], ws.data_ptr()))
        seq += 1

    monkeypatch.setattr(pisa, "pisa_build_pyramid", lambda K, N=None: torch.empty(0))
    monkeypatch.setattr(pisa, "pisa_decode_step", decode)
    _no_device(monkeypatch)
    w = W.WORKLOADS["decode_128k"].with_(B=2, N=500)
    res = bench.secondary_decode(w, "cpu")
    assert res["steps"] == w.decode_steps == 256
    assert len(seen) == 3 + 256 and seen[0][0] == 500
    assert all(pos < n_cap for pos, n_cap, _ in seen) and seen[-1][0] == seen[-1][1] - 1   # the cache fills exactly
    assert len({p for _, _, p in seen}) == 1
    assert res["step_us_mean"] == res["step_us_p50"] == 125.0


def test_a_failing_section_is_reported_not_fatal():
    def boom(x):
        raise RuntimeError(f"device error word {x}")
    assert bench.section(boom, 5) == {"error": "RuntimeError: device error word 5"}
    assert bench.section(lambda a, b=0: a + b, 1, b=2) == 3


def test_work_counts():
    """The algorithmic work the per-kernel rooflines divide by: decode bytes count the selected
    blocks' keys once (they are among the 2K candidate leaves), the walk's child rows follow
    the level geometry, and Stage 2's flops count the visible keys of each eligible leaf child."""
    w = W.WORKLOADS["decode_128k"]
    # 131073 tokens: 7 scored levels x 64 child rows, 32 candidate leaves of keys, 16 of values
    assert bench.decode_hbm_bytes(w) == 64 * 8 * (7 * 64 + 32 * 64 + 16 * 64) * 128 * 2
    assert bench.level_sizes(262144) == [4096 >> i for i in range(13)]
    assert bench.level_sizes(65) == [2, 1] and bench.level_sizes(0) == []
    r = bench.stage1_work(262144, 16, 1, 128, 16)
    # the last query scores levels 8..2 (32 candidates each, 64 child rows): 448 rows; the
    # first 17 * 64 queries see at most 16 leaves, and no level is scored
    assert bench.stage1_work(64 * 17, 16, 1, 128, 16)["child_rows"] == 0
    assert r["child_rows"] <= 448 * 262144 and r["flops"] == 2.0 * 128 * 16 * r["child_rows"]
    tail = bench.stage1_work(262144, 16, 1, 128, 16)["child_rows"] - bench.stage1_work(262143, 16, 1, 128, 16)["child_rows"]
    assert tail == 448
    s2 = torch.full((1, 1, 200, 2), -1, dtype=torch.int32)
    s2[0, 0, 10, 0] = 0      # t = 10: leaf 0 holds keys 0..10 visible, leaf 1 none
    s2[0, 0, 199, 0] = 1     # t = 199: leaf 2 keys 128..199 -> 64 visible, leaf 3 (key 192..) 8 visible
    got = bench.leaf_lse_work(s2, 200, 8, 2, 64)
    assert got["visible_keys"] == 11 + 64 + 8 and got["flops"] == 2.0 * 64 * 4 * (11 + 64 + 8)


def test_phase_rooflines_fields(monkeypatch):
    times = {"pyramid": (0.1, 2), "stage1": (4.0, 2), "cluster": (0.2, 2), "leaf_lse": (5.0, 2), "topk": (0.3, 2),
             "sparse_attn": (16.0, 2), "bsa_select": (0.0, 0), "decode": (0.0, 0), "attn_backward": (0.0, 0)}
    state = []
    monkeypatch.setattr(pisa, "pisa_phase_timing", lambda on=True: state.append(on))
    monkeypatch.setattr(pisa, "pisa_phase_times", lambda: times)
    _no_device(monkeypatch)
    steps = []
    w = W.WORKLOADS["tiny"]
    s2 = torch.zeros(w.B, w.H_kv, w.N, w.K, dtype=torch.int32)
    res = bench.phase_rooflines(w, lambda: steps.append(1), s2, attn_flops=1e9, steps=2)
    assert state == [True, False] and len(steps) == 2
    assert set(res) >= {"pyramid", "stage1", "cluster", "leaf_lse", "topk", "sparse_attn"}
    assert res["stage1"]["ms"] == 2.0 and res["stage1"]["bound"] == "hbm" and res["leaf_lse"]["bound"] == "tensor"
    a = res["sparse_attn"]
    assert abs(a["achieved"] - 1e9 / 8e-3 / 1e12) < 1e-12 and abs(a["frac"] - a["achieved"] / a["peak"]) < 1e-12
