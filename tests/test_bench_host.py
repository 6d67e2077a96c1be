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

    def decode(q, k, v, Kc, Vc, Pc, seq, K_sel, o=None, lse=None):
        seen.append((int(seq[0]), Kc.shape[2]))
        seq += 1

    monkeypatch.setattr(pisa, "pisa_build_pyramid", lambda K, N=None: torch.empty(0))
    monkeypatch.setattr(pisa, "pisa_decode_step", decode)
    _no_device(monkeypatch)
    w = W.WORKLOADS["decode_128k"].with_(B=2, N=500)
    res = bench.secondary_decode(w, "cpu")
    assert res["steps"] == w.decode_steps == 256
    assert len(seen) == 3 + 256 and seen[0][0] == 500
    assert all(pos < n_cap for pos, n_cap in seen) and seen[-1][0] == seen[-1][1] - 1   # the cache fills exactly
    assert res["step_us_mean"] == res["step_us_p50"] == 125.0


def test_a_failing_section_is_reported_not_fatal():
    def boom(x):
        raise RuntimeError(f"device error word {x}")
    assert bench.section(boom, 5) == {"error": "RuntimeError: device error word 5"}
    assert bench.section(lambda a, b=0: a + b, 1, b=2) == 3
