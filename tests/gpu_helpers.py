"""Helpers for the GPU parity tests: run the library through its C ABI and compare with
the oracle on the same seeded inputs.

Tolerances (the bar the tests hold the GPU path to):
  pyramid            bit-exact (both sides round one exact-to-2^-40 mean to bf16, nearest even)
  S2 / idx           identical where the oracle's smallest K-th/(K+1)-th gap over the walk is
                     >= 1e-3; elsewhere the GPU set must be reachable by a walk whose every
                     SelectK is a top-K within 1e-3 (checked by the oracle)
  leaf scores        |gpu - oracle| <= 1e-3 (head-summed natural-log LSE, fp32 vs fp64)
  attention O, LSE   max-abs <= 2e-2 and relative L2 <= 1e-2, on the GPU's own idx
"""
from __future__ import annotations

import math

import numpy as np
import torch

import hierarchical_top_block_gb300 as pisa
import workloads as W

GAP_TOL = 1e-3
SCORE_TOL = 1e-3
ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2


def to_np_bits(t: torch.Tensor) -> np.ndarray:
    return W.bits(t)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def level_sizes(n, C=64):
    out = []
    m = (n + C - 1) // C
    while m >= 1:
        out.append(m)
        if m == 1:
            break
        m = (m + 1) // 2
    return out if n > 0 else []


def pyramid_equal(P_gpu, P_ref, n, n_cap):
    """Compare the rows that hold the pyramid of n tokens inside an n_cap layout [nodes, d]."""
    off = 0
    for l, (m, mcap) in enumerate(zip(level_sizes(n) + [0] * 64, level_sizes(n_cap))):
        if m and not np.array_equal(P_gpu[off:off + m], P_ref[off:off + m]):
            return False
        off += mcap
    return True


def check_selection(o, Qb, Kb, Pb, K_sel, rows, gpu_idx, gpu_s2=None, gpu_score=None, causal=True, scoring=0):
    """rows: int64 [R, 3] (b, h_kv, t); gpu_*: arrays [R, ...].  Returns a small report dict."""
    ref = o.select(Qb, Kb, Pb, K_sel, rows, causal=causal, scoring=scoring)
    clear = ref["min_gap"] >= GAP_TOL
    same_idx = np.all(ref["idx"] == gpu_idx, axis=1)
    bad_clear = np.where(clear & ~same_idx)[0]
    assert bad_clear.size == 0, f"idx differs on {bad_clear.size} clear-gap rows, e.g. row {rows[bad_clear[0]]}: " \
                                f"gpu {gpu_idx[bad_clear[0]]} oracle {ref['idx'][bad_clear[0]]}"
    if gpu_s2 is not None:
        same_s2 = np.all(ref["s2"] == gpu_s2, axis=1)
        bad = np.where(clear & ~same_s2)[0]
        assert bad.size == 0, f"S2 differs on clear-gap row {rows[bad[0]]}: gpu {gpu_s2[bad[0]]} oracle {ref['s2'][bad[0]]}"
    amb = np.where(~same_idx)[0]
    if amb.size:
        ok = o.admissible(Qb, Kb, Pb, K_sel, rows[amb], gpu_idx[amb], tol=GAP_TOL, causal=causal, scoring=scoring)
        assert np.all(ok == 1), f"{int(np.sum(ok != 1))} ambiguous rows are not admissible: {rows[amb][ok != 1][:3]}"
    if gpu_score is not None and gpu_s2 is not None:
        same_s2 = np.all(ref["s2"] == gpu_s2, axis=1)
        valid = (ref["cand"] >= 0) & same_s2[:, None]
        with np.errstate(invalid="ignore"):
            diff = np.abs(np.where(valid, gpu_score - ref["cand_score"], 0.0))
        assert diff.max() <= SCORE_TOL, f"leaf score differs by {diff.max()}"
        # slots without a candidate leaf (absent survivor, leaf past the end, or not yet
        # visible) read -inf
        empty = (ref["cand"] < 0) & same_s2[:, None]
        assert np.all(np.isneginf(gpu_score[empty])), "a slot without a candidate leaf does not read -inf"
    return dict(rows=len(rows), ambiguous=int(amb.size), clear=int(clear.sum()))


def check_attention(o, Qb, Kb, Vb, idx_np, rows_bt, gpu_O, gpu_LSE, causal=True):
    """rows_bt: int64 [R, 2] (b, t); gpu_O [R, H_q, d] float; gpu_LSE [R, H_q]."""
    O, LSE, ws = o.sparse_attention(Qb, Kb, Vb, idx_np, rows_bt, causal=causal)
    fin = np.isfinite(LSE)
    assert np.array_equal(fin, np.isfinite(gpu_LSE)), "LSE finiteness differs"
    err_o = np.abs(gpu_O - O).max() if O.size else 0.0
    err_l = np.abs(np.where(fin, gpu_LSE - LSE, 0.0)).max() if LSE.size else 0.0
    assert err_o <= ATTN_MAX_ABS, f"O max-abs error {err_o}"
    assert rel_l2(gpu_O, O) <= ATTN_REL_L2, f"O relative L2 {rel_l2(gpu_O, O)}"
    assert err_l <= ATTN_MAX_ABS, f"LSE max-abs error {err_l}"
    assert rel_l2(np.where(fin, gpu_LSE, 0), np.where(fin, LSE, 0)) <= ATTN_REL_L2
    assert np.all(np.abs(ws[fin] - 1.0) <= 1e-3)
    return dict(max_abs_O=float(err_o), max_abs_LSE=float(err_l))


def run_gpu_prefill(Q, K, V, K_sel, causal=True, scoring=0):
    """Runs pyramid, selection and attention; returns CPU copies."""
    P = pisa.pisa_build_pyramid(K)
    idx, score, s2 = pisa.pisa_select_prefill(Q, K, P, K_sel, causal=causal, want_scores=True, want_s2=True,
                                              scoring=scoring)
    O, LSE = pisa.pisa_sparse_attn_prefill(Q, K, V, idx, causal=causal)
    torch.cuda.synchronize()
    assert pisa.pisa_get_last_device_error() == 0
    return dict(P=P, idx=idx.cpu().numpy(), score=score.cpu().numpy(), s2=s2.cpu().numpy(), O=O, LSE=LSE.cpu().numpy())


def full_prefill_check(o, Q, K, V, K_sel, causal=True, sample=None, seed=0, scoring=0):
    """Q, K, V on the GPU; the oracle gets bit-identical CPU copies."""
    B, N, H_q, d = Q.shape
    H_kv = K.shape[1]
    res = run_gpu_prefill(Q, K, V, K_sel, causal, scoring)
    Qb, Kb, Vb = to_np_bits(Q), to_np_bits(K), to_np_bits(V)
    Pb = o.build_pyramid(Kb)
    assert np.array_equal(to_np_bits(res["P"]), Pb), "pyramid differs from the oracle"
    if sample is None:
        rows = np.array([(b, g, t) for b in range(B) for g in range(H_kv) for t in range(N)], np.int64)
    else:
        rng = np.random.default_rng(seed)
        rows = np.stack([rng.integers(0, B, sample), rng.integers(0, H_kv, sample), rng.integers(0, N, sample)], 1)
        rows[: min(sample, 4), 2] = np.array([0, N - 1, min(N - 1, 63), min(N - 1, 64)])[: min(sample, 4)]
    rows = rows.astype(np.int64)
    gi = res["idx"][rows[:, 0], rows[:, 1], rows[:, 2]]
    gs2 = res["s2"][rows[:, 0], rows[:, 1], rows[:, 2]]
    gsc = res["score"][rows[:, 0], rows[:, 1], rows[:, 2]]
    rep = check_selection(o, Qb, Kb, Pb, K_sel, rows, gi, gs2, gsc, causal=causal, scoring=scoring)
    bt = np.unique(rows[:, [0, 2]], axis=0)
    O = res["O"].float().cpu().numpy()[bt[:, 0], bt[:, 1]]
    LSE = np.transpose(res["LSE"], (0, 2, 1))[bt[:, 0], bt[:, 1]]
    rep.update(check_attention(o, Qb, Kb, Vb, res["idx"], bt, O, LSE, causal=causal))
    return rep


def check_bsa(o, Qb, Pb, K_sel, rows, gpu_idx, causal=True):
    """BSA selection parity: identical to the oracle's set where its K-th/(K+1)-th score gap is
    >= 1e-3; elsewhere the GPU's set must be a top-K within 1e-3 of the oracle's fp64 scores
    (own block present in causal mode, as many ranked blocks as the oracle's)."""
    ref = o.select_bsa(Qb, Pb, K_sel, rows, causal=causal, want_scores=True)
    clear = ref["min_gap"] >= GAP_TOL
    same = np.all(ref["idx"] == gpu_idx, axis=1)
    bad = np.where(clear & ~same)[0]
    assert bad.size == 0, f"BSA idx differs on {bad.size} clear-gap rows, e.g. row {rows[bad[0]]}: " \
                          f"gpu {gpu_idx[bad[0]]} oracle {ref['idx'][bad[0]]}"
    for i in np.where(~same)[0]:
        t = int(rows[i, 2])
        own = t // 64 if causal else -1
        got = [int(x) for x in gpu_idx[i] if x >= 0]
        want = [int(x) for x in ref["idx"][i] if x >= 0]
        assert got == sorted(set(got)) and len(got) == len(want), (rows[i], got, want)
        if causal:
            assert own in got, (rows[i], got)
        sc = ref["score"][i]
        chosen = [j for j in got if j != own]
        assert all(np.isfinite(sc[j]) for j in chosen), (rows[i], got)
        others = [j for j in range(sc.size) if np.isfinite(sc[j]) and j not in chosen]
        if chosen and others:
            assert min(sc[j] for j in chosen) >= max(sc[j] for j in others) - GAP_TOL, (rows[i], got, want)
    return dict(rows=len(rows), ambiguous=int((~same).sum()), clear=int(clear.sum()))
