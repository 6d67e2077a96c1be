"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each function takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with a closed form, an invariant, a special case that reduces to a textbook
routine, or brute force on a tiny input.  The same functions run against the real oracle
(all must pass) and against copies of it with one planted mistake (at least one must fail).

Sources: paper summary page "Block Sparse Attention with Log-Linear Complexity"
(Tang et al.): section "Core method" (eq. 21, the LSE block score; leaf level uses raw
keys), section "Method step details" (step 1 pyramid eqs 10-15, step 2 selection with the
eq. 22 head sum and SelectK, step 3 decode, step 4 attention), section "Prerequisites"
(LSE Taylor form, GQA groups share one selected set); the blog post of the same title,
section 3.3 (softmax over connected positions only; weights sum to one within 1e-3).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------
def f2b(x) -> np.ndarray:
    """float values that are exact in bf16 -> uint16 bit patterns (asserts exactness)."""
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def b2f(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def random_bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = x.view(np.uint32)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def level_offsets(sizes):
    off = [0]
    for m in sizes[:-1]:
        off.append(off[-1] + m)
    return off


def brute_leaf_lse(Qf, Kf, scale, t, C, causal=True):
    """Exact LSE of every leaf for one query row: Qf [G, d], Kf [N, d] (float64).
    Returns {leaf: sum over heads of LSE over the leaf's (causal) keys}."""
    N = Kf.shape[0]
    M1 = (N + C - 1) // C
    z = scale * (Qf @ Kf.T)  # [G, N]
    out = {}
    for j in range(M1):
        c0, c1 = j * C, min(N, j * C + C)
        if causal:
            if c0 > t:
                continue
            c1 = min(c1, t + 1)
        zz = z[:, c0:c1]
        m = zz.max(axis=1, keepdims=True)
        out[j] = float(np.sum(m[:, 0] + np.log(np.exp(zz - m).sum(axis=1))))
    return out


# ------------------------------------------------------------------------------------
# step 1: the pyramid
# ------------------------------------------------------------------------------------
def pin_level_sizes(o):
    """Level sizes are the closed form of the pages' pyramid (golden table)."""
    for row in read_golden("pyramid_levels.txt"):
        n = int(row[0])
        want = [int(x) for x in row[1:]]
        assert o.level_sizes(n) == want, (n, o.level_sizes(n), want)
        assert o.num_levels(n) == len(want)
        assert o.pyramid_nodes(n) == sum(want)
        # L = 1 + ceil(log2 M_1)
        assert len(want) == 1 + math.ceil(math.log2(want[0]))


def pin_bf16_rounding(o):
    for xs, bs in read_golden("bf16_rounding.txt"):
        assert o.f64_to_bf16(float.fromhex(xs)) == int(bs, 16), (xs, bs, hex(o.f64_to_bf16(float.fromhex(xs))))


def pin_pyramid_constant_keys(o):
    """Constant keys: every summary at every level equals that key (ragged nodes too)."""
    d, C = 16, 64
    for N in (1, 63, 337, 64 * 5 + 1, 1024):
        vec = f2b(np.arange(d, dtype=np.float32) * 0.25 - 1.5)
        K = np.tile(vec, (1, 2, N, 1)).astype(np.uint16)
        P = o.build_pyramid(K, C=C)
        sizes = o.level_sizes(N)
        assert P.shape[2] == sum(sizes)
        assert np.all(P == vec[None, None, None, :]), N


def pin_pyramid_raw_mean(o):
    """Each summary is within accumulated rounding of the mean of the raw keys it covers
    (mean of means of equal-size groups = overall mean; each level adds <= 2^-8 relative)."""
    rng = np.random.default_rng(1)
    d, C = 32, 64
    for N in (64 * 16, 64 * 13 + 5):
        K = random_bf16(rng, (1, 1, N, d))
        # a ramp so that a wrong child index shows up clearly
        Kf = b2f(K[0, 0]) + np.linspace(-4, 4, N)[:, None]
        K[0, 0] = f2b_round(Kf)
        Kf = b2f(K[0, 0])
        P = b2f(o.build_pyramid(K, C=C)[0, 0])
        sizes = o.level_sizes(N)
        off = level_offsets(sizes)
        for l, m in enumerate(sizes, start=1):
            span = C * 2 ** (l - 1)
            for i in range(m):
                c0, c1 = i * span, min(N, (i + 1) * span)
                full = (c1 - c0) == span
                raw = Kf[c0:c1].mean(axis=0)
                got = P[off[l - 1] + i]
                tol = l * 2.0 ** -8 * np.abs(Kf[c0:c1]).max(axis=0) + 1e-6
                if full:
                    assert np.all(np.abs(got - raw) <= tol), (N, l, i, np.abs(got - raw).max())


def f2b_round(x):
    a = np.asarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def pin_pyramid_ragged_leaf_mean(o):
    """A ragged last leaf of n keys is the mean of those n keys (not divided by C)."""
    d, C = 8, 64
    N = 64 + 3
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 64:67] = f2b([[2.0] * d, [4.0] * d, [6.0] * d])
    P = o.build_pyramid(K, C=C)
    assert np.all(b2f(P[0, 0, 1]) == 4.0)       # leaf 1 = mean(2, 4, 6)
    assert np.all(b2f(P[0, 0, 2]) == 2.0)       # root = mean(leaf0 = 0, leaf1 = 4)


# ------------------------------------------------------------------------------------
# step 2: scores and selection
# ------------------------------------------------------------------------------------
def _spike_case(o, t, K_sel=2):
    """Two leaves (N=128), one query head, d=64, q = 8 e_0 so that logit = k[0] exactly."""
    d, C, N = 64, 64, 128
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 0:64, 0] = f2b(1.0)                 # leaf 0: all logits 1
    K[0, 0, 64 + 10, 0] = f2b(6.0)              # leaf 1: one logit 6 at key 74
    P = o.build_pyramid(K)
    r = o.select(Q, K, P, K_sel, np.array([[0, 0, t]]), scale=1.0 / 8.0)
    return r


def pin_leaf_lse_closed_forms(o):
    g = {name: float(v) for name, v in read_golden("leaf_lse_closed_forms.txt")}
    r = _spike_case(o, t=127)
    cand, cs = r["cand"][0], r["cand_score"][0]
    got = {int(j): s for j, s in zip(cand, cs) if j >= 0}
    assert abs(got[0] - g["uniform_64_logit_1"]) < 1e-12, got
    assert abs(got[1] - g["spike_6_in_64"]) < 1e-12, got
    # causal: query at key 69 sees keys 64..69 of its own leaf (all logits 0); the spike at 74 is masked
    r = _spike_case(o, t=69)
    got = {int(j): s for j, s in zip(r["cand"][0], r["cand_score"][0]) if j >= 0}
    assert abs(got[1] - g["prefix_6_of_zeros"]) < 1e-12, got


def pin_gqa_head_sum(o):
    """Two query heads share one KV head: the block score is the sum of per-head LSEs (eq. 22)."""
    g = {name: float(v) for name, v in read_golden("leaf_lse_closed_forms.txt")}
    d, C, N = 64, 64, 128
    Q = np.zeros((1, N, 2, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    Q[0, :, 1, 1] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 64:128, 0] = f2b(1.0)               # head 0 sees logit 1 on all of leaf 1
    K[0, 0, 64 + 10, 1] = f2b(6.0)              # head 1 sees a spike of 6 in leaf 1
    P = o.build_pyramid(K)
    r = o.select(Q, K, P, 2, np.array([[0, 0, 127]]), scale=1.0 / 8.0)
    got = {int(j): s for j, s in zip(r["cand"][0], r["cand_score"][0]) if j >= 0}
    assert abs(got[1] - g["two_heads_1_and_spike"]) < 1e-12, got
    assert abs(got[0] - 2 * math.log(64)) < 1e-12, got


def pin_lse_beats_mean(o):
    """LSE scoring prefers a leaf with one sharp key over a leaf of uniformly moderate keys,
    which mean-pooled scoring would rank the other way (Taylor view: the variance term)."""
    d, C, N = 64, 64, 64 * 4
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 0:64, 0] = f2b(1.0)                 # leaf 0: mean logit 1.0, LSE = log 64 + 1 = 5.16
    K[0, 0, 64 + 7, 0] = f2b(6.0)               # leaf 1: mean logit 0.09, LSE = 6.15
    P = o.build_pyramid(K)
    # K=2: own leaf (3) + the single best other leaf
    r = o.select(Q, K, P, 2, np.array([[0, 0, N - 1]]), scale=1.0 / 8.0)
    assert list(r["idx"][0]) == [1, 3], r["idx"]


def _spike_case_scored(o, t, scoring, K_sel=2):
    d, C, N = 64, 64, 128
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 0:64, 0] = f2b(1.0)
    K[0, 0, 64 + 10, 0] = f2b(6.0)
    P = o.build_pyramid(K)
    r = o.select(Q, K, P, K_sel, np.array([[0, 0, t]]), scale=1.0 / 8.0, scoring=scoring)
    return {int(j): s for j, s in zip(r["cand"][0], r["cand_score"][0]) if j >= 0}


def pin_scoring_variants_closed_forms(o):
    """PISA-1 and PISA-2 leaf scores are the first- and second-order truncations of the LSE
    around the mean of the block's logits (golden closed forms, population variance)."""
    g = {name: float(v) for name, v in read_golden("scoring_variants.txt")}
    p1, p2 = _spike_case_scored(o, 127, 1), _spike_case_scored(o, 127, 2)
    assert abs(p1[0] - g["pisa1_uniform_64_logit_1"]) < 1e-12, p1
    assert abs(p2[0] - g["pisa1_uniform_64_logit_1"]) < 1e-12, p2  # zero variance
    assert abs(p1[1] - g["pisa1_spike_6_in_64"]) < 1e-12, p1
    assert abs(p2[1] - g["pisa2_spike_6_in_64"]) < 1e-12, p2
    for sc in (1, 2):  # causal prefix of 6 zero logits in the own leaf
        got = _spike_case_scored(o, 69, sc)
        assert abs(got[1] - g["pisa12_prefix_6_of_zeros"]) < 1e-12, (sc, got)


def pin_scoring_variants_order(o):
    """On random inputs where no level prunes (the candidate slots are the same for every
    scoring): PISA-1 <= LSE (Jensen: log mean exp >= mean) and PISA-1 <= PISA-2 (variance
    >= 0), slot by slot; a single visible key gives the same score under all three."""
    Q, K, V = _tiny_inputs(seed=21, N=64 * 6)
    P = o.build_pyramid(K)
    N = Q.shape[1]
    rows = np.array([[0, 0, t] for t in range(0, N, 37)], np.int64)
    r = [o.select(Q, K, P, 4, rows, scoring=s) for s in (0, 1, 2)]
    assert np.array_equal(r[0]["cand"], r[1]["cand"]) and np.array_equal(r[0]["cand"], r[2]["cand"])
    m = r[0]["cand"] >= 0
    lse, p1, p2 = (x["cand_score"][m] for x in r)
    assert np.all(p1 <= lse + 1e-12) and np.all(p1 <= p2 + 1e-12)
    assert np.any(p1 < lse - 1e-6) and np.any(p2 > p1 + 1e-6)
    # query at the first key of a leaf: its own leaf has one visible key
    t = 64 * 5
    own = [o.select(Q, K, P, 4, np.array([[0, 0, t]]), scoring=s) for s in (0, 1, 2)]
    vals = [x["cand_score"][0][list(x["cand"][0]).index(5)] for x in own]
    assert abs(vals[0] - vals[1]) < 1e-12 and abs(vals[0] - vals[2]) < 1e-12, vals


def pin_mean_scoring_ranks_like_the_mean(o):
    """The case where LSE prefers the sharp leaf: first-order (PISA-1) scoring is the mean
    logit plus log m, so it keeps the uniformly moderate leaf instead."""
    d, C, N = 64, 64, 64 * 4
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 0:64, 0] = f2b(1.0)
    K[0, 0, 64 + 7, 0] = f2b(6.0)
    P = o.build_pyramid(K)
    assert list(o.select(Q, K, P, 2, np.array([[0, 0, N - 1]]), scale=1.0 / 8.0, scoring=1)["idx"][0]) == [0, 3]
    assert list(o.select(Q, K, P, 2, np.array([[0, 0, N - 1]]), scale=1.0 / 8.0, scoring=0)["idx"][0]) == [1, 3]
    # the admissibility check ranks by the same score: each scoring's own set is admissible under
    # that scoring and the other scoring's set is not (the gaps are about 0.9)
    row = np.array([[0, 0, N - 1]])
    for scoring, mine, other in ((1, [0, 3], [1, 3]), (0, [1, 3], [0, 3])):
        for target, want in ((mine, 1), (other, 0)):
            got = o.admissible(Q, K, P, 2, row, np.array([target], np.int32), scale=1.0 / 8.0, scoring=scoring)[0]
            assert got == want, (scoring, target, got)


# ------------------------------------------------------------------------------------
# backward of step 4 (the gradient of the forward; the pages give none)
# ------------------------------------------------------------------------------------
def _bwd_case(seed, N=128, H_q=2, H_kv=1, d=16, K_sel=1):
    rng = np.random.default_rng(seed)
    Q, K, V = (random_bf16(rng, s, 0.5) for s in ((1, N, H_q, d), (1, H_kv, N, d), (1, H_kv, N, d)))
    dO = random_bf16(rng, (1, N, H_q, d))
    return Q, K, V, dO


def pin_backward_dense_autograd(o):
    """K >= M_1 keeps every eligible block, so step 4 is dense causal attention: its
    gradients equal PyTorch's autograd of the textbook formula (fp64)."""
    import torch
    Q, K, V, dO = _bwd_case(41, N=130, H_q=4, H_kv=2, d=16)
    N, H_q, H_kv, d = 130, 4, 2, 16
    P = o.build_pyramid(K)
    K_sel = 3                                     # M_1 = 3 leaves
    rows = np.array([[0, g, t] for g in range(H_kv) for t in range(N)], np.int64)
    idx = o.select(Q, K, P, K_sel, rows)["idx"].reshape(1, H_kv, N, K_sel)
    dQ, dK, dV = o.sparse_attention_backward(Q, K, V, idx, dO)
    q = torch.tensor(b2f(Q), dtype=torch.float64, requires_grad=True)
    k = torch.tensor(b2f(K), dtype=torch.float64, requires_grad=True)
    v = torch.tensor(b2f(V), dtype=torch.float64, requires_grad=True)
    G = H_q // H_kv
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)          # [1, H_q, N, d]
    s_ = torch.einsum("bthd,bhnd->bhtn", q, kk) / math.sqrt(d)
    s_ = s_.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
    out = torch.einsum("bhtn,bhnd->bthd", torch.softmax(s_, dim=-1), vv)
    out.backward(torch.tensor(b2f(dO)))
    assert np.abs(dQ - q.grad.numpy()).max() < 1e-10
    assert np.abs(dK - k.grad.numpy()).max() < 1e-10
    assert np.abs(dV - v.grad.numpy()).max() < 1e-10



def pin_backward_dense_autograd_noncausal(o):
    """Without the causal mask and with K >= M_1, step 4 is dense attention over all keys: its
    gradients equal PyTorch's autograd of the unmasked textbook formula (fp64)."""
    import torch
    N, H_q, H_kv, d, K_sel = 150, 4, 2, 16, 3       # M_1 = 3 leaves, the last one ragged
    Q, K, V, dO = _bwd_case(53, N=N, H_q=H_q, H_kv=H_kv, d=d)
    P = o.build_pyramid(K)
    rows = np.array([[0, g, t] for g in range(H_kv) for t in range(N)], np.int64)
    idx = o.select(Q, K, P, K_sel, rows, causal=False)["idx"].reshape(1, H_kv, N, K_sel)
    dQ, dK, dV = o.sparse_attention_backward(Q, K, V, idx, dO, causal=False)
    q = torch.tensor(b2f(Q), dtype=torch.float64, requires_grad=True)
    k = torch.tensor(b2f(K), dtype=torch.float64, requires_grad=True)
    v = torch.tensor(b2f(V), dtype=torch.float64, requires_grad=True)
    G = H_q // H_kv
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    s_ = torch.einsum("bthd,bhnd->bhtn", q, kk) / math.sqrt(d)
    out = torch.einsum("bhtn,bhnd->bthd", torch.softmax(s_, dim=-1), vv)
    out.backward(torch.tensor(b2f(dO)))
    assert np.abs(dQ - q.grad.numpy()).max() < 1e-10
    assert np.abs(dK - k.grad.numpy()).max() < 1e-10
    assert np.abs(dV - v.grad.numpy()).max() < 1e-10

def pin_backward_finite_differences(o):
    """Sparse selection (K=1: the own block only in causal mode, other blocks absent): the
    gradients match central differences of the oracle's own forward of L = sum(O * dO),
    Richardson-extrapolated (steps 2^-6 and 2^-5, both exact in bf16 around the chosen
    entries), for entries of Q, K and V."""
    Q, K, V, dO = _bwd_case(43)
    N, H_q, H_kv, d = 128, 2, 1, 16
    idx = np.zeros((1, H_kv, N, 2), np.int32)
    idx[0, 0, :, 0] = np.arange(N) // 64                 # own block
    idx[0, 0, :, 1] = np.where(np.arange(N) >= 64, 0, -1)  # and block 0 for the second block
    dQ, dK, dV = o.sparse_attention_backward(Q, K, V, idx, dO)
    rows = np.array([[0, t] for t in range(N)], np.int64)
    w = b2f(dO)[0]

    def loss(Qx, Kx, Vx):
        O, _, _ = o.sparse_attention(Qx, Kx, Vx, idx, rows)
        return float((O * w).sum())

    def fd(arr, pos, which):
        base = arr.copy()
        x0 = b2f(base[pos])

        def at(delta):
            a2 = base.copy()
            a2[pos] = f2b(np.float32(x0 + delta))
            args = {"Q": Q, "K": K, "V": V}
            args[which] = a2
            return loss(args["Q"], args["K"], args["V"])
        h = 2.0 ** -6
        d1 = (at(h) - at(-h)) / (2 * h)
        d2 = (at(2 * h) - at(-2 * h)) / (4 * h)
        return (4 * d1 - d2) / 3

    rng = np.random.default_rng(5)
    for which, arr, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for _ in range(4):
            pos = tuple(int(rng.integers(0, n)) for n in arr.shape)
            x0 = float(b2f(arr[pos]))
            arr_c = arr.copy()
            arr_c[pos] = f2b(np.float32(np.round(x0 * 8) / 8))   # a value on a 2^-3 grid, so +-h stay exact
            g = {"Q": Q, "K": K, "V": V}
            g[which] = arr_c
            ref = o.sparse_attention_backward(g["Q"], g["K"], g["V"], idx, dO)["QKV".index(which)][pos]
            num = fd(arr_c, pos, which)
            assert abs(ref - num) <= 2e-5 + 1e-4 * abs(num), (which, pos, ref, num)


def pin_backward_sums(o):
    """Per (sequence, KV head): sum over keys of dV = sum over the group's queries and heads
    of dO (each softmax row sums to one), and sum over keys of dK = 0 (each row of dS sums
    to zero), on a pruned selection."""
    Q, K, V, dO = _bwd_case(47, N=64 * 6, H_q=4, H_kv=2, d=16)
    N, H_q, H_kv = 64 * 6, 4, 2
    P = o.build_pyramid(K)
    rows = np.array([[0, g, t] for g in range(H_kv) for t in range(N)], np.int64)
    idx = o.select(Q, K, P, 2, rows)["idx"].reshape(1, H_kv, N, 2)
    dQ, dK, dV = o.sparse_attention_backward(Q, K, V, idx, dO)
    w = b2f(dO)[0]                                   # [N, H_q, d]
    G = H_q // H_kv
    for g in range(H_kv):
        assert np.abs(dV[0, g].sum(0) - w[:, g * G:(g + 1) * G].sum((0, 1))).max() < 1e-9
        assert np.abs(dK[0, g].sum(0)).max() < 1e-9
    assert np.abs(dK).max() > 1e-3


def pin_backward_sampled_equals_full(o):
    """The sampled backward (dQ of listed positions, dK and dV of listed key blocks) gives the
    full backward's values exactly: the same rows accumulate in the same order.  Pruned
    selections (K = 2 of 7 leaves, ragged N), causal and not, two sequences, G_Q = 2."""
    N, H_q, H_kv, d = 64 * 6 + 29, 4, 2, 16
    rng = np.random.default_rng(61)
    for causal in (True, False):
        Q, K, V = (random_bf16(rng, s, 0.5) for s in ((2, N, H_q, d), (2, H_kv, N, d), (2, H_kv, N, d)))
        dO = random_bf16(rng, (2, N, H_q, d))
        P = o.build_pyramid(K)
        rows = np.array([[b, g, t] for b in range(2) for g in range(H_kv) for t in range(N)], np.int64)
        idx = o.select(Q, K, P, 2, rows, causal=causal)["idx"].reshape(2, H_kv, N, 2)
        dQ, dK, dV = o.sparse_attention_backward(Q, K, V, idx, dO, causal=causal)
        M1 = (N + 63) // 64
        srows = np.array([0, 5, 63, 64, N - 1, N, N + 200, 2 * N - 1], np.int64)          # b * N + t
        sblocks = np.array([0, M1 - 1, M1 + 2, 2 * M1 + 1, 4 * M1 - 1], np.int64)          # (b * H_kv + h) * M1 + j
        sq, sk, sv = o.sparse_attention_backward_sampled(Q, K, V, idx, dO, srows, sblocks, causal=causal)
        for i, r in enumerate(srows):
            assert np.array_equal(sq[i], dQ[r // N, r % N]), (causal, r)
        for i, blk in enumerate(sblocks):
            bg, j = divmod(int(blk), M1)
            b, h = divmod(bg, H_kv)
            n = min(64, N - 64 * j)
            assert np.array_equal(sk[i, :n], dK[b, h, 64 * j:64 * j + n]), (causal, blk)
            assert np.array_equal(sv[i, :n], dV[b, h, 64 * j:64 * j + n]), (causal, blk)
            assert not sk[i, n:].any() and not sv[i, n:].any()
        assert np.abs(sk).max() > 1e-3 and np.abs(sq).max() > 1e-3


def pin_ties_lower_index(o):
    """Identical keys everywhere: equal scores rank the lower block index first."""
    d, C, N = 16, 64, 64 * 6
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, :] = f2b(np.full(d, 0.5))
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, :, :] = f2b(np.full(d, 0.25))
    P = o.build_pyramid(K)
    r = o.select(Q, K, P, 3, np.array([[0, 0, N - 1], [0, 0, 64 * 3 + 1]]))
    assert list(r["idx"][0]) == [0, 1, 5], r["idx"]
    assert list(r["idx"][1]) == [0, 1, 3], r["idx"]



def pin_admissible_sets(o):
    """The parity rule's admissibility check: the oracle's own selection is admissible; on rows
    whose every SelectK has a gap well above the tolerance nothing else is (a set with one block
    swapped for an unselected eligible one is refused); with exactly tied scores every choice
    among the tied blocks is admissible, though the selection itself takes the lower index."""
    Q, K, V = _tiny_inputs(seed=19)              # 16 leaves, K = 2: levels prune
    P = o.build_pyramid(K)
    N, Ksel = Q.shape[1], 2
    rows = np.array([(0, 0, t) for t in range(200, N, 37)], np.int64)
    r = o.select(Q, K, P, Ksel, rows)
    assert np.all(o.admissible(Q, K, P, Ksel, rows, r["idx"]) == 1)
    clear = np.where(r["min_gap"] > 0.05)[0]
    assert clear.size >= 5, clear.size
    for i in clear:
        t = int(rows[i, 2])
        row = list(r["idx"][i])
        other = next(j for j in range(t // 64 + 1) if j not in row)      # an eligible, unselected leaf
        swapped = sorted([b for b in row if b != t // 64][1:] + [other, t // 64])
        assert o.admissible(Q, K, P, Ksel, rows[i:i + 1], np.array([swapped], np.int32))[0] == 0, (t, row, swapped)
    # identical keys: all scores tie
    d, N = 16, 64 * 6
    Qt = np.zeros((1, N, 1, d), np.uint16)
    Qt[0, :, 0, :] = f2b(np.full(d, 0.5))
    Kt = np.zeros((1, 1, N, d), np.uint16)
    Kt[0, 0, :, :] = f2b(np.full(d, 0.25))
    Pt = o.build_pyramid(Kt)
    row = np.array([[0, 0, N - 1]], np.int64)
    assert list(o.select(Qt, Kt, Pt, 3, row)["idx"][0]) == [0, 1, 5]
    for alt in ([0, 1, 5], [0, 4, 5], [2, 3, 5], [1, 4, 5]):
        assert o.admissible(Qt, Kt, Pt, 3, row, np.array([alt], np.int32))[0] == 1, alt
    assert o.admissible(Qt, Kt, Pt, 3, row, np.array([[0, 1, 4]], np.int32))[0] == 0   # the own block is forced

def _tiny_inputs(seed=3, N=1024, H_q=4, H_kv=1, d=64, offsets=True):
    rng = np.random.default_rng(seed)
    Q = random_bf16(rng, (1, N, H_q, d))
    Kf = rng.standard_normal((1, H_kv, N, d))
    if offsets:
        M1 = (N + 63) // 64
        off = 0.5 * rng.standard_normal((1, H_kv, M1, d))
        Kf = Kf + np.repeat(off, 64, axis=2)[:, :, :N]
    K = f2b_round(Kf)
    V = random_bf16(rng, (1, H_kv, N, d))
    return Q, K, V


def pin_brute_force_topk(o):
    """When the leaves fit (M_1 <= g K, so no level prunes), the selection is the exact top-K
    of the leaf LSE over the eligible leaves, with the own leaf always kept (brute force)."""
    for (N, H_q, H_kv, Ksel) in ((1024, 4, 1, 8), (64 * 11 + 9, 4, 2, 6)):
        Q, K, V = _tiny_inputs(N=N, H_q=H_q, H_kv=H_kv)
        P = o.build_pyramid(K)
        G = H_q // H_kv
        d = Q.shape[-1]
        scale = 1.0 / math.sqrt(d)
        rows = np.array([(0, g, t) for g in range(H_kv) for t in range(0, N, 7)])
        r = o.select(Q, K, P, Ksel, rows)
        for i, (b, g, t) in enumerate(rows):
            Qf = b2f(Q[b, t, g * G:(g + 1) * G])
            lse = brute_leaf_lse(Qf, b2f(K[b, g]), scale, t, 64)
            own = t // 64
            others = sorted((j for j in lse if j != own), key=lambda j: (-lse[j], j))
            want = sorted([own] + others[:Ksel - 1])
            got = [x for x in r["idx"][i] if x >= 0]
            assert got == want, (N, t, got, want)
            # cand scores equal the brute-force leaf LSE
            for j, s in zip(r["cand"][i], r["cand_score"][i]):
                if j >= 0:
                    assert abs(s - lse[int(j)]) < 1e-9, (t, j, s, lse[int(j)])



def pin_brute_force_topk_noncausal(o):
    """Without the causal mask every leaf of the sequence is a candidate and none is forced:
    when no level prunes (M_1 <= g K) the selection is the plain top-K of the leaf LSE over
    all keys of every leaf, ragged last leaf included (brute force, ties to the lower index)."""
    for (N, H_q, H_kv, Ksel) in ((1024, 4, 1, 8), (64 * 11 + 9, 4, 2, 6)):
        Q, K, V = _tiny_inputs(seed=13, N=N, H_q=H_q, H_kv=H_kv)
        P = o.build_pyramid(K)
        G = H_q // H_kv
        scale = 1.0 / math.sqrt(Q.shape[-1])
        rows = np.array([(0, g, t) for g in range(H_kv) for t in range(0, N, 11)])
        r = o.select(Q, K, P, Ksel, rows, causal=False)
        for i, (b, g, t) in enumerate(rows):
            lse = brute_leaf_lse(b2f(Q[b, t, g * G:(g + 1) * G]), b2f(K[b, g]), scale, t, 64, causal=False)
            assert len(lse) == (N + 63) // 64
            want = sorted(sorted(lse, key=lambda j: (-lse[j], j))[:Ksel])
            got = [x for x in r["idx"][i] if x >= 0]
            assert got == want, (N, t, got, want)
            for j, sc in zip(r["cand"][i], r["cand_score"][i]):
                if j >= 0:
                    assert abs(sc - lse[int(j)]) < 1e-9, (t, j, sc, lse[int(j)])
        # the admissibility check without the mask accepts the plain top-K (no forced block)
        assert np.all(o.admissible(Q, K, P, Ksel, rows, r["idx"], causal=False) == 1)
        # queries early in the sequence select leaves after their own position
        assert any(x * 64 > t for (_, _, t), row in zip(rows, r["idx"]) for x in row if x >= 0)

def pin_final_set_invariants(o):
    """Final sets: ascending, unique, -1 padded at the end, own leaf present,
    |I_t| = min(K, #eligible leaves) when no level prunes; <= gK candidates; |S2| <= K."""
    Q, K, V = _tiny_inputs(seed=5)
    P = o.build_pyramid(K)
    N = Q.shape[1]
    for Ksel in (1, 3, 16):
        rows = np.array([(0, 0, t) for t in range(N)])
        r = o.select(Q, K, P, Ksel, rows)
        for t in range(N):
            row = list(r["idx"][t])
            val = [x for x in row if x >= 0]
            assert row == val + [-1] * (Ksel - len(val))
            assert val == sorted(set(val))
            assert t // 64 in val
            assert all(x * 64 <= t for x in val)
            assert sum(1 for x in r["cand"][t] if x >= 0) <= 2 * Ksel
            assert sum(1 for x in r["s2"][t] if x >= 0) <= Ksel
            if Ksel >= 8:  # M_1 = 16 <= g K: every eligible leaf is a candidate
                assert len(val) == min(Ksel, t // 64 + 1)


def pin_walk_prunes_by_summary_lse(o):
    """A hand-built 3-level case where the level walk must prune: 4 leaves, K=1.
    Leaf summaries decide level 2; the subtree whose leaf summary has the larger logit wins."""
    d, C, N = 64, 64, 64 * 4
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    K[0, 0, 0:64, 0] = f2b(-2.0)                # leaf 0 mean -2
    K[0, 0, 64:128, 0] = f2b(-2.0)              # leaf 1 mean -2   -> node (level 2) 0
    K[0, 0, 128:192, 0] = f2b(3.0)              # leaf 2 mean 3    -> node (level 2) 1
    K[0, 0, 192:256, 0] = f2b(-2.0)             # leaf 3 mean -2
    P = o.build_pyramid(K)
    # K=2 at t in leaf 3: level 2 has candidates {0, 1} <= K, so both kept; leaves 0..3 candidates.
    r = o.select(Q, K, P, 2, np.array([[0, 0, N - 1]]), scale=1.0 / 8.0)
    assert list(r["idx"][0]) == [2, 3], r["idx"]
    # 8 leaves, K=2: level 3 has 2 nodes (kept), level 2 has 4 candidates, scored by the LSE
    # of their two leaf summaries (eq. 21).  Leaf logits (0..7): -3 3 | 1 1 | 1.5 1.5 | -3 -3.
    # node 0 = LSE(-3,3) = 3.0025, node 1 = LSE(1,1) = 1.693, node 2 = LSE(1.5,1.5) = 2.193,
    # node 3 = -2.307  ->  keep {0, 2} (gap 0.5).  Scoring a node by its own mean summary
    # would keep {1, 2} instead.  Leaves 0,1,4,5 are candidates; the own leaf 7 is added; the
    # best other leaf is 1 (logit 3, gap 1.5 to leaves 4/5).
    N = 64 * 8
    Q = np.zeros((1, N, 1, d), np.uint16)
    Q[0, :, 0, 0] = f2b(8.0)
    K = np.zeros((1, 1, N, d), np.uint16)
    for leaf, v in enumerate([-3.0, 3.0, 1.0, 1.0, 1.5, 1.5, -3.0, -3.0]):
        K[0, 0, 64 * leaf:64 * (leaf + 1), 0] = f2b(v)
    P = o.build_pyramid(K)
    r = o.select(Q, K, P, 2, np.array([[0, 0, N - 1]]), scale=1.0 / 8.0)
    assert list(r["s2"][0]) == [0, 2], r["s2"]
    assert list(r["cand"][0]) == [0, 1, 4, 5], r["cand"]
    assert list(r["idx"][0]) == [1, 7], r["idx"]
    assert abs(r["min_gap"][0] - 0.5) < 1e-12, r["min_gap"]


# ------------------------------------------------------------------------------------
# step 4: attention
# ------------------------------------------------------------------------------------
def pin_dense_equivalence(o):
    """K >= M_1 selects every eligible leaf, so the output is dense causal attention
    (textbook softmax over keys c <= t)."""
    for H_kv in (1, 2):
        Q, K, V = _tiny_inputs(seed=7, N=64 * 9 + 13, H_q=4, H_kv=H_kv)
        N, H_q, d = Q.shape[1], Q.shape[2], Q.shape[3]
        G = H_q // H_kv
        Ksel = (N + 63) // 64
        P = o.build_pyramid(K)
        sel = o.select(Q, K, P, Ksel, np.array([(0, g, t) for g in range(H_kv) for t in range(N)]))
        idx = sel["idx"].reshape(1, H_kv, N, Ksel)
        rows = np.array([(0, t) for t in range(0, N, 5)])
        O, LSE, ws = o.sparse_attention(Q, K, V, idx, rows)
        scale = 1.0 / math.sqrt(d)
        for i, (b, t) in enumerate(rows):
            for h in range(H_q):
                g = h // G
                z = scale * (b2f(K[0, g, :t + 1]) @ b2f(Q[0, t, h]))
                m = z.max()
                w = np.exp(z - m)
                lse = m + math.log(w.sum())
                out = (w / w.sum()) @ b2f(V[0, g, :t + 1])
                assert abs(LSE[i, h] - lse) < 1e-9, (t, h, LSE[i, h], lse)
                assert np.abs(O[i, h] - out).max() < 1e-9, (t, h)



def pin_dense_equivalence_noncausal(o):
    """Without the causal mask and with K >= M_1 every leaf is selected, so the output of every
    query is dense attention over all N keys (textbook softmax), ragged last leaf included."""
    Q, K, V = _tiny_inputs(seed=17, N=64 * 5 + 21, H_q=4, H_kv=2)
    N, H_q, d = Q.shape[1], Q.shape[2], Q.shape[3]
    H_kv = 2
    G = H_q // H_kv
    Ksel = (N + 63) // 64
    P = o.build_pyramid(K)
    sel = o.select(Q, K, P, Ksel, np.array([(0, g, t) for g in range(H_kv) for t in range(N)]), causal=False)
    idx = sel["idx"].reshape(1, H_kv, N, Ksel)
    assert np.all(idx == np.arange(Ksel))
    rows = np.array([(0, t) for t in range(0, N, 3)])
    O, LSE, _ = o.sparse_attention(Q, K, V, idx, rows, causal=False)
    scale = 1.0 / math.sqrt(d)
    for i, (b, t) in enumerate(rows):
        for h in range(H_q):
            g = h // G
            z = scale * (b2f(K[0, g]) @ b2f(Q[0, t, h]))
            m = z.max()
            w = np.exp(z - m)
            assert abs(LSE[i, h] - (m + math.log(w.sum()))) < 1e-9, (t, h)
            assert np.abs(O[i, h] - (w / w.sum()) @ b2f(V[0, g])).max() < 1e-9, (t, h)

def pin_weights_sum_to_one(o):
    Q, K, V = _tiny_inputs(seed=9)
    N = Q.shape[1]
    P = o.build_pyramid(K)
    sel = o.select(Q, K, P, 4, np.array([(0, 0, t) for t in range(N)]))
    _, _, ws = o.sparse_attention(Q, K, V, sel["idx"].reshape(1, 1, N, 4), np.array([(0, t) for t in range(N)]))
    assert np.all(np.abs(ws - 1.0) <= 1e-3)


def pin_single_block_at_start(o):
    """Only the own block selected and t its first key: the output is v_t itself."""
    Q, K, V = _tiny_inputs(seed=11, N=64 * 4)
    N = Q.shape[1]
    idx = np.full((1, 1, N, 1), -1, np.int32)
    idx[0, 0, :, 0] = np.arange(N) // 64
    rows = np.array([(0, t) for t in (0, 64, 128, 192)])
    O, LSE, _ = o.sparse_attention(Q, K, V, idx, rows)
    for i, (b, t) in enumerate(rows):
        for h in range(Q.shape[2]):
            assert np.array_equal(O[i, h], b2f(V[0, 0, t])), (t, h)
            z = (b2f(Q[0, t, h]) @ b2f(K[0, 0, t])) / math.sqrt(Q.shape[3])
            assert abs(LSE[i, h] - z) < 1e-12


# ------------------------------------------------------------------------------------
# step 3: decode
# ------------------------------------------------------------------------------------
def pin_decode(o):
    """Decode: the incrementally kept pyramid equals a full rebuild bit for bit, and each
    step's output equals the prefill row T over the same T+1 tokens."""
    rng = np.random.default_rng(13)
    B, H_q, H_kv, d, Ksel = 2, 4, 2, 32, 3
    N0, steps, N_cap = 60, 150, 256
    G = H_q // H_kv
    Kc = np.zeros((B, H_kv, N_cap, d), np.uint16)
    Vc = np.zeros((B, H_kv, N_cap, d), np.uint16)
    seq = np.array([N0, N0 + 5], np.int32)   # sequences of different lengths
    Kc[:, :, :N0 + 5] = random_bf16(rng, (B, H_kv, N0 + 5, d))
    Vc[:, :, :N0 + 5] = random_bf16(rng, (B, H_kv, N0 + 5, d))
    for b in range(B):
        Kc[b, :, seq[b]:] = 0
        Vc[b, :, seq[b]:] = 0
    Pc = np.concatenate([o.build_pyramid(Kc[b:b + 1], N=int(seq[b])) for b in range(B)])
    Qs = random_bf16(rng, (steps, B, H_q, d))
    ks = random_bf16(rng, (steps, B, H_kv, d))
    vs = random_bf16(rng, (steps, B, H_kv, d))
    for s in range(steps):
        T = seq.copy()
        out, lse, idx = o.decode_step(Qs[s], ks[s], vs[s], Kc, Vc, Pc, seq, Ksel)
        assert list(seq) == list(T + 1)
        for b in range(B):
            n = int(T[b]) + 1
            sizes = o.level_sizes(n)
            off_cap = level_offsets(o.level_sizes(N_cap))
            Pfull = o.build_pyramid(Kc[b:b + 1, :, :n].copy())
            off_n = level_offsets(sizes)
            for l, m in enumerate(sizes, start=1):
                assert np.array_equal(Pc[b, :, off_cap[l - 1]:off_cap[l - 1] + m], Pfull[0, :, off_n[l - 1]:off_n[l - 1] + m]), (s, b, l)
            if s % 37 == 0 or s == steps - 1:
                Qp = np.zeros((1, n, H_q, d), np.uint16)
                Qp[0, n - 1] = Qs[s, b]
                Kp, Vp = Kc[b:b + 1, :, :n].copy(), Vc[b:b + 1, :, :n].copy()
                sel = o.select(Qp, Kp, Pfull, Ksel, np.array([(0, g, n - 1) for g in range(H_kv)]))
                assert np.array_equal(sel["idx"], idx[b]), (s, b)
                idxf = np.full((1, H_kv, n, Ksel), -1, np.int32)
                idxf[0, :, n - 1] = sel["idx"]
                O, L, _ = o.sparse_attention(Qp, Kp, Vp, idxf, np.array([(0, n - 1)]))
                assert np.array_equal(O[0], out[b]) and np.array_equal(L[0], lse[b]), (s, b)



def pin_decode_scoring_variants(o):
    """Decode under the PISA-1 and PISA-2 block scores: each step's selection and output equal
    the prefill row over the same tokens under the same score (the walk prunes: M_1 > g K), and
    on these inputs the two scores select differently from the LSE on some steps."""
    rng = np.random.default_rng(29)
    B, H_q, H_kv, d, Ksel, N0, steps, N_cap = 1, 4, 2, 32, 2, 64 * 9 + 5, 12, 1024
    K0 = random_bf16(rng, (B, H_kv, N0, d))
    V0 = random_bf16(rng, (B, H_kv, N0, d))
    Qs = random_bf16(rng, (steps, B, H_q, d), 2.0)
    ks = random_bf16(rng, (steps, B, H_kv, d))
    vs = random_bf16(rng, (steps, B, H_kv, d))
    picks = {}
    for scoring in (0, 1, 2):
        Kc = np.zeros((B, H_kv, N_cap, d), np.uint16)
        Vc = np.zeros((B, H_kv, N_cap, d), np.uint16)
        Kc[:, :, :N0], Vc[:, :, :N0] = K0, V0
        Pc = o.build_pyramid(Kc, N=N0)
        seq = np.array([N0], np.int32)
        picks[scoring] = []
        for s in range(steps):
            n = int(seq[0]) + 1
            out, lse, idx = o.decode_step(Qs[s], ks[s], vs[s], Kc, Vc, Pc, seq, Ksel, scoring=scoring)
            picks[scoring].append(idx.copy())
            Qp = np.zeros((1, n, H_q, d), np.uint16)
            Qp[0, n - 1] = Qs[s, 0]
            Kp, Vp = Kc[:, :, :n].copy(), Vc[:, :, :n].copy()
            sel = o.select(Qp, Kp, o.build_pyramid(Kp), Ksel, np.array([(0, g, n - 1) for g in range(H_kv)]),
                           scoring=scoring)
            assert np.array_equal(sel["idx"], idx[0]), (scoring, s)
            idxf = np.full((1, H_kv, n, Ksel), -1, np.int32)
            idxf[0, :, n - 1] = sel["idx"]
            O, L, _ = o.sparse_attention(Qp, Kp, Vp, idxf, np.array([(0, n - 1)]))
            assert np.array_equal(O[0], out[0]) and np.array_equal(L[0], lse[0]), (scoring, s)
    for scoring in (1, 2):
        assert any(not np.array_equal(a, b) for a, b in zip(picks[0], picks[scoring])), scoring


# ------------------------------------------------------------------------------------
# BSA flat selection (the single-level baseline of the paper's selection-speed figure)
# ------------------------------------------------------------------------------------
def _bsa_constant_blocks(c, d=16, lanes=(0,)):
    """Keys of block j all equal to sum over lane e of c[e][j] * unit vector e (bf16-exact), so
    the block's mean summary is exactly that vector."""
    M = len(c[0])
    K = np.zeros((1, 1, 64 * M, d), np.float32)
    for e, ce in zip(lanes, c):
        for j in range(M):
            K[0, 0, 64 * j:64 * (j + 1), e] = ce[j]
    return f2b(K)


def pin_bsa_closed_form(o):
    """Blocks of constant keys c_j along one axis and queries along that axis: every BSA score is
    G_Q * scale * (q . axis) * c_j, so the selection is the own block plus the K - 1 largest (or,
    for a negative query, smallest) c_j among the earlier blocks; a second head on another axis
    enters the head sum and changes the ranking."""
    c = [3.0, -1.0, 5.0, 2.0, 7.0, 0.5, 4.0, 6.0]
    d, N = 16, 64 * 8
    K = _bsa_constant_blocks([c], d)
    P = o.build_pyramid(K)
    Q = np.zeros((1, N, 1, d), np.float32)
    Q[0, :, 0, 0] = 1.0
    Qp = f2b(Q)
    rows = np.array([(0, 0, t) for t in (511, 200, 64, 10)], np.int64)
    r = o.select_bsa(Qp, P, 3, rows, want_scores=True)
    assert [list(x) for x in r["idx"]] == [[2, 4, 7], [0, 2, 3], [0, 1, -1], [0, -1, -1]], r["idx"]
    assert abs(r["score"][0, 4] - 7.0 / 4.0) < 1e-12 and np.isneginf(r["score"][0, 7])   # own block not ranked
    assert abs(r["min_gap"][0] - (5.0 - 4.0) / 4.0) < 1e-12
    nc = o.select_bsa(Qp, P, 3, np.array([[0, 0, 0]]), causal=False)
    assert list(nc["idx"][0]) == [2, 4, 7], nc["idx"]
    Q[0, :, 0, 0] = -1.0
    neg = o.select_bsa(f2b(Q), P, 3, rows[:1])
    assert list(neg["idx"][0]) == [1, 5, 7], neg["idx"]
    # two heads: head 0 along axis 0 (weight 2), head 1 along axis 1; block j's keys are
    # c_j on axis 0 and b_j on axis 1, so the head sum ranks by 2 c_j + b_j
    b = [9.0, 0.0, -6.0, 0.0, -8.0, 0.0, 0.0, 0.0]
    K2 = _bsa_constant_blocks([c, b], d, lanes=(0, 1))
    P2 = o.build_pyramid(K2)
    Q2 = np.zeros((1, N, 2, d), np.float32)
    Q2[0, :, 0, 0] = 2.0
    Q2[0, :, 1, 1] = 1.0
    r2 = o.select_bsa(f2b(Q2), P2, 3, rows[:1])
    # 2c + b over blocks 0..6: 15, -2, 4, 4, 6, 1, 8 -> the best two are 0 and 6
    assert list(r2["idx"][0]) == [0, 6, 7], r2["idx"]
    # identical blocks: every score ties and the lower indices win
    Kt = _bsa_constant_blocks([[2.0] * 8], d)
    rt = o.select_bsa(Qp, o.build_pyramid(Kt), 3, rows)
    assert [list(x) for x in rt["idx"]] == [[0, 1, 7], [0, 1, 3], [0, 1, -1], [0, -1, -1]], rt["idx"]


def _bsa_exact_mean_inputs(seed, N, H_q, H_kv=1, d=32):
    """Keys whose block means are exact bf16 values: each block holds an offset o_j and
    pairs of keys o_j + r, o_j - r (all multiples of 1/64 below 4 in magnitude, exact in bf16),
    so the fp64 mean over any complete block, and its bf16 summary, equal o_j exactly."""
    rng = np.random.default_rng(seed)
    M1 = (N + 63) // 64
    o_ = rng.integers(-64, 65, size=(1, H_kv, M1, d)) / 64.0
    r = rng.integers(-60, 61, size=(1, H_kv, M1, 32, d)) / 64.0
    blk = np.concatenate([o_[:, :, :, None, :] + r, o_[:, :, :, None, :] - r], axis=3)   # [.., M1, 64, d]
    K = blk.reshape(1, H_kv, M1 * 64, d)[:, :, :N].astype(np.float32)
    Q = (rng.integers(-64, 65, size=(1, N, H_q, d)) / 32.0).astype(np.float32)
    return f2b(Q), f2b(K)


def pin_bsa_equals_pisa1_leaf_ranking(o):
    """PISA-1 scores a leaf by log m + mean of its m visible logits = log m + scale q . mean(k)
    (summary page, "Core method": mean scoring is the first-order truncation of the LSE); with
    no pruning (M_1 <= g K every eligible leaf is a candidate) and full blocks (every ranked
    block in causal mode ends before the query), PISA-1 ranks exactly by BSA's q . kbar.  With
    keys whose block means are exact in bf16 the two selections must be identical."""
    for (N, H_q, H_kv, Ksel, causal) in ((1024, 4, 1, 8, True), (64 * 12, 2, 2, 7, True), (64 * 11 + 64, 4, 1, 6, False)):
        Q, K = _bsa_exact_mean_inputs(7 + N, N, H_q, H_kv)
        P = o.build_pyramid(K)
        M1 = (N + 63) // 64
        assert M1 <= 2 * Ksel
        rows = np.array([(0, g, t) for g in range(H_kv) for t in range(0, N, 5)], np.int64)
        b = o.select_bsa(Q, P, Ksel, rows, causal=causal)
        p1 = o.select(Q, K, P, Ksel, rows, causal=causal, scoring=1)
        ok = (b["min_gap"] > 1e-9) & (p1["min_gap"] > 1e-9)
        assert ok.mean() > 0.95, ok.mean()
        assert np.array_equal(b["idx"][ok], p1["idx"][ok]), (N, np.where(~np.all(b["idx"] == p1["idx"], 1))[0][:3])


def pin_bsa_invariants(o):
    """Final sets ascending, unique, -1 padded at the end, own block present and every block
    eligible (causal); |I_t| = min(K, #eligible); K >= M_1 selects every eligible block."""
    Q, K, V = _tiny_inputs(seed=23)
    P = o.build_pyramid(K)
    N = Q.shape[1]
    rows = np.array([(0, 0, t) for t in range(N)], np.int64)
    for Ksel in (1, 5, 16):
        r = o.select_bsa(Q, P, Ksel, rows)
        for t in range(N):
            row = list(r["idx"][t])
            val = [x for x in row if x >= 0]
            assert row == val + [-1] * (Ksel - len(val))
            assert val == sorted(set(val)) and t // 64 in val and all(x * 64 <= t for x in val)
            assert len(val) == min(Ksel, t // 64 + 1)
            if Ksel >= 16:
                assert val == list(range(t // 64 + 1))

ALL_PINS = [
    pin_level_sizes, pin_bf16_rounding, pin_pyramid_constant_keys, pin_pyramid_raw_mean,
    pin_pyramid_ragged_leaf_mean, pin_leaf_lse_closed_forms, pin_gqa_head_sum, pin_lse_beats_mean,
    pin_ties_lower_index, pin_admissible_sets, pin_brute_force_topk, pin_brute_force_topk_noncausal, pin_final_set_invariants,
    pin_walk_prunes_by_summary_lse, pin_dense_equivalence, pin_dense_equivalence_noncausal, pin_weights_sum_to_one,
    pin_single_block_at_start, pin_decode, pin_decode_scoring_variants,
    pin_scoring_variants_closed_forms, pin_scoring_variants_order, pin_mean_scoring_ranks_like_the_mean,
    pin_backward_dense_autograd, pin_backward_dense_autograd_noncausal, pin_backward_finite_differences,
    pin_backward_sums, pin_backward_sampled_equals_full, pin_bsa_closed_form, pin_bsa_equals_pisa1_leaf_ranking, pin_bsa_invariants,
]
