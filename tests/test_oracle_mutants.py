"""Planted mistakes in the CPU oracle must each fail at least one pin.

Each mutant is a copy of the oracle source with one plausible error (a dropped term, a
wrong sign, index or mask, a missed rounding step), compiled into a temporary library and
run against every pin in a child process (a mutant may also crash, which counts as caught).
This shows the pins are sensitive enough that a mistake of that kind cannot pass.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

MUTANTS = {
    "mean_instead_of_lse": [("return m + std::log(s);",
                             "double mu = 0; for (double v : z) mu += v; return std::log((double)z.size()) + mu / z.size();")],
    "leaf_causal_mask_dropped": [("if (!R.causal || c <= R.t) z.push_back(R.scale * dot_key(R, h, c));",
                                  "z.push_back(R.scale * dot_key(R, h, c));")],
    "level_mean_divides_by_g": [("      double cnt = (double)(r1 - r0);\n      for (int e = 0; e < d; ++e) Pbg[(off[l] + i) * d + e]",
                                 "      double cnt = (double)g;\n      for (int e = 0; e < d; ++e) Pbg[(off[l] + i) * d + e]")],
    "ragged_leaf_divides_by_C": [("    double cnt = (double)(c1 - c0);\n    for (int e = 0; e < d; ++e) Pbg[(off[1] + j) * d + e]",
                                  "    double cnt = (double)C;\n    for (int e = 0; e < d; ++e) Pbg[(off[1] + j) * d + e]")],
    "ties_to_higher_index": [("return ids[a] < ids[b];", "return ids[a] > ids[b];")],
    "topk_ascending": [("if (sc[a] != sc[b]) return sc[a] > sc[b];", "if (sc[a] != sc[b]) return sc[a] < sc[b];")],
    "own_block_not_forced": [("if (out.cand[s] >= 0 && out.cand[s] != own) {", "if (out.cand[s] >= 0) {"),
                             ("fin = topk(ids, sc, R.causal ? R.K - 1 : R.K, &gap);", "fin = topk(ids, sc, R.K, &gap);"),
                             ("  if (R.causal) fin.push_back(own);\n", "")],
    "children_off_by_one": [("    for (long long r = R.g * p; r < R.g * p + R.g; ++r)\n      if (eligible(R, l, r)) out.push_back(r);",
                             "    for (long long r = R.g * p + 1; r < R.g * p + R.g + 1; ++r)\n      if (eligible(R, l, r)) out.push_back(r);")],
    "attention_scale_missing": [("      s.push_back(scale * z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;",
                                 "      s.push_back(z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;")],
    "eligibility_by_last_key": [("return i * ipow(R.g, l - 1) * R.C <= R.t;",
                                 "return ((i + 1) * ipow(R.g, l - 1) * R.C - 1) <= R.t;")],
    "decode_skips_ancestors": [("      for (int l = 2; l <= lv.L; ++l) {\n        node /= g;",
                                "      for (int l = 2; l <= 1; ++l) {\n        node /= g;")],
    "attention_ignores_causal": [("      if (causal && c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;",
                                  "      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;")],
    "double_rounding_to_bf16": [("if (std::isfinite(f) && (double)f != x) {", "if (false) {")],
    "leaf_scored_by_summary": [("if (!R.causal || c <= R.t) z.push_back(R.scale * dot_key(R, h, c));",
                                "if (!R.causal || c <= R.t) z.push_back(R.scale * dot_node(R, h, 1, j));")],
    "internal_scored_by_own_summary": [("if (eligible(R, l - 1, r)) z.push_back(R.scale * dot_node(R, h, l - 1, r));",
                                        "if (eligible(R, l - 1, r)) z.push_back(R.scale * dot_node(R, h, l, i));")],
    "walk_never_prunes": [("    if ((int)A.size() > R.K) {\n      std::vector<double> sc;\n      for (long long i : A) sc.push_back(score_internal(R, l, i));\n      double gap;",
                           "    if (false) {\n      std::vector<double> sc;\n      for (long long i : A) sc.push_back(score_internal(R, l, i));\n      double gap;")],
}

# the ablation scorings (PISA-1 / PISA-2)
MUTANTS["variant_drops_log_m"] = [("  double s = std::log(m) + mean;", "  double s = mean;")]
MUTANTS["variance_sample_divisor"] = [("    s += 0.5 * var / m;", "    s += 0.5 * var / (m > 1 ? m - 1 : 1);")]
MUTANTS["variance_not_halved"] = [("    s += 0.5 * var / m;", "    s += var / m;")]
MUTANTS["pisa1_adds_variance"] = [("  if (scoring == 2) {", "  if (scoring >= 1) {")]

# the backward of step 4
MUTANTS["backward_drops_D"] = [("    const double dS = P[i] * (dP - D);", "    const double dS = P[i] * dP;")]
MUTANTS["backward_dk_without_scale"] = [("      if (dK) dK[c * d + e] += scale * dS * q[e];",
                                         "      if (dK) dK[c * d + e] += dS * q[e];")]
MUTANTS["backward_dv_uses_dS"] = [("      if (dV) dV[c * d + e] += P[i] * dO[e];", "      if (dV) dV[c * d + e] += dS * dO[e];")]
MUTANTS["backward_ignores_causal"] = [("      if (causal && c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  if (pos.empty()) return;",
                                       "      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  if (pos.empty()) return;")]

# the non-causal mode (every block a candidate, none forced, no key masked)
MUTANTS["noncausal_leaf_masked"] = [("if (!R.causal || c <= R.t) z.push_back(R.scale * dot_key(R, h, c));",
                                     "if (c <= R.t) z.push_back(R.scale * dot_key(R, h, c));")]
MUTANTS["noncausal_eligibility_masked"] = [("  if (!R.causal) return true;\n  return i * ipow(R.g, l - 1) * R.C <= R.t;",
                                            "  return i * ipow(R.g, l - 1) * R.C <= R.t;")]
MUTANTS["noncausal_own_forced"] = [
    ("  long long own = R.causal ? R.t / R.C : -1;\n  for (size_t s = 0; s < out.cand.size(); ++s)\n    if (out.cand[s] >= 0 && out.cand[s] != own) {",
     "  long long own = R.t / R.C;\n  for (size_t s = 0; s < out.cand.size(); ++s)\n    if (out.cand[s] >= 0 && out.cand[s] != own) {"),
    ("fin = topk(ids, sc, R.causal ? R.K - 1 : R.K, &gap);", "fin = topk(ids, sc, R.K - 1, &gap);"),
    ("  if (R.causal) fin.push_back(own);\n", "  fin.push_back(own);\n")]
MUTANTS["attention_noncausal_masked"] = [("      if (causal && c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;",
                                          "      if (c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  for (int e = 0; e < d; ++e) o[e] = 0;")]
MUTANTS["backward_noncausal_masked"] = [("      if (causal && c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  if (pos.empty()) return;",
                                         "      if (c > t) continue;\n      double z = 0;\n      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);\n      pos.push_back(c);\n      s.push_back(scale * z);\n    }\n  if (pos.empty()) return;")]
MUTANTS["decode_ignores_scoring"] = [("n, T, d, C, g, Ksel, GQ, 1, scale, scoring);\n      Selection S = select_row(R);",
                                      "n, T, d, C, g, Ksel, GQ, 1, scale, 0);\n      Selection S = select_row(R);")]

# the admissibility check behind the parity rule for near-ties
MUTANTS["admissible_accepts_anything"] = [("    if (f == target) return 1;", "    return 1;")]
MUTANTS["admissible_without_tolerance"] = [("    if (mn >= mx - tol) {", "    if (mn > mx) {")]
MUTANTS["admissible_drops_own_block"] = [("    if (R.causal) f.push_back(own);", "")]
MUTANTS["admissible_ignores_scoring"] = [("GQ, causal, scale, scoring);\n      std::vector<long long> target;",
                                          "GQ, causal, scale, 0);\n      std::vector<long long> target;")]
MUTANTS["admissible_noncausal_forces_own"] = [
    ("  long long own = R.causal ? R.t / R.C : -1;\n  for (long long p : S)", "  long long own = R.t / R.C;\n  for (long long p : S)"),
    ("admissible_sets(ids, sc, R.causal ? R.K - 1 : R.K, tol, sets, 4096);", "admissible_sets(ids, sc, R.K - 1, tol, sets, 4096);"),
    ("    if (R.causal) f.push_back(own);", "    f.push_back(own);")]

# "head_sum_drops_heads" needs two edits (internal and leaf scores): sum only head 0
MUTANTS["head_sum_drops_heads"] = [
    ("  double u = 0;\n  for (int h = 0; h < R.GQ; ++h) {\n    std::vector<double> z;\n    for (long long r",
     "  double u = 0;\n  for (int h = 0; h < 1; ++h) {\n    std::vector<double> z;\n    for (long long r"),
    ("  double u = 0;\n  for (int h = 0; h < R.GQ; ++h) {\n    std::vector<double> z;\n    for (long long c",
     "  double u = 0;\n  for (int h = 0; h < 1; ++h) {\n    std::vector<double> z;\n    for (long long c"),
]


# the BSA flat selection (the baseline of the selection-speed comparison)
MUTANTS["bsa_sign_flipped"] = [("    for (int h = 0; h < R.GQ; ++h) u += R.scale * dot_node(R, h, 1, j);",
                                "    for (int h = 0; h < R.GQ; ++h) u -= R.scale * dot_node(R, h, 1, j);")]
MUTANTS["bsa_level2_summaries"] = [("    for (int h = 0; h < R.GQ; ++h) u += R.scale * dot_node(R, h, 1, j);",
                                    "    for (int h = 0; h < R.GQ; ++h) u += R.scale * dot_node(R, h, 2, j / 2);")]
MUTANTS["bsa_first_head_only"] = [("    for (int h = 0; h < R.GQ; ++h) u += R.scale * dot_node(R, h, 1, j);",
                                   "    for (int h = 0; h < 1; ++h) u += R.scale * dot_node(R, h, 1, j);")]
MUTANTS["bsa_own_not_forced"] = [("    if (!eligible(R, 1, j) || j == own) continue;", "    if (!eligible(R, 1, j)) continue;"),
                                 ("  const int keep = R.causal ? R.K - 1 : R.K;", "  const int keep = R.K;"),
                                 ("  if (R.causal) ranked.push_back(own);", "")]
MUTANTS["bsa_ignores_causal"] = [("    if (!eligible(R, 1, j) || j == own) continue;", "    if (j == own) continue;")]
MUTANTS["bsa_ties_to_higher_index"] = [("    double u = 0;\n    for (int h = 0; h < R.GQ; ++h) u += R.scale",
                                        "    double u = 1e-12 * j;\n    for (int h = 0; h < R.GQ; ++h) u += R.scale")]


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def _mutant_source(name):
    src = open(oracle.SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
        src = src.replace(old, new)
    return src


@pytest.fixture(scope="module")
def mutant_libs(mutant_dir):
    """Every mutant compiled once, the independent g++ runs side by side; each test takes its
    own result (a missing mutation site raises there)."""
    def build(name):
        path = os.path.join(mutant_dir, f"{name}.cpp")
        with open(path, "w") as f:
            f.write(_mutant_source(name))
        return oracle.compile_source(path, os.path.join(mutant_dir, f"lib{name}.so"))

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        futures = {name: ex.submit(build, name) for name in MUTANTS}
        return {name: fut.exception() or fut.result() for name, fut in futures.items()}


RUNNER = """
import sys
sys.path[:0] = [{root!r}, {here!r}]
import oracle, pins
o = oracle.Oracle({lib!r})
failed = []
for pin in pins.ALL_PINS:
    try:
        pin(o)
    except Exception as e:
        failed.append(pin.__name__)
        break  # one failing pin is enough to catch the mutant
print("FAILED_PINS", ",".join(failed))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_libs):
    lib = mutant_libs[name]
    if isinstance(lib, BaseException):
        raise lib
    code = RUNNER.format(root=os.path.dirname(HERE), here=HERE, lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    failed = [ln.split(" ", 1)[1] for ln in res.stdout.splitlines() if ln.startswith("FAILED_PINS ")]
    caught = res.returncode != 0 or (failed and failed[0].strip() != "")
    assert caught, f"no pin catches the planted mistake {name}: {res.stdout[-500:]}"
