// PISA oracle: a plain, slow CPU implementation of pyramid-LSE block-sparse attention.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
// file; it exists so that the GPU library can be checked against an independent
// statement of what the method computes.  It shares no code, header, table or helper
// with the GPU library.
//
// Source of every step: "Block Sparse Attention with Log-Linear Complexity" (Tang, Qin,
// Pan, Li, Liu), read through its summary page, sections "Core method" (eq. 21) and
// "Method step details" (step 1: pyramid, eqs 10-15; step 2: coarse-to-fine selection
// with GQA head sum, eq. 22, SelectK, exact leaf LSE and a final top-K; step 3: decode
// with incremental leaf/ancestor update; step 4: attention over the selected blocks).
// The rule that the softmax runs over the connected positions only, with weights that
// sum to one, is from the blog post of the same title, section 3.3.
//
// Readings where the pages are silent (each is listed in the design notes):
//  R1 summaries are means of the children's stored bf16 summaries, accumulated in fp64
//     and rounded once to bf16 (round to nearest even); the leaf mean divides by the
//     actual key count of a ragged last leaf.
//  R2 causal eligibility: a node is eligible for query t iff its first key index <= t.
//     Summaries stay the static means of their full blocks.
//  R3 levels are numbered from the leaves: level 1 = leaf blocks of C keys, level L is
//     the single root.  A level-l candidate is scored with the LSE of its eligible
//     level-(l-1) children (eq. 21); the level walk keeps all candidates while there are
//     at most K of them.
//  R4 the query's own leaf is scored like any candidate but never ranked.
//  R5 the own leaf always belongs to the final set and counts toward K (causal mode).
//  R6 ties rank the lower block index first.
//  R7 attention output is rounded to bf16 by the caller; here it is returned in fp64.
//  R8 decode recomputes the new token's leaf and every ancestor from stored values, so
//     the cache pyramid equals a fresh build bit for bit.
//  R9 scores are natural-log LSEs, summed over the group's heads without weights;
//     logits are scale * q.k with scale = 1/sqrt(d) unless given.
//  R10 the two ablation scorings are the first- and second-order truncations of the
//     LSE's expansion around the mean of the block's m eligible child logits z ("Core
//     method", eqs. 32-34): PISA-1 = log m + mean(z), PISA-2 = log m + mean(z) +
//     Var(z) / 2 with the population variance (divisor m).  They replace the LSE at
//     every scored level and at the exact leaf level; the head sum, SelectK and the
//     final top-K are unchanged.
//
// Precision: bf16 inputs are widened exactly; every sum, exp and log is fp64.
// Parallelism: independent rows are split across std::threads; every output element is
// written by exactly one thread, so results do not depend on the thread count.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double NEG_INF = -std::numeric_limits<double>::infinity();
const double POS_INF = std::numeric_limits<double>::infinity();

double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// fp64 -> bf16, round to nearest even, without double rounding: round to float with
// round-to-odd first (float keeps 16 more bits than bf16), then to bf16.
uint16_t f64_to_bf16_rne(double x) {
  if (std::isnan(x)) return 0x7FC0;
  float f = (float)x;
  if (std::isfinite(f) && (double)f != x) {
    if (std::fabs((double)f) > std::fabs(x)) f = std::nextafter(f, 0.0f);
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u |= 1u;
    std::memcpy(&f, &u, 4);
  }
  return f32_to_bf16_rne(f);
}

// ---------------------------------------------------------------------------------------
// pyramid geometry
// ---------------------------------------------------------------------------------------
struct Levels {
  int L = 0;                    // number of levels; level l in [1, L]
  std::vector<long long> M;     // M[l] = nodes at level l (M[0] unused)
};

Levels level_sizes(long long n, int C, int g) {
  Levels lv;
  lv.M.push_back(0);
  if (n <= 0) return lv;
  long long m = (n + C - 1) / C;
  lv.M.push_back(m);
  while (m > 1) {
    m = (m + g - 1) / g;
    lv.M.push_back(m);
  }
  lv.L = (int)lv.M.size() - 1;
  return lv;
}

// node offsets of the stored layout (from the capacity), off[l] for l in [1, L]
std::vector<long long> level_offsets(long long n_cap, int C, int g) {
  Levels lv = level_sizes(n_cap, C, g);
  std::vector<long long> off(lv.L + 2, 0);
  for (int l = 1; l <= lv.L; ++l) off[l + 1] = off[l] + lv.M[l];
  return off;
}

long long ipow(long long b, int e) {
  long long r = 1;
  for (int i = 0; i < e; ++i) r *= b;
  return r;
}

void run_parallel(long long n, int nthreads, const std::function<void(long long, long long)>& fn) {
  if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (n <= 0) return;
  if (nthreads == 1 || n == 1) {
    fn(0, n);
    return;
  }
  nthreads = (int)std::min<long long>(nthreads, n);
  std::vector<std::thread> th;
  for (int i = 0; i < nthreads; ++i) {
    long long a = n * i / nthreads, b = n * (i + 1) / nthreads;
    th.emplace_back([&fn, a, b] { fn(a, b); });
  }
  for (auto& t : th) t.join();
}

// ---------------------------------------------------------------------------------------
// step 1: the key pyramid (eqs 10-15)
// ---------------------------------------------------------------------------------------
// Kbg: rows of one (b, h_kv), row c at Kbg + c*d.  Pbg: nodes in the capacity layout.
// Writes leaf j (level 1) and, for every level above, node i = mean of its children.
void build_one(const uint16_t* Kbg, uint16_t* Pbg, long long n, const std::vector<long long>& off, int d, int C,
               int g) {
  Levels lv = level_sizes(n, C, g);
  if (lv.L == 0) return;
  std::vector<double> acc(d);
  for (long long j = 0; j < lv.M[1]; ++j) {
    long long c0 = j * C, c1 = std::min<long long>(n, c0 + C);
    std::fill(acc.begin(), acc.end(), 0.0);
    for (long long c = c0; c < c1; ++c)
      for (int e = 0; e < d; ++e) acc[e] += bf16_to_f64(Kbg[c * d + e]);
    double cnt = (double)(c1 - c0);
    for (int e = 0; e < d; ++e) Pbg[(off[1] + j) * d + e] = f64_to_bf16_rne(acc[e] / cnt);
  }
  for (int l = 2; l <= lv.L; ++l) {
    for (long long i = 0; i < lv.M[l]; ++i) {
      long long r0 = g * i, r1 = std::min<long long>(lv.M[l - 1], g * i + g);
      std::fill(acc.begin(), acc.end(), 0.0);
      for (long long r = r0; r < r1; ++r)
        for (int e = 0; e < d; ++e) acc[e] += bf16_to_f64(Pbg[(off[l - 1] + r) * d + e]);
      double cnt = (double)(r1 - r0);
      for (int e = 0; e < d; ++e) Pbg[(off[l] + i) * d + e] = f64_to_bf16_rne(acc[e] / cnt);
    }
  }
}

// ---------------------------------------------------------------------------------------
// selection for one query row (steps 2, eqs 16-22, and the final top-K)
// ---------------------------------------------------------------------------------------
struct Row {
  const uint16_t* Kbg;                 // raw keys of this (b, h_kv)
  const uint16_t* Pbg;                 // pyramid of this (b, h_kv), capacity layout
  const std::vector<long long>* off;
  Levels lv;                           // level sizes for n tokens
  long long n, t;
  int d, C, g, K, GQ;
  bool causal;
  double scale;
  int scoring;                         // 0 LSE, 1 PISA-1, 2 PISA-2
  std::vector<double> q;               // GQ x d, widened
};

bool eligible(const Row& R, int l, long long i) {
  if (i < 0 || i >= R.lv.M[l]) return false;
  if (!R.causal) return true;
  return i * ipow(R.g, l - 1) * R.C <= R.t;
}

double dot_node(const Row& R, int h, int l, long long i) {
  const uint16_t* p = R.Pbg + ((*R.off)[l] + i) * R.d;
  double s = 0;
  for (int e = 0; e < R.d; ++e) s += R.q[h * R.d + e] * bf16_to_f64(p[e]);
  return s;
}

double dot_key(const Row& R, int h, long long c) {
  const uint16_t* k = R.Kbg + c * R.d;
  double s = 0;
  for (int e = 0; e < R.d; ++e) s += R.q[h * R.d + e] * bf16_to_f64(k[e]);
  return s;
}

double logsumexp(const std::vector<double>& z) {
  if (z.empty()) return NEG_INF;
  double m = *std::max_element(z.begin(), z.end());
  if (m == NEG_INF) return NEG_INF;
  double s = 0;
  for (double v : z) s += std::exp(v - m);
  return m + std::log(s);
}

// The score of one block from its m eligible child logits z: the LSE (eq. 21), or its
// first- (PISA-1) or second-order (PISA-2) truncation around the mean (reading R10).
double block_score(const std::vector<double>& z, int scoring) {
  if (scoring == 0) return logsumexp(z);
  if (z.empty()) return NEG_INF;
  const double m = (double)z.size();
  double mean = 0;
  for (double v : z) mean += v;
  mean /= m;
  double s = std::log(m) + mean;
  if (scoring == 2) {
    double var = 0;
    for (double v : z) var += (v - mean) * (v - mean);
    s += 0.5 * var / m;
  }
  return s;
}

// eq. 21 for a level-l candidate (l >= 2): the score of its eligible level-(l-1) children,
// summed over the group's heads (eq. 22).
double score_internal(const Row& R, int l, long long i) {
  double u = 0;
  for (int h = 0; h < R.GQ; ++h) {
    std::vector<double> z;
    for (long long r = R.g * i; r < R.g * i + R.g; ++r)
      if (eligible(R, l - 1, r)) z.push_back(R.scale * dot_node(R, h, l - 1, r));
    u += block_score(z, R.scoring);
  }
  return u;
}

// eq. 21 at the leaf level: exact LSE over the raw keys of leaf j (causal: keys <= t),
// summed over heads.
double score_leaf(const Row& R, long long j) {
  long long c0 = j * R.C, c1 = std::min<long long>(R.n, c0 + R.C);
  double u = 0;
  for (int h = 0; h < R.GQ; ++h) {
    std::vector<double> z;
    for (long long c = c0; c < c1; ++c)
      if (!R.causal || c <= R.t) z.push_back(R.scale * dot_key(R, h, c));
    u += block_score(z, R.scoring);
  }
  return u;
}

// top-k of (id, score) by score descending, ties to the lower id; result ascending by id.
// gap = k-th best minus (k+1)-th best score (infinite if there are at most k candidates).
std::vector<long long> topk(const std::vector<long long>& ids, const std::vector<double>& sc, int k, double* gap) {
  std::vector<int> ord(ids.size());
  for (size_t i = 0; i < ids.size(); ++i) ord[i] = (int)i;
  std::sort(ord.begin(), ord.end(), [&](int a, int b) {
    if (sc[a] != sc[b]) return sc[a] > sc[b];
    return ids[a] < ids[b];
  });
  if (gap) *gap = ((int)ids.size() > k && k > 0) ? sc[ord[k - 1]] - sc[ord[k]] : POS_INF;
  std::vector<long long> out;
  for (int i = 0; i < (int)ord.size() && i < k; ++i) out.push_back(ids[ord[i]]);
  std::sort(out.begin(), out.end());
  return out;
}

std::vector<long long> eligible_children(const Row& R, int l, const std::vector<long long>& parents) {
  std::vector<long long> out;
  for (long long p : parents)
    for (long long r = R.g * p; r < R.g * p + R.g; ++r)
      if (eligible(R, l, r)) out.push_back(r);
  return out;
}

struct Selection {
  std::vector<long long> S2;          // survivors at level 2 (ascending)
  std::vector<long long> cand;        // slot g*i + c -> leaf or -1
  std::vector<double> cand_score;     // slot -> leaf score or -inf
  std::vector<long long> final_set;   // ascending
  double min_gap = POS_INF;
};

Selection select_row(const Row& R) {
  Selection out;
  if (R.lv.L == 0) return out;
  std::vector<long long> S = {0};  // the root at level L
  for (int l = R.lv.L - 1; l >= 2; --l) {
    std::vector<long long> A = eligible_children(R, l, S);
    if ((int)A.size() > R.K) {
      std::vector<double> sc;
      for (long long i : A) sc.push_back(score_internal(R, l, i));
      double gap;
      S = topk(A, sc, R.K, &gap);
      out.min_gap = std::min(out.min_gap, gap);
    } else {
      S = A;
    }
  }
  out.S2 = S;
  // leaf candidates: eligible children of the level-2 survivors, slot g*i + c
  out.cand.assign((size_t)R.g * R.K, -1);
  out.cand_score.assign((size_t)R.g * R.K, NEG_INF);
  std::vector<long long> A1;
  for (size_t i = 0; i < S.size(); ++i)
    for (int c = 0; c < R.g; ++c) {
      long long j = R.g * S[i] + c;
      if (eligible(R, 1, j)) {
        out.cand[R.g * i + c] = j;
        out.cand_score[R.g * i + c] = score_leaf(R, j);
        A1.push_back(j);
      }
    }
  // final top-K over exact leaf scores
  std::vector<long long> ids;
  std::vector<double> sc;
  long long own = R.causal ? R.t / R.C : -1;
  for (size_t s = 0; s < out.cand.size(); ++s)
    if (out.cand[s] >= 0 && out.cand[s] != own) {
      ids.push_back(out.cand[s]);
      sc.push_back(out.cand_score[s]);
    }
  double gap;
  std::vector<long long> fin = topk(ids, sc, R.causal ? R.K - 1 : R.K, &gap);
  out.min_gap = std::min(out.min_gap, gap);
  if (R.causal) fin.push_back(own);
  std::sort(fin.begin(), fin.end());
  out.final_set = fin;
  return out;
}

// all size-k subsets S of the candidates with  min_{S} score >= max_{not S} score - tol
void admissible_sets(const std::vector<long long>& ids, const std::vector<double>& sc, int k, double tol,
                     std::vector<std::vector<long long>>& out, size_t cap) {
  int n = (int)ids.size();
  if (n <= k) {
    std::vector<long long> all = ids;
    std::sort(all.begin(), all.end());
    out.push_back(all);
    return;
  }
  std::vector<double> s = sc;
  std::sort(s.begin(), s.end(), std::greater<double>());
  double sk = s[k - 1], sk1 = s[k];
  std::vector<int> sure, band;
  for (int i = 0; i < n; ++i) {
    if (sc[i] > sk1 + tol) sure.push_back(i);
    else if (sc[i] >= sk - tol) band.push_back(i);
  }
  int need = k - (int)sure.size();
  if (need < 0 || need > (int)band.size()) return;
  std::vector<int> pick(band.size(), 0);
  std::fill(pick.begin(), pick.begin() + need, 1);
  std::sort(pick.begin(), pick.end(), std::greater<int>());
  do {
    std::vector<char> in(n, 0);
    for (int i : sure) in[i] = 1;
    for (size_t b = 0; b < band.size(); ++b)
      if (pick[b]) in[band[b]] = 1;
    double mn = POS_INF, mx = NEG_INF;
    for (int i = 0; i < n; ++i) {
      if (in[i]) mn = std::min(mn, sc[i]);
      else mx = std::max(mx, sc[i]);
    }
    if (mn >= mx - tol) {
      std::vector<long long> S;
      for (int i = 0; i < n; ++i)
        if (in[i]) S.push_back(ids[i]);
      std::sort(S.begin(), S.end());
      out.push_back(S);
      if (out.size() >= cap) return;
    }
  } while (std::prev_permutation(pick.begin(), pick.end()));
}

// Is `target` (ascending final set) reachable by a walk in which every SelectK picks a
// top-K within `tol`?  Returns 1 yes, 0 no, -1 search cap exceeded.
int admissible_walk(const Row& R, int l, const std::vector<long long>& S, const std::vector<long long>& target,
                    double tol, long long& budget) {
  if (--budget < 0) return -1;
  if (l >= 2) {
    std::vector<long long> A = eligible_children(R, l, S);
    if ((int)A.size() <= R.K) return admissible_walk(R, l - 1, A, target, tol, budget);
    std::vector<double> sc;
    for (long long i : A) sc.push_back(score_internal(R, l, i));
    std::vector<std::vector<long long>> sets;
    admissible_sets(A, sc, R.K, tol, sets, 64);
    int res = 0;
    for (auto& s2 : sets) {
      int r = admissible_walk(R, l - 1, s2, target, tol, budget);
      if (r == 1) return 1;
      if (r < 0) res = -1;
    }
    return res;
  }
  // l == 1: S holds the level-2 survivors; rank their eligible leaf children
  std::vector<long long> ids;
  std::vector<double> sc;
  long long own = R.causal ? R.t / R.C : -1;
  for (long long p : S)
    for (long long j = R.g * p; j < R.g * p + R.g; ++j)
      if (eligible(R, 1, j) && j != own) {
        ids.push_back(j);
        sc.push_back(score_leaf(R, j));
      }
  std::vector<std::vector<long long>> sets;
  admissible_sets(ids, sc, R.causal ? R.K - 1 : R.K, tol, sets, 4096);
  for (auto& f : sets) {
    if (R.causal) f.push_back(own);
    std::sort(f.begin(), f.end());
    if (f == target) return 1;
  }
  return 0;
}

// ---------------------------------------------------------------------------------------
// BSA flat selection, the single-level baseline PISA is compared with (summary page,
// "Prerequisites": block sparse attention keeps K blocks per query, chosen by the dot
// product of the query with each block's summary, q . kbar_i / sqrt(d), over all
// M = ceil(N / C) blocks; GQA: the group's heads share one selected set, their scores summed).
// Readings: the summaries are the mean-pooled level-1 nodes of the pyramid (eqs 10-15);
// causal eligibility, the forced own block and the tie rule are those of the PISA walk
// (R2, R5, R6).
// ---------------------------------------------------------------------------------------
struct BsaSelection {
  std::vector<long long> final_set;   // ascending
  std::vector<double> score;          // per leaf: head-summed score, -inf if not ranked
  double min_gap = POS_INF;           // K-th / (K+1)-th gap of the ranked blocks
};

BsaSelection select_bsa_row(const Row& R) {
  BsaSelection out;
  if (R.lv.L == 0) return out;
  const long long M1 = R.lv.M[1];
  out.score.assign((size_t)M1, NEG_INF);
  const long long own = R.causal ? R.t / R.C : -1;
  std::vector<long long> ids;
  std::vector<double> sc;
  for (long long j = 0; j < M1; ++j) {
    if (!eligible(R, 1, j) || j == own) continue;
    double u = 0;
    for (int h = 0; h < R.GQ; ++h) u += R.scale * dot_node(R, h, 1, j);
    ids.push_back(j);
    sc.push_back(u);
    out.score[(size_t)j] = u;
  }
  double gap;
  const int keep = R.causal ? R.K - 1 : R.K;  // the own block takes one of the K places
  std::vector<long long> ranked = topk(ids, sc, keep, &gap);
  out.min_gap = gap;
  if (R.causal) ranked.push_back(own);
  std::sort(ranked.begin(), ranked.end());
  out.final_set = ranked;
  return out;
}

Row make_row(const uint16_t* Q_row /* GQ x d for this (b, t, group) */, const uint16_t* Kbg, const uint16_t* Pbg,
             const std::vector<long long>* off, long long n, long long t, int d, int C, int g, int K, int GQ,
             int causal, double scale, int scoring) {
  Row R;
  R.scoring = scoring;
  R.Kbg = Kbg;
  R.Pbg = Pbg;
  R.off = off;
  R.lv = level_sizes(n, C, g);
  R.n = n;
  R.t = t;
  R.d = d;
  R.C = C;
  R.g = g;
  R.K = K;
  R.GQ = GQ;
  R.causal = causal != 0;
  R.scale = scale;
  R.q.resize((size_t)GQ * d);
  for (int i = 0; i < GQ * d; ++i) R.q[i] = bf16_to_f64(Q_row[i]);
  return R;
}

// ---------------------------------------------------------------------------------------
// step 4: attention over the selected blocks (softmax over connected positions only)
// ---------------------------------------------------------------------------------------
// blocks: selected leaf indices (entries < 0 ignored; the union is used, so a repeated
// block counts once).  Writes o[d], returns lse; *wsum = sum of the weights.
double attend(const uint16_t* qh, const uint16_t* Kbg, const uint16_t* Vbg, long long n, long long t, int d, int C,
              bool causal, double scale, const int32_t* blocks, int nb, double* o, double* wsum) {
  std::vector<long long> bl;
  long long M1 = (n + C - 1) / C;
  for (int i = 0; i < nb; ++i)
    if (blocks[i] >= 0 && blocks[i] < M1) bl.push_back(blocks[i]);
  std::sort(bl.begin(), bl.end());
  bl.erase(std::unique(bl.begin(), bl.end()), bl.end());
  std::vector<double> q(d);
  for (int e = 0; e < d; ++e) q[e] = bf16_to_f64(qh[e]);
  std::vector<long long> pos;
  std::vector<double> s;
  for (long long j : bl)
    for (long long c = j * C; c < std::min<long long>(n, j * C + C); ++c) {
      if (causal && c > t) continue;
      double z = 0;
      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);
      pos.push_back(c);
      s.push_back(scale * z);
    }
  for (int e = 0; e < d; ++e) o[e] = 0;
  *wsum = 0;
  if (pos.empty()) return NEG_INF;
  double lse = logsumexp(s);
  for (size_t i = 0; i < pos.size(); ++i) {
    double w = std::exp(s[i] - lse);
    *wsum += w;
    for (int e = 0; e < d; ++e) o[e] += w * bf16_to_f64(Vbg[pos[i] * d + e]);
  }
  return lse;
}

// Backward of attend() for one query head (the gradient of the forward function; the pages
// give no backward): with the forward's visible positions c, s_c = scale q.k_c,
// P_c = exp(s_c - lse), O = sum P_c v_c, D = dO.O, dP_c = dO.v_c, dS_c = P_c (dP_c - D):
// dq += scale sum dS_c k_c, dk_c += scale dS_c q, dv_c += P_c dO.  dO is d values (fp64).
// dK and dV may be null (only dq wanted).
void attend_backward(const uint16_t* qh, const uint16_t* Kbg, const uint16_t* Vbg, long long n, long long t, int d,
                     int C, bool causal, double scale, const int32_t* blocks, int nb, const double* dO, double* dq,
                     double* dK, double* dV) {
  std::vector<long long> bl;
  long long M1 = (n + C - 1) / C;
  for (int i = 0; i < nb; ++i)
    if (blocks[i] >= 0 && blocks[i] < M1) bl.push_back(blocks[i]);
  std::sort(bl.begin(), bl.end());
  bl.erase(std::unique(bl.begin(), bl.end()), bl.end());
  std::vector<double> q(d);
  for (int e = 0; e < d; ++e) q[e] = bf16_to_f64(qh[e]);
  std::vector<long long> pos;
  std::vector<double> s;
  for (long long j : bl)
    for (long long c = j * C; c < std::min<long long>(n, j * C + C); ++c) {
      if (causal && c > t) continue;
      double z = 0;
      for (int e = 0; e < d; ++e) z += q[e] * bf16_to_f64(Kbg[c * d + e]);
      pos.push_back(c);
      s.push_back(scale * z);
    }
  if (pos.empty()) return;
  const double lse = logsumexp(s);
  std::vector<double> P(pos.size()), o(d, 0.0);
  for (size_t i = 0; i < pos.size(); ++i) {
    P[i] = std::exp(s[i] - lse);
    for (int e = 0; e < d; ++e) o[e] += P[i] * bf16_to_f64(Vbg[pos[i] * d + e]);
  }
  double D = 0;
  for (int e = 0; e < d; ++e) D += dO[e] * o[e];
  for (size_t i = 0; i < pos.size(); ++i) {
    const long long c = pos[i];
    double dP = 0;
    for (int e = 0; e < d; ++e) dP += dO[e] * bf16_to_f64(Vbg[c * d + e]);
    const double dS = P[i] * (dP - D);
    for (int e = 0; e < d; ++e) {
      dq[e] += scale * dS * bf16_to_f64(Kbg[c * d + e]);
      if (dK) dK[c * d + e] += scale * dS * q[e];
      if (dV) dV[c * d + e] += P[i] * dO[e];
    }
  }
}

}  // namespace

// =======================================================================================
// C ABI (consumed by the test suite and the benchmark's CPU baseline through ctypes)
// =======================================================================================
extern "C" {

int oracle_num_levels(long long n, int C, int g) { return level_sizes(n, C, g).L; }

// level sizes for n tokens: sizes[l-1] = M_l, l = 1..L; returns L
int oracle_level_sizes(long long n, int C, int g, long long* sizes, int max_levels) {
  Levels lv = level_sizes(n, C, g);
  for (int l = 1; l <= lv.L && l <= max_levels; ++l) sizes[l - 1] = lv.M[l];
  return lv.L;
}

long long oracle_pyramid_nodes(long long n, int C, int g) {
  Levels lv = level_sizes(n, C, g);
  long long s = 0;
  for (int l = 1; l <= lv.L; ++l) s += lv.M[l];
  return s;
}

// K [B][H_kv][N_cap][d] (first N rows used) -> P [B][H_kv][nodes(N_cap)][d]
int oracle_build_pyramid(const uint16_t* K, uint16_t* P, int B, int H_kv, long long N, long long N_cap, int d,
                         int C, int g, int nthreads) {
  if (N < 0 || N > N_cap) return 1;
  std::vector<long long> off = level_offsets(N_cap, C, g);
  long long nodes = oracle_pyramid_nodes(N_cap, C, g);
  run_parallel((long long)B * H_kv, nthreads, [&](long long a, long long b) {
    for (long long bg = a; bg < b; ++bg)
      build_one(K + bg * N_cap * d, P + bg * nodes * d, N, off, d, C, g);
  });
  return 0;
}

// Selection for a list of rows.  rows[3*r] = b, rows[3*r+1] = h_kv, rows[3*r+2] = t.
// Q [B][N][H_q][d]; K [B][H_kv][N][d]; P [B][H_kv][nodes(N)][d].
// Outputs per row (nullable except idx):
//   idx [K] final set ascending, -1 padded
//   s2 [K] level-2 survivors ascending, -1 padded
//   cand [g*K] leaf candidates by slot (-1 = empty), cand_score [g*K] (-inf = empty)
//   min_gap: smallest K-th/(K+1)-th score gap met at any SelectK of the walk
int oracle_select(const uint16_t* Q, const uint16_t* K, const uint16_t* P, int B, long long N, int H_q, int H_kv,
                  int d, int C, int g, int Ksel, int causal, double scale, int nrows, const long long* rows,
                  int32_t* idx, int32_t* s2, int32_t* cand, double* cand_score, double* min_gap, int nthreads,
                  int scoring) {
  if (H_kv <= 0 || H_q % H_kv != 0 || Ksel < 1 || scoring < 0 || scoring > 2) return 1;
  int GQ = H_q / H_kv;
  std::vector<long long> off = level_offsets(N, C, g);
  long long nodes = oracle_pyramid_nodes(N, C, g);
  std::atomic<int> bad(0);
  run_parallel(nrows, nthreads, [&](long long a, long long e) {
    for (long long r = a; r < e; ++r) {
      long long b = rows[3 * r], hk = rows[3 * r + 1], t = rows[3 * r + 2];
      if (b < 0 || b >= B || hk < 0 || hk >= H_kv || t < 0 || t >= N) {
        bad = 1;
        continue;
      }
      const uint16_t* qrow = Q + ((b * N + t) * H_q + hk * GQ) * d;
      Row R = make_row(qrow, K + (b * H_kv + hk) * N * d, P + (b * H_kv + hk) * nodes * d, &off, N, t, d, C, g, Ksel,
                       GQ, causal, scale, scoring);
      Selection S = select_row(R);
      for (int i = 0; i < Ksel; ++i) idx[r * Ksel + i] = i < (int)S.final_set.size() ? (int32_t)S.final_set[i] : -1;
      if (s2)
        for (int i = 0; i < Ksel; ++i) s2[r * Ksel + i] = i < (int)S.S2.size() ? (int32_t)S.S2[i] : -1;
      if (cand)
        for (int i = 0; i < g * Ksel; ++i) cand[r * g * Ksel + i] = (int32_t)S.cand[i];
      if (cand_score)
        for (int i = 0; i < g * Ksel; ++i) cand_score[r * g * Ksel + i] = S.cand_score[i];
      if (min_gap) min_gap[r] = S.min_gap;
    }
  });
  return bad.load();
}

// BSA flat selection for the given rows (b, h_kv, t): idx [nrows][K] (ascending, -1 padded),
// score [nrows][M_1] nullable (head-summed score of every ranked block, -inf for blocks not
// ranked: ineligible, or the forced own block), min_gap [nrows] nullable.
int oracle_select_bsa(const uint16_t* Q, const uint16_t* P, int B, long long N, int H_q, int H_kv, int d, int C, int g,
                      int Ksel, int causal, double scale, int nrows, const long long* rows, int32_t* idx,
                      double* score, double* min_gap, int nthreads) {
  if (H_kv <= 0 || H_q % H_kv != 0 || Ksel < 1) return 1;
  const int GQ = H_q / H_kv;
  std::vector<long long> off = level_offsets(N, C, g);
  const long long nodes = oracle_pyramid_nodes(N, C, g);
  const long long M1 = N > 0 ? (N + C - 1) / C : 0;
  std::atomic<int> bad(0);
  run_parallel(nrows, nthreads, [&](long long a, long long e) {
    for (long long r = a; r < e; ++r) {
      long long b = rows[3 * r], hk = rows[3 * r + 1], t = rows[3 * r + 2];
      if (b < 0 || b >= B || hk < 0 || hk >= H_kv || t < 0 || t >= N) {
        bad = 1;
        continue;
      }
      const uint16_t* qrow = Q + ((b * N + t) * H_q + hk * GQ) * d;
      Row R = make_row(qrow, nullptr, P + (b * H_kv + hk) * nodes * d, &off, N, t, d, C, g, Ksel, GQ, causal, scale, 0);
      BsaSelection S = select_bsa_row(R);
      for (int i = 0; i < Ksel; ++i) idx[r * Ksel + i] = i < (int)S.final_set.size() ? (int32_t)S.final_set[i] : -1;
      if (score)
        for (long long j = 0; j < M1; ++j) score[r * M1 + j] = S.score[(size_t)j];
      if (min_gap) min_gap[r] = S.min_gap;
    }
  });
  return bad.load();
}

// For rows whose selection differs from the oracle's: is `target_idx` [nrows][K]
// (ascending, -1 padded) the outcome of some walk whose every SelectK is a top-K within
// `tol`?  ok[r] = 1 yes, 0 no, -1 undecided (search cap).
int oracle_selection_admissible(const uint16_t* Q, const uint16_t* K, const uint16_t* P, int B, long long N, int H_q,
                                int H_kv, int d, int C, int g, int Ksel, int causal, double scale, int nrows,
                                const long long* rows, const int32_t* target_idx, double tol, int32_t* ok,
                                int nthreads, int scoring) {
  int GQ = H_q / H_kv;
  std::vector<long long> off = level_offsets(N, C, g);
  long long nodes = oracle_pyramid_nodes(N, C, g);
  run_parallel(nrows, nthreads, [&](long long a, long long e) {
    for (long long r = a; r < e; ++r) {
      long long b = rows[3 * r], hk = rows[3 * r + 1], t = rows[3 * r + 2];
      const uint16_t* qrow = Q + ((b * N + t) * H_q + hk * GQ) * d;
      Row R = make_row(qrow, K + (b * H_kv + hk) * N * d, P + (b * H_kv + hk) * nodes * d, &off, N, t, d, C, g, Ksel,
                       GQ, causal, scale, scoring);
      std::vector<long long> target;
      for (int i = 0; i < Ksel; ++i)
        if (target_idx[r * Ksel + i] >= 0) target.push_back(target_idx[r * Ksel + i]);
      long long budget = 200000;
      if (R.lv.L == 0) {
        ok[r] = target.empty() ? 1 : 0;
        continue;
      }
      std::vector<long long> root = {0};
      ok[r] = admissible_walk(R, R.lv.L - 1, root, target, tol, budget);
    }
  });
  return 0;
}

// Attention for rows (b, t) over all H_q heads; head h uses idx of its group h / G_Q.
// rows[2*r] = b, rows[2*r+1] = t.  idx [B][H_kv][N][Ksel].
// Outputs: O [nrows][H_q][d] fp64, LSE [nrows][H_q], wsum [nrows][H_q] (nullable).
int oracle_sparse_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx, int B,
                            long long N, int H_q, int H_kv, int d, int C, int Ksel, int causal, double scale,
                            int nrows, const long long* rows, double* O, double* LSE, double* wsum, int nthreads) {
  if (H_kv <= 0 || H_q % H_kv != 0) return 1;
  int GQ = H_q / H_kv;
  run_parallel(nrows, nthreads, [&](long long a, long long e) {
    for (long long r = a; r < e; ++r) {
      long long b = rows[2 * r], t = rows[2 * r + 1];
      for (int h = 0; h < H_q; ++h) {
        int hk = h / GQ;
        double ws;
        double l = attend(Q + ((b * N + t) * H_q + h) * d, K + (b * H_kv + hk) * N * d, V + (b * H_kv + hk) * N * d,
                          N, t, d, C, causal != 0, scale, idx + ((b * H_kv + hk) * N + t) * Ksel, Ksel,
                          O + (r * H_q + h) * d, &ws);
        LSE[r * H_q + h] = l;
        if (wsum) wsum[r * H_q + h] = ws;
      }
    }
  });
  return 0;
}

// Backward of step 4 for every query (the gradient of the forward; the pages specify none).
// dO bf16 [B][N][H_q][d] (same layout as Q).  Outputs fp64, overwritten: dQ [B][N][H_q][d],
// dK, dV [B][H_kv][N][d].  Work is split by (b, h_kv), so each thread owns its dK/dV rows.
int oracle_sparse_attention_backward(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                     const uint16_t* dO, int B, long long N, int H_q, int H_kv, int d, int C, int Ksel,
                                     int causal, double scale, double* dQ, double* dK, double* dV, int nthreads) {
  if (H_kv <= 0 || H_q % H_kv != 0) return 1;
  const int GQ = H_q / H_kv;
  std::fill(dQ, dQ + (size_t)B * N * H_q * d, 0.0);
  std::fill(dK, dK + (size_t)B * H_kv * N * d, 0.0);
  std::fill(dV, dV + (size_t)B * H_kv * N * d, 0.0);
  run_parallel((long long)B * H_kv, nthreads, [&](long long a, long long e) {
    std::vector<double> go(d);
    for (long long bg = a; bg < e; ++bg) {
      const long long b = bg / H_kv, hk = bg % H_kv;
      for (long long t = 0; t < N; ++t)
        for (int g = 0; g < GQ; ++g) {
          const long long h = hk * GQ + g;
          const size_t row = ((size_t)(b * N + t) * H_q + h) * d;
          for (int x = 0; x < d; ++x) go[x] = bf16_to_f64(dO[row + x]);
          attend_backward(Q + row, K + bg * N * d, V + bg * N * d, N, t, d, C, causal != 0, scale,
                          idx + (bg * N + t) * Ksel, Ksel, go.data(), dQ + row, dK + bg * N * d, dV + bg * N * d);
        }
    }
  });
  return 0;
}

// The same backward restricted to samples, for parity checks at sizes where the full one
// takes too long: dQ of the listed query positions (row = b * N + t, every head) and dK, dV of
// the listed key blocks (block = (b * H_kv + h_kv) * M1 + j, its C rows).  Every value is
// accumulated from the same rows, in the same (t, head) order, as oracle_sparse_attention_backward
// does, so the two functions give equal values.  Outputs fp64, overwritten:
// dQ_rows [nrows][H_q][d], dK_blk and dV_blk [nblocks][C][d] (rows past N stay zero).
int oracle_sparse_attention_backward_sampled(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                             const int32_t* idx, const uint16_t* dO, int B, long long N, int H_q,
                                             int H_kv, int d, int C, int Ksel, int causal, double scale,
                                             const long long* rows, int nrows, const long long* blocks, int nblocks,
                                             double* dQ_rows, double* dK_blk, double* dV_blk, int nthreads) {
  if (H_kv <= 0 || H_q % H_kv != 0) return 1;
  const int GQ = H_q / H_kv;
  const long long M1 = (N + C - 1) / C;
  for (int i = 0; i < nrows; ++i)
    if (rows[i] < 0 || rows[i] >= (long long)B * N) return 2;
  for (int i = 0; i < nblocks; ++i)
    if (blocks[i] < 0 || blocks[i] >= (long long)B * H_kv * M1) return 3;
  std::fill(dQ_rows, dQ_rows + (size_t)nrows * H_q * d, 0.0);
  std::fill(dK_blk, dK_blk + (size_t)nblocks * C * d, 0.0);
  std::fill(dV_blk, dV_blk + (size_t)nblocks * C * d, 0.0);
  // dQ: each listed position, every head
  run_parallel(nrows, nthreads, [&](long long a, long long e) {
    std::vector<double> go(d);
    for (long long i = a; i < e; ++i) {
      const long long b = rows[i] / N, t = rows[i] % N;
      for (int hk = 0; hk < H_kv; ++hk) {
        const long long bg = b * H_kv + hk;
        for (int g = 0; g < GQ; ++g) {
          const long long h = (long long)hk * GQ + g;
          const size_t row = ((size_t)(b * N + t) * H_q + h) * d;
          for (int x = 0; x < d; ++x) go[x] = bf16_to_f64(dO[row + x]);
          attend_backward(Q + row, K + bg * N * d, V + bg * N * d, N, t, d, C, causal != 0, scale,
                          idx + (bg * N + t) * Ksel, Ksel, go.data(), dQ_rows + ((size_t)i * H_q + h) * d, nullptr,
                          nullptr);
        }
      }
    }
  });
  // dK, dV: for each listed block, every (t, head) whose selection holds it, in order
  run_parallel(nblocks, nthreads, [&](long long a, long long e) {
    std::vector<double> go(d), dq(d), sk((size_t)N * d), sv((size_t)N * d);
    for (long long i = a; i < e; ++i) {
      const long long bg = blocks[i] / M1, j = blocks[i] % M1;
      const long long b = bg / H_kv, hk = bg % H_kv;
      std::fill(sk.begin(), sk.end(), 0.0);
      std::fill(sv.begin(), sv.end(), 0.0);
      for (long long t = 0; t < N; ++t) {
        const int32_t* sel = idx + (bg * N + t) * Ksel;
        bool has = false;
        for (int k = 0; k < Ksel; ++k) has = has || sel[k] == j;
        if (!has) continue;
        for (int g = 0; g < GQ; ++g) {
          const long long h = hk * GQ + g;
          const size_t row = ((size_t)(b * N + t) * H_q + h) * d;
          for (int x = 0; x < d; ++x) go[x] = bf16_to_f64(dO[row + x]);
          std::fill(dq.begin(), dq.end(), 0.0);
          attend_backward(Q + row, K + bg * N * d, V + bg * N * d, N, t, d, C, causal != 0, scale, sel, Ksel,
                          go.data(), dq.data(), sk.data(), sv.data());
        }
      }
      for (long long c = j * C; c < std::min<long long>(N, j * C + C); ++c)
        for (int x = 0; x < d; ++x) {
          dK_blk[((size_t)i * C + (c - j * C)) * d + x] = sk[c * d + x];
          dV_blk[((size_t)i * C + (c - j * C)) * d + x] = sv[c * d + x];
        }
    }
  });
  return 0;
}

// One decode step for every sequence (step 3): append k, v at position T = seq_len[b],
// recompute leaf T/C and its ancestors, select for the query at T over T+1 tokens, and
// attend.  Caches: Kc, Vc [B][H_kv][N_cap][d]; Pc [B][H_kv][nodes(N_cap)][d].
// q [B][H_q][d]; k, v [B][H_kv][d].  Outputs o [B][H_q][d] fp64, lse [B][H_q],
// idx_out [B][H_kv][Ksel] (nullable).  seq_len is advanced by one.
int oracle_decode_step(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                       uint16_t* Pc, int32_t* seq_len, long long N_cap, int B, int H_q, int H_kv, int d, int C, int g,
                       int Ksel, double scale, double* o, double* lse, int32_t* idx_out, int nthreads, int scoring) {
  if (H_kv <= 0 || H_q % H_kv != 0) return 1;
  for (int b = 0; b < B; ++b)
    if (seq_len[b] < 0 || seq_len[b] + 1 > N_cap) return 2;
  int GQ = H_q / H_kv;
  std::vector<long long> off = level_offsets(N_cap, C, g);
  long long nodes = oracle_pyramid_nodes(N_cap, C, g);
  run_parallel((long long)B * H_kv, nthreads, [&](long long a, long long e) {
    std::vector<double> acc(d);
    for (long long bg = a; bg < e; ++bg) {
      long long b = bg / H_kv, hk = bg % H_kv;
      long long T = seq_len[b], n = T + 1;
      uint16_t* Kbg = Kc + bg * N_cap * d;
      uint16_t* Vbg = Vc + bg * N_cap * d;
      uint16_t* Pbg = Pc + bg * nodes * d;
      for (int e2 = 0; e2 < d; ++e2) {
        Kbg[T * d + e2] = k[bg * d + e2];
        Vbg[T * d + e2] = v[bg * d + e2];
      }
      // the new token's leaf, from its raw keys
      Levels lv = level_sizes(n, C, g);
      long long leaf = T / C;
      {
        long long c0 = leaf * C, c1 = n;
        std::fill(acc.begin(), acc.end(), 0.0);
        for (long long c = c0; c < c1; ++c)
          for (int e2 = 0; e2 < d; ++e2) acc[e2] += bf16_to_f64(Kbg[c * d + e2]);
        for (int e2 = 0; e2 < d; ++e2) Pbg[(off[1] + leaf) * d + e2] = f64_to_bf16_rne(acc[e2] / (double)(c1 - c0));
      }
      // each ancestor, from its children
      long long node = leaf;
      for (int l = 2; l <= lv.L; ++l) {
        node /= g;
        long long r0 = g * node, r1 = std::min<long long>(lv.M[l - 1], g * node + g);
        std::fill(acc.begin(), acc.end(), 0.0);
        for (long long r = r0; r < r1; ++r)
          for (int e2 = 0; e2 < d; ++e2) acc[e2] += bf16_to_f64(Pbg[(off[l - 1] + r) * d + e2]);
        for (int e2 = 0; e2 < d; ++e2) Pbg[(off[l] + node) * d + e2] = f64_to_bf16_rne(acc[e2] / (double)(r1 - r0));
      }
      // selection for the query at T
      Row R = make_row(q + (b * H_q + hk * GQ) * d, Kbg, Pbg, &off, n, T, d, C, g, Ksel, GQ, 1, scale, scoring);
      Selection S = select_row(R);
      std::vector<int32_t> blocks(Ksel, -1);
      for (int i = 0; i < Ksel && i < (int)S.final_set.size(); ++i) blocks[i] = (int32_t)S.final_set[i];
      if (idx_out)
        for (int i = 0; i < Ksel; ++i) idx_out[bg * Ksel + i] = blocks[i];
      for (int hh = 0; hh < GQ; ++hh) {
        int h = (int)hk * GQ + hh;
        double ws;
        lse[b * H_q + h] = attend(q + (b * H_q + h) * d, Kbg, Vbg, n, T, d, C, true, scale, blocks.data(), Ksel,
                                  o + (b * H_q + h) * d, &ws);
      }
    }
  });
  for (int b = 0; b < B; ++b) seq_len[b] += 1;
  return 0;
}

// Rounding helper exposed for the pins: fp64 -> bf16 bits, round to nearest even.
uint16_t oracle_f64_to_bf16(double x) { return f64_to_bf16_rne(x); }

}  // extern "C"
