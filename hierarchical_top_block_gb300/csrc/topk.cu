// Final top-K over the exact leaf scores (summary page of "Block Sparse Attention with
// Log-Linear Complexity", section "Method step details", step 2: a separate kernel takes
// the final top-K after the exact leaf LSE).  Causal mode keeps the query's own block and
// fills the other K-1 places with the best-scoring eligible candidates (ties to the lower
// block index); the row is written ascending and padded with -1.
//
// One warp per (b, h_kv, t); lane s owns candidate slot s = 2i + c (child c of the i-th
// level-2 survivor), so g*K <= 32 slots fit one warp; for K up to 32 each lane owns two.
#include "kernels.cuh"
#include "pdl.cuh"

namespace pisa {
namespace {

constexpr int THREADS = 256;


__global__ void __launch_bounds__(THREADS) topk_kernel(const int32_t* __restrict__ S2,
                                                       float* __restrict__ score, int32_t* __restrict__ idx,
                                                       int BH, int N, int t_lo, int nq, int Ksel, int M1, int causal) {
  pdl_trigger();
  pdl_wait();  // the leaf scores come from Stage 2
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const long long gw = (long long)blockIdx.x * (THREADS / 32) + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * (THREADS / 32);
  const int st_bh = (int)(nwarps / nq), st_t = (int)(nwarps % nq);  // grid stride as (bh, t) steps
  const int twoK = 2 * Ksel;
  const int keep_n = causal ? Ksel - 1 : Ksel;
  // lane s reads slot s of an item: its level-2 survivor and its leaf score (both in bounds;
  // the score of an empty slot is never used), and the next item's pair is read while the
  // current item is ranked
  auto fetch = [&](int fbh, int ft, int& node, float& sc) {
    node = -1;
    sc = NEG_INF;
    if (fbh < BH && lane < twoK) {
      const long long fitem = (long long)fbh * N + ft;
      node = S2[fitem * Ksel + (lane >> 1)];
      sc = score[fitem * twoK + lane];
    }
  };
  int bh = (int)(gw / nq), t = t_lo + (int)(gw % nq);
  int node_n;
  float sc_n;
  fetch(bh, t, node_n, sc_n);
  while (bh < BH) {
    const int node = node_n, cbh = bh, ct = t;
    const float sc_raw = sc_n;
    t += st_t;
    bh += st_bh;
    if (t >= t_lo + nq) {
      t -= nq;
      ++bh;
    }
    fetch(bh, t, node_n, sc_n);
    const long long item = (long long)cbh * N + ct;
    const int own = causal ? ct / 64 : -1;
    // slots of absent level-2 survivors hold no leaf: their score reads -inf
    if (lane < twoK && node < 0) score[item * twoK + lane] = NEG_INF;
    int leaf = -1;
    float sc = NEG_INF;
    if (node >= 0) {
      const int j = 2 * node + (lane & 1);
      if (j < M1 && (!causal || j <= ct / 64) && j != own) {
        leaf = j;
        sc = sc_raw;
      }
    }
    // The survivors, hence the slots, are in ascending block order, so ranking by (score
    // desc, slot asc) is ranking by (score desc, block index asc): bitonic sort over the lanes
    float sv = sc;
    int si = lane;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, sv, j);
        const int oi = __shfl_xor_sync(0xffffffffu, si, j);
        const bool other_better = ov > sv || (ov == sv && oi < si);
        const bool lower = (lane & j) == 0, desc = (lane & k) == 0;
        if ((lower == desc) == other_better) {
          sv = ov;
          si = oi;
        }
      }
    }
    const unsigned valid = __ballot_sync(0xffffffffu, leaf >= 0);
    const unsigned km = __reduce_or_sync(0xffffffffu, lane < keep_n ? (1u << si) : 0u) & valid;
    const bool keep = (km >> lane) & 1u;
    // output position = kept blocks with a smaller index (+1 if the own block is smaller)
    int32_t* out = idx + item * Ksel;
    if (keep) out[__popc(km & lt_mask) + ((causal && own < leaf) ? 1 : 0)] = leaf;
    const unsigned below = __ballot_sync(0xffffffffu, leaf >= 0 && leaf < own);  // eligible blocks under own
    if (causal && lane == 0) out[__popc(km & below)] = own;
    const int filled = __popc(km) + (causal ? 1 : 0);
    if (lane >= filled && lane < Ksel) out[lane] = -1;
  }
}

// The same for K in 17..32: lane l owns slots l and l + 32 (g*K <= 64), ranked with the
// warp's 64-entry bitonic ranking.
__global__ void __launch_bounds__(THREADS) topk64_kernel(const int32_t* __restrict__ S2,
                                                         float* __restrict__ score, int32_t* __restrict__ idx,
                                                         int BH, int N, int t_lo, int nq, int Ksel, int M1, int causal) {
  pdl_trigger();
  pdl_wait();  // the leaf scores come from Stage 2
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const long long gw = (long long)blockIdx.x * (THREADS / 32) + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * (THREADS / 32);
  const int twoK = 2 * Ksel;
  const int keep_n = causal ? Ksel - 1 : Ksel;
  for (long long it = gw; it < (long long)BH * nq; it += nwarps) {
    const int bh = (int)(it / nq), t = t_lo + (int)(it - (long long)bh * nq);
    const long long item = (long long)bh * N + t;
    const int own = causal ? t / 64 : -1;
    float v[2];
    int key[2], id[2], leaf[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int slot = 32 * e + lane;
      int node = -1;
      float sc = NEG_INF;
      if (slot < twoK) {
        node = S2[item * Ksel + (slot >> 1)];
        sc = score[item * twoK + slot];
        // slots of absent level-2 survivors hold no leaf: their score reads -inf
        if (node < 0) score[item * twoK + slot] = NEG_INF;
      }
      leaf[e] = -1;
      v[e] = NEG_INF;
      if (node >= 0) {
        const int j = 2 * node + (slot & 1);
        if (j < M1 && (!causal || j <= own) && j != own) {
          leaf[e] = j;
          v[e] = sc;
        }
      }
      key[e] = slot;  // slots are in ascending block order: ties go to the lower block
      id[e] = slot;
    }
    const unsigned valid0 = __ballot_sync(0xffffffffu, leaf[0] >= 0), valid1 = __ballot_sync(0xffffffffu, leaf[1] >= 0);
    warp_top32_of64(v, key, id);
    // kept slots: the first keep_n ranked entries that hold a leaf
    const bool take = lane < keep_n;
    const unsigned k0 = __reduce_or_sync(0xffffffffu, take && id[0] < 32 ? (1u << id[0]) : 0u) & valid0;
    const unsigned k1 = __reduce_or_sync(0xffffffffu, take && id[0] >= 32 ? (1u << (id[0] - 32)) : 0u) & valid1;
    int32_t* out = idx + item * Ksel;
    const int n0 = __popc(k0);
    const unsigned b0 = __ballot_sync(0xffffffffu, leaf[0] >= 0 && leaf[0] < own);
    const unsigned b1 = __ballot_sync(0xffffffffu, leaf[1] >= 0 && leaf[1] < own);
    // output position = kept blocks with a smaller index (+1 if the own block is smaller)
    if ((k0 >> lane) & 1u) out[__popc(k0 & lt_mask) + ((causal && own < leaf[0]) ? 1 : 0)] = leaf[0];
    if ((k1 >> lane) & 1u) out[n0 + __popc(k1 & lt_mask) + ((causal && own < leaf[1]) ? 1 : 0)] = leaf[1];
    if (causal && lane == 0) out[__popc(k0 & b0) + __popc(k1 & b1)] = own;
    const int filled = n0 + __popc(k1) + (causal ? 1 : 0);
    if (lane >= filled && lane < Ksel) out[lane] = -1;
  }
}

}  // namespace

cudaError_t launch_topk(const int32_t* S2, float* leaf_score, int32_t* idx, const Problem& p,
                        const Geometry& geo, int num_sms, cudaStream_t s) {
  const int nq = p.t_hi - p.t_lo;
  const long long total = (long long)p.B * p.H_kv * nq;
  if (total <= 0) return cudaSuccess;
  // one wave of resident CTAs, each warp walking items with a grid stride (so that the next
  // item's rows are in flight while the current one is ranked)
  long long blocks = (total + (THREADS / 32) - 1) / (THREADS / 32);
  if (blocks > (long long)num_sms * 8) blocks = (long long)num_sms * 8;
  // a programmatic dependent of Stage 2
  return launch_pdl(p.K > 16 ? topk64_kernel : topk_kernel, dim3((unsigned)blocks), dim3(THREADS), 0, s, S2, leaf_score,
                    idx, p.B * p.H_kv, p.N, p.t_lo, nq, p.K, geo.M[1], p.causal);
}

}  // namespace pisa
