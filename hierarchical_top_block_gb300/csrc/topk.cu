// Final top-K over the exact leaf scores (summary page of "Block Sparse Attention with
// Log-Linear Complexity", section "Method step details", step 2: a separate kernel takes
// the final top-K after the exact leaf LSE).  Causal mode keeps the query's own block and
// fills the other K-1 places with the best-scoring eligible candidates (ties to the lower
// block index); the row is written ascending and padded with -1.
//
// One warp per (b, h_kv, t); lane s owns candidate slot s = 2i + c (child c of the i-th
// level-2 survivor), so g*K <= 32 slots fit one warp.
#include "kernels.cuh"

namespace pisa {
namespace {

constexpr int THREADS = 256;


__global__ void __launch_bounds__(THREADS) topk_kernel(const int32_t* __restrict__ S2,
                                                       const float* __restrict__ score, int32_t* __restrict__ idx,
                                                       long long total, int N, int Ksel, int M1, int causal) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (THREADS / 32);
  const int twoK = 2 * Ksel;
  for (long long item = (long long)blockIdx.x * (THREADS / 32) + (threadIdx.x >> 5); item < total; item += nwarps) {
    const int t = (int)(item % N);
    const int own = causal ? t / 64 : -1;
    int leaf = -1;
    float sc = NEG_INF;
    if (lane < twoK) {
      const int node = S2[item * Ksel + (lane >> 1)];
      if (node >= 0) {
        const int j = 2 * node + (lane & 1);
        if (j < M1 && (!causal || (long long)j * 64 <= t) && j != own) {
          leaf = j;
          sc = score[item * twoK + lane];
        }
      }
    }
    const unsigned valid = __ballot_sync(0xffffffffu, leaf >= 0);
    // rank among the valid candidates: (score desc, block index asc)
    int rank = 0;
    for (int j = 0; j < 32; ++j) {
      if (!((valid >> j) & 1u)) continue;
      const float sj = __shfl_sync(0xffffffffu, sc, j);
      const int lj = __shfl_sync(0xffffffffu, leaf, j);
      rank += (leaf >= 0 && (sj > sc || (sj == sc && lj < leaf))) ? 1 : 0;
    }
    const int keep_n = causal ? Ksel - 1 : Ksel;
    const bool keep = leaf >= 0 && rank < keep_n;
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    // output position = number of kept blocks with a smaller index (+1 if the own block is smaller)
    int pos = 0;
    for (int j = 0; j < 32; ++j) {
      if (!((km >> j) & 1u)) continue;
      const int lj = __shfl_sync(0xffffffffu, leaf, j);
      pos += (keep && lj < leaf) ? 1 : 0;
    }
    int32_t* out = idx + item * Ksel;
    const int nkept = __popc(km);
    if (keep) out[pos + ((causal && own < leaf) ? 1 : 0)] = leaf;
    if (causal) {
      // own block position: kept blocks below it
      int below = 0;
      for (int j = 0; j < 32; ++j) {
        if (!((km >> j) & 1u)) continue;
        const int lj = __shfl_sync(0xffffffffu, leaf, j);
        below += lj < own ? 1 : 0;
      }
      if (lane == 0) out[below] = own;
    }
    const int filled = nkept + (causal ? 1 : 0);
    if (lane >= filled && lane < Ksel) out[lane] = -1;
  }
}

}  // namespace

cudaError_t launch_topk(const int32_t* S2, const float* leaf_score, int32_t* idx, const Problem& p,
                        const Geometry& geo, cudaStream_t s) {
  const long long total = (long long)p.B * p.H_kv * p.N;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + (THREADS / 32) - 1) / (THREADS / 32);
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  topk_kernel<<<(int)blocks, THREADS, 0, s>>>(S2, leaf_score, idx, total, p.N, p.K, geo.M[1], p.causal);
  return cudaGetLastError();
}

}  // namespace pisa
