// Stage 1 of the two-stage selection (summary page of "Block Sparse Attention with
// Log-Linear Complexity", section "Method step details", step 2; section "Core method",
// eq. 21; GQA head sum eq. 22): for every query, start at the root, and at each level
// expand the survivors to their eligible children; when more than K candidates remain,
// score each one with the LSE of its children's logits q.k/sqrt(d), summed over the G_Q
// query heads of the group, and keep the K best (ties to the lower index).  The result is
// the set of level-2 survivors S2 (<= K nodes); their eligible children are the leaf
// candidates that Stage 2 scores exactly.
//
// One warp owns one (b, h_kv, t) at a time.  The group's G_Q query rows (padded to 16)
// stay in registers as mma.sync A fragments for the whole walk; each scored level gathers
// the <= 2K x 2 child summaries straight from L2/L1 into registers with 16-byte loads and
// multiplies them with m16n8k16 (16 heads x 8 children per MMA).  The d index is permuted
// identically in A and B so that each lane loads 8 contiguous values per child row.
// Candidate lists, LSE, head sums and the rank-based SelectK stay in registers and warp
// shuffles: no query-key score matrix is materialised.
#include "kernels.cuh"

namespace pisa {
namespace {

constexpr int THREADS = 256;


// log2(2^a + 2^b), with -inf inputs allowed (not both)
__device__ __forceinline__ float lse2_pair(float a, float b) {
  const float m = fmaxf(a, b);
  const float n = fminf(a, b);
  return m + fast_log2(1.0f + fast_exp2(n - m));
}

template <int D>
__global__ void __launch_bounds__(THREADS, D == 128 ? 2 : 3) stage1_kernel(const uint16_t* __restrict__ Q,
                                                         const uint16_t* __restrict__ P, int32_t* __restrict__ S2,
                                                         int B, int N, int H_q, int H_kv, int GQ, int Ksel, int causal,
                                                         float scale_log2, Geometry geo) {
  constexpr int NCH = D / 32;  // 32-wide d chunks; each feeds two k16 steps
  constexpr int NB = 2;        // n-tiles (8 children each) whose loads are in flight together
  __shared__ int lists[THREADS / 32][32];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, q = lane & 3;
  const unsigned lt_mask = (1u << lane) - 1u;
  int* lst = lists[warp];
  const long long total = (long long)B * H_kv * N;
  const long long nwarps = (long long)gridDim.x * (THREADS / 32);

  for (long long item = (long long)blockIdx.x * (THREADS / 32) + warp; item < total; item += nwarps) {
    const int bh = (int)(item / N);
    const int t = (int)(item - (long long)bh * N);
    const int b = bh / H_kv, hk = bh - b * H_kv;

    // query fragments: rows r and r+8 of the group (zero beyond G_Q), 8 contiguous d values
    // per chunk: chunk j of lane q covers d in [32j + 8q, 32j + 8q + 8)
    uint4 qa[NCH], qb[NCH];
    const uint16_t* qrow = Q + (((size_t)b * N + t) * H_q + (size_t)hk * GQ) * D;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      qa[j] = r < GQ ? ldg16(qrow + (size_t)r * D + 32 * j + 8 * q) : make_uint4(0, 0, 0, 0);
      qb[j] = r + 8 < GQ ? ldg16(qrow + (size_t)(r + 8) * D + 32 * j + 8 * q) : make_uint4(0, 0, 0, 0);
    }
    const uint16_t* Pb = P + (size_t)bh * geo.nodes * D;

    int surv = lane == 0 ? 0 : -1;  // survivors of level l+1 (lane i holds the i-th, ascending)
    int ns = 1;
    for (int l = geo.L - 1; l >= 2; --l) {
      // eligible children of the survivors, in ascending order
      const long long span = 64LL << (l - 1);  // keys under one level-l node
      const int c0 = 2 * surv, c1 = 2 * surv + 1;
      const bool e0 = lane < ns && c0 < geo.M[l] && (!causal || (long long)c0 * span <= t);
      const bool e1 = lane < ns && c1 < geo.M[l] && (!causal || (long long)c1 * span <= t);
      const unsigned b0 = __ballot_sync(0xffffffffu, e0), b1 = __ballot_sync(0xffffffffu, e1);
      const int pos = __popc(b0 & lt_mask) + __popc(b1 & lt_mask);
      const int nc = __popc(b0) + __popc(b1);
      if (e0) lst[pos] = c0;
      if (e1) lst[pos + (e0 ? 1 : 0)] = c1;
      __syncwarp();
      const int cand = lane < nc ? lst[lane] : -1;
      __syncwarp();
      if (nc <= Ksel) {
        surv = cand;
        ns = nc;
        continue;
      }

      // score the nc candidates with their level-(l-1) children: slot 2i+c = child c of cand i
      const long long cspan = 64LL << (l - 2);
      const long long lvl_off = geo.off[l - 1];
      const int Mc = geo.M[l - 1];
      // start every child row of this level on its way to L1 before the batched loads, so
      // the level costs one memory round trip instead of one per batch
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int ci = 4 * nt + (r >> 1);
        const int cnode = __shfl_sync(0xffffffffu, cand, ci);
        const int child = 2 * cnode + (r & 1);
        const bool valid = ci < nc && child < Mc && (!causal || (long long)child * cspan <= t);
        if (valid && 64 * (q >> 1) < D && (q & 1) == 0) prefetch_l1(Pb + (size_t)(lvl_off + child) * D + 64 * (q >> 1));
      }
      float my = NEG_INF;  // score of candidate `lane`
#pragma unroll
      for (int half = 0; half < 8 / NB; ++half) {
        uint4 kv[NB][NCH];
        bool valid[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) {
          const int nt = half * NB + k;
          const int ci = 4 * nt + (r >> 1);
          const int cnode = __shfl_sync(0xffffffffu, cand, ci);
          const int child = 2 * cnode + (r & 1);
          valid[k] = ci < nc && child < Mc && (!causal || (long long)child * cspan <= t);
          const uint16_t* prow = Pb + (size_t)(lvl_off + (valid[k] ? child : 0)) * D;
#pragma unroll
          for (int j = 0; j < NCH; ++j) kv[k][j] = valid[k] ? ldg16(prow + 32 * j + 8 * q) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < NB; ++k) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            mma_bf16_16816(acc, qa[j].x, qb[j].x, qa[j].y, qb[j].y, kv[k][j].x, kv[k][j].y);
            mma_bf16_16816(acc, qa[j].z, qb[j].z, qa[j].w, qb[j].w, kv[k][j].z, kv[k][j].w);
          }
          // acc: (row r | r+8) x (col 2q | 2q+1) = heads x children 0/1 of candidate 4nt+q
          const unsigned vm = __ballot_sync(0xffffffffu, valid[k]);
          const bool v0 = (vm >> (8 * q)) & 1u, v1 = (vm >> (8 * q + 4)) & 1u;
          float part = 0.f;
          if (v0) {
            const float x0 = acc[0] * scale_log2, x1 = v1 ? acc[1] * scale_log2 : NEG_INF;
            const float y0 = acc[2] * scale_log2, y1 = v1 ? acc[3] * scale_log2 : NEG_INF;
            if (r < GQ) part += lse2_pair(x0, x1);
            if (r + 8 < GQ) part += lse2_pair(y0, y1);
          }
          part += __shfl_xor_sync(0xffffffffu, part, 4);
          part += __shfl_xor_sync(0xffffffffu, part, 8);
          part += __shfl_xor_sync(0xffffffffu, part, 16);
          // candidate 4nt+q's score to lane 4nt+q (lanes hold one candidate each)
          const float val = __shfl_sync(0xffffffffu, v0 ? part : NEG_INF, lane & 3);
          if ((lane >> 2) == half * NB + k) my = val;
        }
      }
      if (lane >= nc) my = NEG_INF;
      // SelectK: rank by (score desc, index asc)
      int rank = 0;
      for (int j = 0; j < nc; ++j) {
        const float uj = __shfl_sync(0xffffffffu, my, j);
        rank += (uj > my || (uj == my && j < lane)) ? 1 : 0;
      }
      const bool keep = lane < nc && rank < Ksel;
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) lst[__popc(km & lt_mask)] = cand;
      __syncwarp();
      ns = __popc(km);
      surv = lane < ns ? lst[lane] : -1;
      __syncwarp();
    }
    if (lane < Ksel) S2[item * Ksel + lane] = lane < ns ? surv : -1;
  }
}

}  // namespace

cudaError_t launch_stage1(const uint16_t* Q, const uint16_t* P, int32_t* S2, const Problem& p, const Geometry& geo,
                          int num_sms, uint32_t* err, cudaStream_t s) {
  (void)err;
  const long long total = (long long)p.B * p.H_kv * p.N;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + (THREADS / 32) - 1) / (THREADS / 32);
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  const float sl2 = p.scale * LOG2E;
  if (p.d == 128)
    stage1_kernel<128><<<(int)blocks, THREADS, 0, s>>>(Q, P, S2, p.B, p.N, p.H_q, p.H_kv, p.GQ, p.K, p.causal, sl2, geo);
  else
    stage1_kernel<64><<<(int)blocks, THREADS, 0, s>>>(Q, P, S2, p.B, p.N, p.H_q, p.H_kv, p.GQ, p.K, p.causal, sl2, geo);
  return cudaGetLastError();
}

}  // namespace pisa
