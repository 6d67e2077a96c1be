// Stage 1 of the two-stage selection (summary page of "Block Sparse Attention with
// Log-Linear Complexity", section "Method step details", step 2; section "Core method",
// eq. 21; GQA head sum eq. 22): for every query, start at the root, and at each level
// expand the survivors to their eligible children; when more than K candidates remain,
// score each one with the LSE of its children's logits q.k/sqrt(d), summed over the G_Q
// query heads of the group, and keep the K best (ties to the lower index).  The result is
// the set of level-2 survivors S2 (<= K nodes); their eligible children are the leaf
// candidates that Stage 2 scores exactly.
//
// One warp owns one (b, h_kv, t) at a time, claimed from a counter.  The group's G_Q query rows (padded to 16)
// stay in registers as mma.sync B fragments for the whole walk; each scored level gathers
// the <= 2K x 2 child summaries straight from L2/L1 into registers with 16-byte loads and
// multiplies them with m16n8k16 (the two children of 8 candidates x 8 heads per MMA, so a
// lane holds both children of one candidate and the pair LSE needs no exchange).  The d
// index is permuted identically in A and B so that each lane loads 8 contiguous values per
// row.  Candidate lists, LSE, head sums and a bitonic SelectK stay in registers and warp
// shuffles: no query-key score matrix is materialised.  Each survivor is also counted into
// the clustering histogram, and the count returned is stored as its place in its list.
#include "kernels.cuh"
#include "pdl.cuh"

namespace pisa {
namespace {

constexpr int THREADS = 128;
// resident CTAs per SM the register budget is sized for (the walk is latency-bound: more
// warps in flight hide the per-level L2 round trip and the MMA/shuffle dependency chains)
constexpr int MIN_BLOCKS_128 = 5, MIN_BLOCKS_64 = 6;


// SC: the block score (0 LSE, 1 log m + mean, 2 log m + mean + variance / 2), fixed at compile
// time so that the pair score carries no branch.  W: candidates per lane, 1 for K <= 16 (2K <= 32
// candidates per level), 2 for K in 17..32 (lane l also holds candidate l + 32).
template <int D, int SC, int W>
__global__ void __launch_bounds__(THREADS, D == 128 ? MIN_BLOCKS_128 : MIN_BLOCKS_64) stage1_kernel(const uint16_t* __restrict__ Q,
                                                         const uint16_t* __restrict__ P, int32_t* __restrict__ S2,
                                                         ClusterBuffers cb,
                                                         int B, int N, int H_q, int H_kv, int GQ, int Ksel, int causal,
                                                         float scale_log2, int t_lo, int nq, Geometry geo) {
  pdl_trigger();  // the clustering's first kernel may launch (it waits for this one to end)
  constexpr int scoring = SC;
  constexpr int NCH = D / 32;  // 32-wide d chunks; each feeds two k16 steps
  constexpr int KH = NCH / 2;      // chunks loaded together
  __shared__ int lists[THREADS / 32][32 * W];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, q = lane & 3;
  const unsigned lt_mask = (1u << lane) - 1u;
  int* lst = lists[warp];
  const int BH = B * H_kv;
  // Items i = bh * nq + (t - t_lo) are claimed one at a time from a counter, so that CTAs
  // that start late (their SM still held by a kernel of another stream) take fewer of them
  // and the kernel ends on a tail of one walk.  The claim of the item after next is issued
  // as a walk starts and read when it ends, so its round trip overlaps the walk.  The count
  // fits 32 bits: the clustering lists already bound B * H_kv * N * K below 2^31.
  const int total = BH * nq;
  auto claim = [&]() {
    int v = 0;
    if (lane == 0) v = atomicAdd(cb.sched, 1);
    return __shfl_sync(0xffffffffu, v, 0);
  };
  int cur = claim();
  int nxt = claim();

  bool pend = false;  // this lane holds the list place of a survivor not yet stored
  int pend_rank = 0;
  int pend_item = 0;  // bh * N + t, below B * H_kv * N < 2^31
  while (cur < total) {
    int fut = 0;
    if (lane == 0) fut = atomicAdd(cb.sched, 1);
    const int bh = cur / nq, t = t_lo + (cur - bh * nq);
    const long long item = (long long)bh * N + t;
    const int b = bh / H_kv, hk = bh - b * H_kv;
    if (nxt < total) {  // move the next item's Q rows towards L2 while this walk runs (128 bytes per lane)
      const int nbh = nxt / nq, nt = t_lo + (nxt - nbh * nq);
      const int nb = nbh / H_kv, nhk = nbh - nb * H_kv;
      const uint16_t* nq = Q + (((size_t)nb * N + nt) * H_q + (size_t)nhk * GQ) * D;
      if (lane * 64 < GQ * D) prefetch_l2(nq + (size_t)lane * 64);
    }

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
    const bool two_tiles = GQ > 8;  // heads 8..15 exist

    int surv = lane == 0 ? 0 : -1;  // survivors of level l+1 (lane i holds the i-th, ascending)
    int ns = 1;
    for (int l = geo.L - 1; l >= 2; --l) {
      // eligible children of the survivors, in ascending order
      // a level-l node covers 2^(l+5) keys and starts at key c * 2^(l+5): visible iff c <= t >> (l+5)
      const int tl = t >> (l + 5);
      const int c0 = 2 * surv, c1 = 2 * surv + 1;
      const bool e0 = lane < ns && c0 < geo.M[l] && (!causal || c0 <= tl);
      const bool e1 = lane < ns && c1 < geo.M[l] && (!causal || c1 <= tl);
      const unsigned b0 = __ballot_sync(0xffffffffu, e0), b1 = __ballot_sync(0xffffffffu, e1);
      const int pos = __popc(b0 & lt_mask) + __popc(b1 & lt_mask);
      const int nc = __popc(b0) + __popc(b1);
      if (e0) lst[pos] = c0;
      if (e1) lst[pos + (e0 ? 1 : 0)] = c1;
      __syncwarp();
      const int cand = lane < nc ? lst[lane] : -1;
      int cand_hi = -1;  // candidates 32..63 (W == 2)
      if constexpr (W == 2) cand_hi = lane + 32 < nc ? lst[lane + 32] : -1;
      __syncwarp();
      if (nc <= Ksel) {  // Ksel <= 32: the candidates fit one per lane
        surv = cand;
        ns = nc;
        continue;
      }

      // score the nc candidates with their level-(l-1) children.  MMA rows are children
      // (row r: child 0 of candidate 8m + r, row r + 8: its child 1), columns are heads, so
      // lane (r, q) ends with both children of one candidate for heads 2q, 2q+1 (n-tile 0)
      // and 8+2q, 9+2q (n-tile 1).
      const int tc = t >> (l + 4);  // the same for level-(l-1) nodes
      const uint16_t* Pl = Pb + (size_t)geo.off[l - 1] * D;
      const int Mc = geo.M[l - 1];
      float my = NEG_INF;     // score of candidate `lane`
      float my_hi = NEG_INF;  // score of candidate `lane + 32` (W == 2)
      const int nmt = (nc + 7) >> 3;
      for (int mt = 0; mt < nmt; ++mt) {
        const int ci = 8 * mt + r;
        int cnode;
        if constexpr (W == 2) cnode = __shfl_sync(0xffffffffu, mt >= 4 ? cand_hi : cand, ci & 31);
        else cnode = __shfl_sync(0xffffffffu, cand, ci);
        const bool vc = ci < nc;
        const int ch = 2 * cnode;
        const bool v1 = vc && ch + 1 < Mc && (!causal || ch + 1 <= tc);
        // rows are read unconditionally (an absent child 1 or candidate only feeds scores that
        // are masked below); row ch + 1 <= Mc stays inside the pyramid: level l-1 is followed
        // by level l
        const uint16_t* row = Pl + (size_t)(vc ? ch : 0) * D;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jh = 0; jh < NCH; jh += KH) {  // KH chunks of both child rows per load group
          uint4 k0[KH], k1[KH];
#pragma unroll
          for (int u = 0; u < KH; ++u) {
            k0[u] = ldg16(row + 32 * (jh + u) + 8 * q);
            k1[u] = ldg16(row + D + 32 * (jh + u) + 8 * q);
          }
#pragma unroll
          for (int u = 0; u < KH; ++u) {
            mma_bf16_16816(a0, k0[u].x, k1[u].x, k0[u].y, k1[u].y, qa[jh + u].x, qa[jh + u].y);
            mma_bf16_16816(a0, k0[u].z, k1[u].z, k0[u].w, k1[u].w, qa[jh + u].z, qa[jh + u].w);
          }
          if (two_tiles) {
#pragma unroll
            for (int u = 0; u < KH; ++u) {
              mma_bf16_16816(a1, k0[u].x, k1[u].x, k0[u].y, k1[u].y, qb[jh + u].x, qb[jh + u].y);
              mma_bf16_16816(a1, k0[u].z, k1[u].z, k0[u].w, k1[u].w, qb[jh + u].z, qb[jh + u].w);
            }
          }
        }
        // per head: the pair score (LSE or one of its truncations), log2 units; child 1 may be absent
        float part = 0.f;
        if (scoring == 0 && GQ >= 16 && v1) {
          // the four pair LSEs two heads per instruction (packed fp32, same roundings as the
          // scalar form, summed in the same order)
          const unsigned long long s2 = pack_f32x2(scale_log2, scale_log2);
          const unsigned long long one2 = pack_f32x2(1.f, 1.f);
          float r[4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float* c = hh == 0 ? a0 : a1;
            const float m0 = fmaxf(c[0], c[2]), m1 = fmaxf(c[1], c[3]);
            const float n0 = fminf(c[0], c[2]), n1 = fminf(c[1], c[3]);
            float d0, d1;
            unpack_f32x2(mul_f32x2(add_f32x2(pack_f32x2(n0, n1), pack_f32x2(-m0, -m1)), s2), d0, d1);
            float e0, e1;
            unpack_f32x2(add_f32x2(one2, pack_f32x2(fast_exp2(d0), fast_exp2(d1))), e0, e1);
            unpack_f32x2(fma_f32x2(pack_f32x2(m0, m1), s2, pack_f32x2(fast_log2(e0), fast_log2(e1))), r[2 * hh],
                         r[2 * hh + 1]);
          }
          part = ((r[0] + r[1]) + r[2]) + r[3];
        } else {
          if (2 * q < GQ) part += pair_score(a0[0], a0[2], v1, scale_log2, scoring);
          if (2 * q + 1 < GQ) part += pair_score(a0[1], a0[3], v1, scale_log2, scoring);
          if (8 + 2 * q < GQ) part += pair_score(a1[0], a1[2], v1, scale_log2, scoring);
          if (9 + 2 * q < GQ) part += pair_score(a1[1], a1[3], v1, scale_log2, scoring);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        // candidate 8mt + r's score (held by lanes 4r..4r+3) to lane 8mt + r
        const float val = __shfl_sync(0xffffffffu, part, 4 * (lane & 7));
        if ((lane >> 3) == mt) my = val;
        if constexpr (W == 2)
          if ((lane >> 3) == mt - 4) my_hi = val;
      }
      if (lane >= nc) my = NEG_INF;
      if constexpr (W == 2) {
        if (lane + 32 >= nc) my_hi = NEG_INF;
        // SelectK over up to 64 candidates (ranked by score desc, list position asc), then the
        // kept ones compacted in list (ascending node) order
        float sv2[2] = {my, my_hi};
        int key2[2] = {lane, lane + 32}, id2[2] = {lane, lane + 32};
        warp_top32_of64(sv2, key2, id2);
        const bool take = lane < Ksel;
        const unsigned k0 = __reduce_or_sync(0xffffffffu, take && id2[0] < 32 ? (1u << id2[0]) : 0u);
        const unsigned k1 = __reduce_or_sync(0xffffffffu, take && id2[0] >= 32 ? (1u << (id2[0] - 32)) : 0u);
        if ((k0 >> lane) & 1u) lst[__popc(k0 & lt_mask)] = cand;
        if ((k1 >> lane) & 1u) lst[__popc(k0) + __popc(k1 & lt_mask)] = cand_hi;
        __syncwarp();
        ns = __popc(k0) + __popc(k1);
        surv = lane < ns ? lst[lane] : -1;
        __syncwarp();
        continue;
      }
      // SelectK: bitonic sort of the 32 (score desc, index asc) pairs; the first Ksel lanes
      // then hold the kept candidates.  For Ksel = 16 the network stops after the first merge
      // step of the last stage: the two sorted halves then face each other, so each of lanes
      // 0..15 holds the better of a pair whose partners rank i and 15-i, i.e. the best 16 as
      // a set (their order is not needed)
      float sv = my;
      int si = lane;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          if (k == 32 && j < 16 && Ksel == 16) break;
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
      const unsigned km = __reduce_or_sync(0xffffffffu, lane < Ksel ? (1u << si) : 0u);
      const bool keep = (km >> lane) & 1u;
      if (keep) lst[__popc(km & lt_mask)] = cand;
      __syncwarp();
      ns = __popc(km);
      surv = lane < ns ? lst[lane] : -1;
      __syncwarp();
    }
    if (lane < Ksel) S2[item * Ksel + lane] = lane < ns ? surv : -1;
    // the clustering histogram: one entry per survivor in the list of key (b, h_kv, window,
    // node); the count returned is the entry's place in that list, stored one item later so
    // that the atomic's round trip overlaps the next walk
    if (pend) cb.rank[(long long)pend_item * (2 * Ksel) + lane] = pend_rank;
    pend = lane < ns;
    if (pend) {
      pend_rank = atomicAdd(&cb.counts[((long long)bh * cb.nwin + t / cb.win) * cb.M2 + surv], 1);
      pend_item = (int)item;
    }
    cur = nxt;
    nxt = __shfl_sync(0xffffffffu, fut, 0);
  }
  if (pend) cb.rank[(long long)pend_item * (2 * Ksel) + lane] = pend_rank;
}

}  // namespace

cudaError_t launch_stage1(const uint16_t* Q, const uint16_t* P, int32_t* S2, const ClusterBuffers& cb, const Problem& p,
                          const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s) {
  (void)err;
  const int nq = p.t_hi - p.t_lo;
  const long long total = (long long)p.B * p.H_kv * nq;
  if (total <= 0) return cudaSuccess;
  // persistent grid: exactly the CTAs that are resident at once, each warp claiming items from
  // the counter, so no second partial wave
  auto go = [&](auto kern) -> cudaError_t {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    long long blocks = (total + (THREADS / 32) - 1) / (THREADS / 32);
    const long long cap = (long long)num_sms * per_sm;
    if (blocks > cap) blocks = cap;
    kern<<<(int)blocks, THREADS, 0, s>>>(Q, P, S2, cb, p.B, p.N, p.H_q, p.H_kv, p.GQ, p.K, p.causal, p.scale * LOG2E, p.t_lo,
                                         nq, geo);
    return cudaGetLastError();
  };
  if (p.K > 16) {  // 2K > 32 candidates per level: two per lane
    if (p.d == 128) {
      if (p.scoring == 1) return go(stage1_kernel<128, 1, 2>);
      if (p.scoring == 2) return go(stage1_kernel<128, 2, 2>);
      return go(stage1_kernel<128, 0, 2>);
    }
    if (p.scoring == 1) return go(stage1_kernel<64, 1, 2>);
    if (p.scoring == 2) return go(stage1_kernel<64, 2, 2>);
    return go(stage1_kernel<64, 0, 2>);
  }
  if (p.d == 128) {
    if (p.scoring == 1) return go(stage1_kernel<128, 1, 1>);
    if (p.scoring == 2) return go(stage1_kernel<128, 2, 1>);
    return go(stage1_kernel<128, 0, 1>);
  }
  if (p.scoring == 1) return go(stage1_kernel<64, 1, 1>);
  if (p.scoring == 2) return go(stage1_kernel<64, 2, 1>);
  return go(stage1_kernel<64, 0, 1>);
}

}  // namespace pisa
