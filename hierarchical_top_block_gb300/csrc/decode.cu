// Step 3 of the method (summary page of "Block Sparse Attention with Log-Linear
// Complexity", section "Method step details", step 3): one decode step per sequence in a
// single fused kernel.  The pyramid cache is updated only along the new token's path
// (its leaf from the raw keys, then every ancestor from its children, so the cache equals
// a fresh build bit for bit), one kernel walks every level down to the leaves (eq. 21
// scores, eq. 22 head sum, SelectK), scores the leaf candidates exactly, takes the final
// top-K with the own block, and attends over the selected blocks (step 4).
//
// One CTA (4 warps) per (sequence, KV head).  The level walk runs in warp 0 with the
// query group in mma.sync fragments and child summaries loaded straight into registers
// (d permuted identically in both operands); the leaf scoring and the attention split
// the blocks over the 4 warps; V blocks are staged in shared memory for ldmatrix.trans;
// the 4 partial softmax states are merged in shared memory.  seq_len is advanced by a
// second, one-thread-per-sequence kernel so that no CTA reads a length another changed.
#include "kernels.cuh"

namespace pisa {
namespace {

constexpr int WARPS = 4;
constexpr int THREADS = 32 * WARPS;


struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* Kc;
  uint16_t* Vc;
  uint16_t* Pc;
  const int32_t* seq_len;
  uint16_t* o;
  float* lse;
  int32_t* idx_out;
  // logits of the leaf candidates, kept for the attention (nullable): per (sequence, KV head)
  // [2K slots][8 key octets][sc_halves][sc_lanes] float2, in the MMA accumulator layout (lane
  // 4r + q holds head r; the lanes of heads past G_Q are not kept)
  float2* sc;
  int sc_halves;  // 2 when G_Q > 8 (rows r + 8 hold heads), else 1
  int sc_lanes;   // 4 min(G_Q, 8)
  int H_q, H_kv, GQ, Ksel, N_cap;
  int scoring;  // 0 LSE, 1 log m + mean, 2 log m + mean + variance / 2
  float sl2;
  long long nodes;          // P rows per (b, h_kv) in the capacity layout
  long long off[MAX_LEVELS + 1];
};

// level sizes for n tokens (C = 64, g = 2)
__device__ __forceinline__ int level_size(long long n, int l) {
  long long m = (n + 63) >> 6;
  for (int i = 1; i < l; ++i) m = (m + 1) >> 1;
  return (int)m;
}

// 4 CTAs per SM (<= 128 registers, 33 KB of shared memory): a batch of 64 sequences x 8 KV
// heads runs in one wave.  W: candidates per lane, 1 for K <= 16 (2K <= 32 per level and 2K
// leaf slots), 2 for K in 17..32 (lane l also holds candidate or slot l + 32).
template <int D, int W>
__global__ void __launch_bounds__(THREADS, 4) decode_kernel(DecodeParams p, uint32_t* err) {
  // L2 priorities: candidate K blocks may be read again by the attention (keep them), the
  // attention's K and V reads are their last use (let them go first)
  const uint64_t pol_keep = l2_evict_last_policy(), pol_last_use = l2_evict_first_policy();
  constexpr int NCH = D / 32;
  constexpr int NDT = D / 8;
  __shared__ int wlst[WARPS][32 * W];
  __shared__ float lvl_score[2][32 * W];
  __shared__ int cand_leaf[32 * W];
  __shared__ float cand_score[32 * W];
  __shared__ int ncand_s, nsel_s;
  __shared__ int sel[32];
  __shared__ int sel_slot[32];  // the candidate slot of each selected block, -1 if none
  __shared__ float part_m[WARPS][16], part_l[WARPS][16];
  extern __shared__ __align__(1024) uint8_t vbuf_raw[];
  uint8_t* vbuf = (uint8_t*)(((uintptr_t)vbuf_raw + 1023) & ~(uintptr_t)1023);  // [WARPS][32 x D bf16]

  const int bh = blockIdx.x;
  const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, q = lane & 3;
  const long long T = p.seq_len[b];
  const long long n = T + 1;
  if (T < 0 || T >= p.N_cap) {  // no room in the caches: report, write nothing
    if (tid == 0) report_error(err, ERR_BAD_INDEX);
    return;
  }
  uint16_t* Kb = p.Kc + (size_t)bh * p.N_cap * D;
  uint16_t* Vb = p.Vc + (size_t)bh * p.N_cap * D;
  uint16_t* Pb = p.Pc + (size_t)bh * p.nodes * D;

  // ---- append k, v and update the pyramid path of the new token ----
  if (tid < D) {
    Kb[(size_t)T * D + tid] = p.k[(size_t)bh * D + tid];
    Vb[(size_t)T * D + tid] = p.v[(size_t)bh * D + tid];
  }
  __syncthreads();
  int L = 1;
  while (level_size(n, L) > 1) ++L;
  if (tid < D) {
    // the new token's leaf: the mean of its <= 64 keys, summed in key order (the same
    // arithmetic as the pyramid build, so the cache equals a fresh build bit for bit); the
    // column is loaded in one batch first
    const long long leaf = T >> 6;
    const int cnt = (int)(T - leaf * 64 + 1);
    const uint16_t* kcol = Kb + (size_t)leaf * 64 * D + tid;
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < 64; i0 += 32) {  // 32 rows per batch of loads
      uint16_t kv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) kv[i] = i0 + i < cnt ? kcol[(size_t)(i0 + i) * D] : (uint16_t)0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (i0 + i < cnt) {
          float s, e;
          two_sum(hi, bf16_to_f32(kv[i]), s, e);
          hi = s;
          lo += e;
        }
      }
    }
    uint16_t cur = bf16_mean(hi, lo, cnt);
    Pb[(size_t)(p.off[1] + leaf) * D + tid] = cur;
    // ancestors: each is the mean of its (one or two) children; the child off the path is
    // unchanged by this step, so a chunk of levels' siblings is loaded first and the chain
    // runs in registers
    constexpr int CHUNK = 8;
    long long size = (n + 63) >> 6;  // size of level l-1
    for (int l0 = 2; l0 <= L; l0 += CHUNK) {
      float sib[CHUNK];
      long long sz = size;
#pragma unroll
      for (int u = 0; u < CHUNK; ++u) {
        const int l = l0 + u;
        if (l <= L) {
          const long long child = leaf >> (l - 2);
          sib[u] = (child | 1) < sz ? bf16_to_f32(Pb[(size_t)(p.off[l - 1] + (child ^ 1)) * D + tid]) : 0.f;
          sz = (sz + 1) >> 1;
        }
      }
#pragma unroll
      for (int u = 0; u < CHUNK; ++u) {
        const int l = l0 + u;
        if (l <= L) {
          const long long child = leaf >> (l - 2);
          const bool pair = (child | 1) < size;
          const float mine = bf16_to_f32(cur);
          float s, e;
          if (child & 1)
            two_sum(sib[u], mine, s, e);
          else
            two_sum(mine, sib[u], s, e);
          cur = bf16_mean(s, e, pair ? 2 : 1);
          Pb[(size_t)(p.off[l] + (child >> 1)) * D + tid] = cur;
          size = (size + 1) >> 1;
        }
      }
    }
  }
  __syncthreads();

  // query fragments, d permuted: chunk j of lane q holds d in [32j + 8q, 32j + 8q + 8)
  uint4 qa[NCH], qb[NCH];
  const uint16_t* qrow = p.q + ((size_t)b * p.H_q + (size_t)hk * p.GQ) * D;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    qa[j] = r < p.GQ ? ldg16(qrow + (size_t)r * D + 32 * j + 8 * q) : make_uint4(0, 0, 0, 0);
    qb[j] = r + 8 < p.GQ ? ldg16(qrow + (size_t)(r + 8) * D + 32 * j + 8 * q) : make_uint4(0, 0, 0, 0);
  }
  const unsigned lt_mask = (1u << lane) - 1u;

  // ---- level walk: every warp follows the same survivor list; a scored level's <= 32
  // candidates are split over the 4 warps (8 each), scored with the two children of each
  // candidate as MMA rows and the heads as columns, and meet in shared memory ----
  {
    int* mylst = wlst[warp];
    int surv = lane == 0 ? 0 : -1, ns = 1, par = 0;
    for (int l = L - 1; l >= 2; --l) {
      const int Ml = level_size(n, l);
      const int tl = (int)(T >> (l + 5));  // level-l node c starts at key c * 2^(l+5)
      const int c0 = 2 * surv, c1 = 2 * surv + 1;
      const bool e0 = lane < ns && c0 < Ml && c0 <= tl;
      const bool e1 = lane < ns && c1 < Ml && c1 <= tl;
      const unsigned b0 = __ballot_sync(0xffffffffu, e0), b1 = __ballot_sync(0xffffffffu, e1);
      const int pos = __popc(b0 & lt_mask) + __popc(b1 & lt_mask);
      const int nc = __popc(b0) + __popc(b1);
      if (e0) mylst[pos] = c0;
      if (e1) mylst[pos + (e0 ? 1 : 0)] = c1;
      __syncwarp();
      const int cand = lane < nc ? mylst[lane] : -1;
      int cand_hi = -1;  // candidates 32..63 (W == 2)
      if constexpr (W == 2) cand_hi = lane + 32 < nc ? mylst[lane + 32] : -1;
      __syncwarp();
      if (nc <= p.Ksel) {  // Ksel <= 32: the candidates fit one per lane
        surv = cand;
        ns = nc;
        continue;
      }
      const int Mc = level_size(n, l - 1);
      const int tc = (int)(T >> (l + 4));
      const uint16_t* Pl = Pb + (size_t)p.off[l - 1] * D;
      for (int mt = warp; 8 * mt < nc; mt += WARPS) {  // groups of 8 candidates over the warps
        const int ci = 8 * mt + r;
        const int cnode = __shfl_sync(0xffffffffu, mt >= 4 ? cand_hi : cand, ci & 31);
        const bool vc = ci < nc;
        const int ch = 2 * cnode;
        const bool v1 = vc && ch + 1 < Mc && ch + 1 <= tc;
        // read unconditionally: rows of an absent child or candidate only feed masked
        // scores, and row ch + 1 <= Mc lies inside the level's capacity or the next level
        const uint16_t* row = Pl + (size_t)(vc ? ch : 0) * D;
        uint4 k0[NCH], k1[NCH];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          k0[j] = ldg16(row + 32 * j + 8 * q);
          k1[j] = ldg16(row + D + 32 * j + 8 * q);
        }
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          mma_bf16_16816(a0, k0[j].x, k1[j].x, k0[j].y, k1[j].y, qa[j].x, qa[j].y);
          mma_bf16_16816(a0, k0[j].z, k1[j].z, k0[j].w, k1[j].w, qa[j].z, qa[j].w);
        }
        if (p.GQ > 8) {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            mma_bf16_16816(a1, k0[j].x, k1[j].x, k0[j].y, k1[j].y, qb[j].x, qb[j].y);
            mma_bf16_16816(a1, k0[j].z, k1[j].z, k0[j].w, k1[j].w, qb[j].z, qb[j].w);
          }
        }
        float part = 0.f;
        if (2 * q < p.GQ) part += pair_score(a0[0], a0[2], v1, p.sl2, p.scoring);
        if (2 * q + 1 < p.GQ) part += pair_score(a0[1], a0[3], v1, p.sl2, p.scoring);
        if (8 + 2 * q < p.GQ) part += pair_score(a1[0], a1[2], v1, p.sl2, p.scoring);
        if (9 + 2 * q < p.GQ) part += pair_score(a1[1], a1[3], v1, p.sl2, p.scoring);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (q == 0) lvl_score[par][ci] = vc ? part : NEG_INF;
      }
      __syncthreads();
      if constexpr (W == 2) {
        // SelectK over up to 64 candidates (every warp, same result), kept ones compacted in
        // list (ascending node) order
        float sv2[2] = {lane < nc ? lvl_score[par][lane] : NEG_INF, lane + 32 < nc ? lvl_score[par][lane + 32] : NEG_INF};
        int key2[2] = {lane, lane + 32}, id2[2] = {lane, lane + 32};
        par ^= 1;
        warp_top32_of64(sv2, key2, id2);
        const bool take = lane < p.Ksel;
        const unsigned k0 = __reduce_or_sync(0xffffffffu, take && id2[0] < 32 ? (1u << id2[0]) : 0u);
        const unsigned k1 = __reduce_or_sync(0xffffffffu, take && id2[0] >= 32 ? (1u << (id2[0] - 32)) : 0u);
        if ((k0 >> lane) & 1u) mylst[__popc(k0 & lt_mask)] = cand;
        if ((k1 >> lane) & 1u) mylst[__popc(k0) + __popc(k1 & lt_mask)] = cand_hi;
        __syncwarp();
        ns = __popc(k0) + __popc(k1);
        surv = lane < ns ? mylst[lane] : -1;
        __syncwarp();
        continue;
      }
      // SelectK (every warp, same result): bitonic sort of (score desc, index asc)
      float sv = lane < nc ? lvl_score[par][lane] : NEG_INF;
      int si = lane;
      par ^= 1;
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
      const unsigned km = __reduce_or_sync(0xffffffffu, lane < p.Ksel ? (1u << si) : 0u);
      const bool keep = (km >> lane) & 1u;
      if (keep) mylst[__popc(km & lt_mask)] = cand;
      __syncwarp();
      ns = __popc(km);
      surv = lane < ns ? mylst[lane] : -1;
      __syncwarp();
    }
    if (warp == 0) {
      // leaf candidates: eligible children of the level-2 survivors, slot 2i + c
      const int M1 = level_size(n, 1);
#pragma unroll
      for (int e = 0; e < W; ++e) {
        const int slot = 32 * e + lane;
        const int node = __shfl_sync(0xffffffffu, surv, (slot >> 1) & 31);
        if (slot < 2 * p.Ksel) {
          const int j = 2 * node + (slot & 1);
          cand_leaf[slot] = (node >= 0 && j < M1 && (long long)j * 64 <= T) ? j : -1;
        }
      }
      if (lane == 0) ncand_s = 2 * p.Ksel;
    }
  }
  __syncthreads();

  // ---- exact leaf LSE of the candidates (slots split over the warps) ----
  const int nslots = ncand_s;
  // with the logits kept, the attention reads no candidate's K rows again: no need to keep them
  const uint64_t pol_leaf_k = p.sc ? pol_last_use : pol_keep;
  for (int sidx = warp; sidx < nslots; sidx += WARPS) {
    const int leaf = cand_leaf[sidx];
    if (leaf < 0) continue;
    const long long key0 = (long long)leaf * 64;
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      const long long key = key0 + 8 * nt + r;
      const bool vis = key <= T;
      const uint16_t* krow = Kb + (size_t)(vis ? key : key0) * D;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const uint4 kv = vis ? ldg16_hint(krow + 32 * j + 8 * q, pol_leaf_k) : make_uint4(0, 0, 0, 0);
        mma_bf16_16816(acc[nt], qa[j].x, qb[j].x, qa[j].y, qb[j].y, kv.x, kv.y);
        mma_bf16_16816(acc[nt], qa[j].z, qb[j].z, qa[j].w, qb[j].w, kv.z, kv.w);
      }
    }
    // acc[nt]: rows (r | r+8) x keys key0 + 8nt + 2q + {0, 1}
    if (p.sc && lane < p.sc_lanes) {  // keep the logits: the attention over this leaf, if selected, reuses them
      const int nl = p.sc_lanes;
      float2* dst = p.sc + (((size_t)bh * 2 * p.Ksel + sidx) * 8) * p.sc_halves * nl + lane;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        st_f2_hint(dst + (size_t)nt * p.sc_halves * nl, make_float2(acc[nt][0], acc[nt][1]), pol_keep);
        if (p.sc_halves == 2) st_f2_hint(dst + (size_t)(nt * 2 + 1) * nl, make_float2(acc[nt][2], acc[nt][3]), pol_keep);
      }
    }
    float lse2_0, lse2_1;
    if (p.scoring != 0) {
      // truncated forms over the m visible keys, log2 units: log2 m + mean (+ ln2/2 Var)
      const int m = (int)min(T - key0 + 1, 64LL);
      float m0 = 0.f, m1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (key0 + 8 * nt + 2 * q + c <= T) {
            m0 += acc[nt][c] * p.sl2;
            m1 += acc[nt][2 + c] * p.sl2;
          }
      m0 += __shfl_xor_sync(0xffffffffu, m0, 1);
      m0 += __shfl_xor_sync(0xffffffffu, m0, 2);
      m1 += __shfl_xor_sync(0xffffffffu, m1, 1);
      m1 += __shfl_xor_sync(0xffffffffu, m1, 2);
      m0 /= (float)m;
      m1 /= (float)m;
      lse2_0 = fast_log2((float)m) + m0;
      lse2_1 = fast_log2((float)m) + m1;
      if (p.scoring == 2) {
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            if (key0 + 8 * nt + 2 * q + c <= T) {
              const float d0 = acc[nt][c] * p.sl2 - m0, d1 = acc[nt][2 + c] * p.sl2 - m1;
              v0 = fmaf(d0, d0, v0);
              v1 = fmaf(d1, d1, v1);
            }
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
        lse2_0 += 0.5f * LN2 * v0 / (float)m;
        lse2_1 += 0.5f * LN2 * v1 / (float)m;
      }
    } else {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const bool vis = key0 + 8 * nt + 2 * q + c <= T;
        s0 += vis ? fast_exp2(acc[nt][c] * p.sl2) : 0.f;
        s1 += vis ? fast_exp2(acc[nt][2 + c] * p.sl2) : 0.f;
      }
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    if (s0 > 0.f && s0 < POS_INF && s1 > 0.f && s1 < POS_INF) {
      lse2_0 = fast_log2(s0);
      lse2_1 = fast_log2(s1);
    } else {  // outside the fp32 exponent range: subtract the row maxima first
      float m0 = NEG_INF, m1 = NEG_INF;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (key0 + 8 * nt + 2 * q + c <= T) {
            m0 = fmaxf(m0, acc[nt][c] * p.sl2);
            m1 = fmaxf(m1, acc[nt][2 + c] * p.sl2);
          }
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
      m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      s0 = s1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (key0 + 8 * nt + 2 * q + c <= T) {
            s0 += fast_exp2(acc[nt][c] * p.sl2 - m0);
            s1 += fast_exp2(acc[nt][2 + c] * p.sl2 - m1);
          }
      s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
      s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      lse2_0 = m0 + fast_log2(s0);
      lse2_1 = m1 + fast_log2(s1);
    }
    }
    float part = (r < p.GQ ? lse2_0 : 0.f) + (r + 8 < p.GQ ? lse2_1 : 0.f);
    if (q != 0) part = 0.f;
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    part += __shfl_xor_sync(0xffffffffu, part, 8);
    part += __shfl_xor_sync(0xffffffffu, part, 16);
    if (lane == 0) cand_score[sidx] = part;
  }
  __syncthreads();

  // ---- final top-K with the own block (warp 0) ----
  // The candidate slots hold their leaves in ascending order; rank the other leaves by
  // (score desc, index asc) with a bitonic sort over the 32 lanes, keep K-1, and write the
  // kept leaves plus the own block in ascending order.
  if (W == 2 && warp == 0) {
    // 2K > 32 slots: two per lane, ranked by (score desc, leaf index asc) with the 64-entry
    // bitonic ranking; kept leaves and the own block written ascending
    const int own = (int)(T >> 6);
    int leaf[2];
    float v2[2];
    int key2[2], id2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int slot = 32 * e + lane;
      leaf[e] = slot < nslots ? cand_leaf[slot] : -1;
      if (leaf[e] == own) leaf[e] = -1;
      v2[e] = leaf[e] >= 0 ? cand_score[slot] : NEG_INF;
      key2[e] = leaf[e] >= 0 ? leaf[e] : 0x7fffffff;
      id2[e] = slot;
    }
    const unsigned valid0 = __ballot_sync(0xffffffffu, leaf[0] >= 0), valid1 = __ballot_sync(0xffffffffu, leaf[1] >= 0);
    warp_top32_of64(v2, key2, id2);
    const bool take = lane < p.Ksel - 1;
    const unsigned k0 = __reduce_or_sync(0xffffffffu, take && id2[0] < 32 ? (1u << id2[0]) : 0u) & valid0;
    const unsigned k1 = __reduce_or_sync(0xffffffffu, take && id2[0] >= 32 ? (1u << (id2[0] - 32)) : 0u) & valid1;
    const int n0 = __popc(k0);
    const unsigned b0 = __ballot_sync(0xffffffffu, leaf[0] >= 0 && leaf[0] < own);
    const unsigned b1 = __ballot_sync(0xffffffffu, leaf[1] >= 0 && leaf[1] < own);
    if ((k0 >> lane) & 1u) {
      const int at = __popc(k0 & lt_mask) + (own < leaf[0] ? 1 : 0);
      sel[at] = leaf[0];
      sel_slot[at] = lane;
    }
    if ((k1 >> lane) & 1u) {
      const int at = n0 + __popc(k1 & lt_mask) + (own < leaf[1] ? 1 : 0);
      sel[at] = leaf[1];
      sel_slot[at] = 32 + lane;
    }
    const unsigned own0 = __ballot_sync(0xffffffffu, lane < nslots && cand_leaf[lane] == own);
    const unsigned own1 = __ballot_sync(0xffffffffu, 32 + lane < nslots && cand_leaf[32 + lane] == own);
    if (lane == 0) {
      const int at = __popc(k0 & b0) + __popc(k1 & b1);
      sel[at] = own;
      sel_slot[at] = own0 ? __ffs(own0) - 1 : own1 ? 32 + __ffs(own1) - 1 : -1;
      nsel_s = n0 + __popc(k1) + 1;
    }
    __syncwarp();
    if (p.idx_out && lane < p.Ksel) p.idx_out[(size_t)bh * p.Ksel + lane] = lane < nsel_s ? sel[lane] : -1;
  } else if (warp == 0) {
    const int own = (int)(T >> 6);
    int leaf = lane < nslots ? cand_leaf[lane] : -1;
    if (leaf == own) leaf = -1;
    float sv = leaf >= 0 ? cand_score[lane] : NEG_INF;
    int sl = leaf >= 0 ? leaf : 0x7fffffff, si = lane;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, sv, j);
        const int ol = __shfl_xor_sync(0xffffffffu, sl, j);
        const int oi = __shfl_xor_sync(0xffffffffu, si, j);
        const bool other_better = ov > sv || (ov == sv && ol < sl);
        const bool lower = (lane & j) == 0, desc = (lane & k) == 0;
        if ((lower == desc) == other_better) {
          sv = ov;
          sl = ol;
          si = oi;
        }
      }
    }
    const unsigned km = __reduce_or_sync(0xffffffffu, (lane < p.Ksel - 1 && sl != 0x7fffffff) ? (1u << si) : 0u);
    const bool keep = (km >> lane) & 1u;
    const int pos = __popc(km & lt_mask);
    const int below = __popc(km & __ballot_sync(0xffffffffu, leaf >= 0 && leaf < own));
    if (keep) {
      sel[pos + (own < leaf ? 1 : 0)] = leaf;
      sel_slot[pos + (own < leaf ? 1 : 0)] = lane;
    }
    const unsigned own_at = __ballot_sync(0xffffffffu, lane < nslots && cand_leaf[lane] == own);
    if (lane == 0) {
      sel[below] = own;
      sel_slot[below] = own_at ? __ffs(own_at) - 1 : -1;
      nsel_s = __popc(km) + 1;
    }
    __syncwarp();
    if (p.idx_out && lane < p.Ksel) p.idx_out[(size_t)bh * p.Ksel + lane] = lane < nsel_s ? sel[lane] : -1;
  }
  __syncthreads();

  // ---- attention over the selected blocks in 32-key halves: warp w takes blocks w, w+4, ...
  // The half's V rows are copied into the warp's swizzled shared buffer asynchronously
  // while S = Q K^T runs on K rows loaded straight into registers; P V then uses
  // ldmatrix.trans on the buffer.
  const int nsel = nsel_s;
  float o[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  constexpr int HKEYS = 32;                 // keys per half block
  constexpr uint32_t HSPAN = HKEYS * 128;  // bytes of one 64-column half of the buffer
  uint8_t* vmine = vbuf + (size_t)warp * HKEYS * D * 2;
  const uint32_t vs = smem_u32(vmine);
  for (int si = warp; si < nsel; si += WARPS) {
    const int blk = sel[si];
    const int slot = p.sc ? sel_slot[si] : -1;  // the leaf phase kept this block's logits
#pragma unroll 1
    for (int hb = 0; hb < 2; ++hb) {
      const long long key0 = (long long)blk * 64 + HKEYS * hb;
      if (key0 > T) break;
      // V rows key0 .. key0 + 31 (rows past T become zero): row k, 16-byte chunk c at
      // (c ^ (k & 7)) within its 128-byte half row
      for (int i = lane; i < HKEYS * (D / 8); i += 32) {
        const int k = i / (D / 8), c = i % (D / 8);
        const long long key = key0 + k;
        const bool in = key <= T;
        cp_async16_hint(vmine + (c >> 3) * HSPAN + k * 128 + (((c & 7) ^ (k & 7)) << 4),
                        Vb + (size_t)(in ? key : key0) * D + 8 * c, in ? 16 : 0, pol_last_use);
      }
      cp_async_commit();
      float s[4][4];
      if (slot >= 0) {  // the same products the leaf phase computed, in the same layout
        const int nl = p.sc_lanes;
        const bool kept = lane < nl;  // rows of heads past G_Q read as zero (their outputs are not written)
        const float2* src = p.sc + (((size_t)bh * 2 * p.Ksel + slot) * 8 + 4 * hb) * p.sc_halves * nl + (kept ? lane : 0);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const float2 a = kept ? ld_f2_hint(src + (size_t)nt * p.sc_halves * nl, pol_last_use) : make_float2(0.f, 0.f);
          const float2 c = p.sc_halves == 2 ? ld_f2_hint(src + (size_t)(nt * 2 + 1) * nl, pol_last_use)
                                            : make_float2(0.f, 0.f);
          s[nt][0] = a.x;
          s[nt][1] = a.y;
          s[nt][2] = c.x;
          s[nt][3] = c.y;
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
          const long long key = key0 + 8 * nt + r;
          const uint16_t* krow = Kb + (size_t)(key <= T ? key : key0) * D;
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const uint4 kv = ldg16_hint(krow + 32 * j + 8 * q, pol_last_use);
            mma_bf16_16816(s[nt], qa[j].x, qb[j].x, qa[j].y, qb[j].y, kv.x, kv.y);
            mma_bf16_16816(s[nt], qa[j].z, qb[j].z, qa[j].w, qb[j].w, kv.z, kv.w);
          }
        }
      }
      // s[nt]: rows (r | r+8) x keys key0 + 8nt + 2q + {0,1}  (the n index maps key order 1:1)
      float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const bool vis = key0 + 8 * nt + 2 * q + c <= T;
          s[nt][c] = vis ? s[nt][c] * p.sl2 : NEG_INF;
          s[nt][2 + c] = vis ? s[nt][2 + c] * p.sl2 : NEG_INF;
          mx0 = fmaxf(mx0, s[nt][c]);
          mx1 = fmaxf(mx1, s[nt][2 + c]);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
      const float c0 = nm0 == NEG_INF ? 1.f : fast_exp2(m0 - nm0);
      const float c1 = nm1 == NEG_INF ? 1.f : fast_exp2(m1 - nm1);
      m0 = nm0;
      m1 = nm1;
      l0 *= c0;
      l1 *= c1;
#pragma unroll
      for (int i = 0; i < NDT; ++i) {
        o[i][0] *= c0;
        o[i][1] *= c0;
        o[i][2] *= c1;
        o[i][3] *= c1;
      }
      uint32_t pa[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float p00 = m0 == NEG_INF ? 0.f : fast_exp2(s[nt][0] - m0);
        const float p01 = m0 == NEG_INF ? 0.f : fast_exp2(s[nt][1] - m0);
        const float p10 = m1 == NEG_INF ? 0.f : fast_exp2(s[nt][2] - m1);
        const float p11 = m1 == NEG_INF ? 0.f : fast_exp2(s[nt][3] - m1);
        l0 += p00 + p01;
        l1 += p10 + p11;
        const int kk = nt >> 1, hi = nt & 1;
        pa[kk][hi ? 2 : 0] = pack_bf16x2(p00, p01);
        pa[kk][hi ? 3 : 1] = pack_bf16x2(p10, p11);
      }
      cp_async_wait_all();
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
        for (int np = 0; np < NDT / 2; ++np) {
          const int d0 = 8 * (2 * np + (lane >> 4));
          const uint32_t addr = vs + (d0 >> 6) * HSPAN + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(addr, b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
          mma_bf16_16816(o[2 * np + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
        }
      }
      __syncwarp();  // every lane is done with the buffer before the next half overwrites it
    }
  }
  // merge the per-warp softmax states (fixed order, deterministic)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (q == 0) {
    part_m[warp][r] = m0;
    part_l[warp][r] = l0;
    part_m[warp][r + 8] = m1;
    part_l[warp][r + 8] = l1;
  }
  __syncthreads();  // every warp is also done with its V staging buffer
  float* po = reinterpret_cast<float*>(vbuf);  // [WARPS][16][D] fp32, reuses the V buffers
  {
    float mm0 = NEG_INF, mm1 = NEG_INF;
    for (int w = 0; w < WARPS; ++w) {
      mm0 = fmaxf(mm0, part_m[w][r]);
      mm1 = fmaxf(mm1, part_m[w][r + 8]);
    }
    const float f0 = m0 == NEG_INF ? 0.f : fast_exp2(m0 - mm0);
    const float f1 = m1 == NEG_INF ? 0.f : fast_exp2(m1 - mm1);
#pragma unroll
    for (int i = 0; i < NDT; ++i)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = 8 * i + 2 * q + c;
        po[((size_t)warp * 16 + r) * D + col] = o[i][c] * f0;
        po[((size_t)warp * 16 + r + 8) * D + col] = o[i][2 + c] * f1;
      }
  }
  __syncthreads();
  for (int i = tid; i < p.GQ * D; i += THREADS) {
    const int row = i / D, col = i - (i / D) * D;
    float mm = NEG_INF;
    for (int w = 0; w < WARPS; ++w) mm = fmaxf(mm, part_m[w][row]);
    float lsum = 0.f, acc = 0.f;
    for (int w = 0; w < WARPS; ++w) {
      if (part_m[w][row] != NEG_INF) lsum += part_l[w][row] * fast_exp2(part_m[w][row] - mm);
      acc += po[((size_t)w * 16 + row) * D + col];
    }
    const size_t orow = (size_t)b * p.H_q + (size_t)hk * p.GQ + row;
    p.o[orow * D + col] = f32_to_bf16_rne(lsum > 0.f ? acc / lsum : 0.f);
    if (col == 0 && p.lse) p.lse[orow] = lsum > 0.f ? (mm + fast_log2(lsum)) * LN2 : NEG_INF;
  }
  (void)err;
}

__global__ void advance_seq_len_kernel(int32_t* seq_len, int B, int N_cap) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B && seq_len[b] >= 0 && seq_len[b] < N_cap) seq_len[b] += 1;
}

template <int D>
cudaError_t launch_d(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                     uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out, float* logits,
                     const Problem& pr, const Geometry& geo_cap, uint32_t* err, cudaStream_t s) {
  DecodeParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.Kc = Kc;
  p.Vc = Vc;
  p.Pc = Pc;
  p.seq_len = seq_len;
  p.o = o;
  p.lse = lse;
  p.idx_out = idx_out;
  p.sc = reinterpret_cast<float2*>(logits);
  p.sc_halves = pr.GQ > 8 ? 2 : 1;
  p.sc_lanes = 4 * (pr.GQ < 8 ? pr.GQ : 8);
  p.H_q = pr.H_q;
  p.H_kv = pr.H_kv;
  p.GQ = pr.GQ;
  p.Ksel = pr.K;
  p.scoring = pr.scoring;
  p.N_cap = pr.N_cap;
  p.sl2 = pr.scale * LOG2E;
  p.nodes = geo_cap.nodes;
  for (int l = 0; l <= MAX_LEVELS; ++l) p.off[l] = geo_cap.off[l];
  // V staging [WARPS][32 keys x D] bf16, also the merge buffer [WARPS][16][D] fp32
  const size_t smem = (size_t)WARPS * 32 * D * 2 + 1024;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<pr.B * pr.H_kv, THREADS, smem, s>>>(p, err);
    return cudaGetLastError();
  };
  cudaError_t e = pr.K > 16 ? go(decode_kernel<D, 2>) : go(decode_kernel<D, 1>);
  if (e != cudaSuccess) return e;
  advance_seq_len_kernel<<<(pr.B + 127) / 128, 128, 0, s>>>(seq_len, pr.B, pr.N_cap);
  return cudaGetLastError();
}

}  // namespace

size_t decode_logits_bytes(const Problem& p) {
  return (size_t)p.B * p.H_kv * 2 * p.K * 8 * (p.GQ > 8 ? 2 : 1) * 4 * (p.GQ < 8 ? p.GQ : 8) * sizeof(float2);
}

cudaError_t launch_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                          uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out, float* logits,
                          const Problem& p, const Geometry& geo_cap, uint32_t* err, cudaStream_t s) {
  if (p.d == 128) return launch_d<128>(q, k, v, Kc, Vc, Pc, seq_len, o, lse, idx_out, logits, p, geo_cap, err, s);
  return launch_d<64>(q, k, v, Kc, Vc, Pc, seq_len, o, lse, idx_out, logits, p, geo_cap, err, s);
}

}  // namespace pisa
