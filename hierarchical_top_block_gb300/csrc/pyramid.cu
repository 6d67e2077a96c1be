// Step 1 of the method (summary page of "Block Sparse Attention with Log-Linear
// Complexity", section "Method step details", eqs 10-15): the mean-pooled key pyramid.
// Leaf j = mean of keys [jC, min(jC+C, N)); node i of level l+1 = mean of its <= g = 2
// children.  Every node is rounded once to bf16 (nearest even) from an exact-to-2^-40
// sum: leaves accumulate with error-free fp32 TwoSum pairs and the level means are exact
// TwoSum pairs; dividing by a power-of-two count is an exact scaling, folded to bf16 by
// round-to-odd in fp32 (only a ragged last leaf divides in fp64, which is slow on GB300).
//
// HBM streaming: K is read once with 16-byte coalesced loads (one warp per leaf);
// each CTA owns a 16-leaf subtree and writes levels 1..5 of it from shared memory; a
// second small kernel builds the levels above (one CTA per (b, h_kv)).
// A build can be limited to a key range [lo, hi): it rewrites every node whose span meets the
// range (from K rows that may be incomplete past hi).  A sequence of builds over consecutive
// ranges, each run once the keys below its hi are in place, leaves every node whose span ends
// at or below the last hi exact: the last build that met its span ran with all its keys.
#include "kernels.cuh"

namespace pisa {
namespace {

constexpr int LPB = 16;           // leaves per CTA subtree
constexpr int SUB_LEVELS = 5;     // levels 1..5 of a 16-leaf subtree
constexpr int THREADS = 256;

template <int D>
__global__ void __launch_bounds__(THREADS) pyramid_leaves_kernel(const uint16_t* __restrict__ K,
                                                                 uint16_t* __restrict__ P, int N, int N_cap,
                                                                 Geometry geo, int top_level, int sub0, long long key_lo) {
  constexpr int LPR = D / 8;        // lanes per key row (16 bytes each)
  constexpr int RPI = 32 / LPR;     // rows per warp iteration
  __shared__ __align__(16) uint16_t buf[2][LPB][D];

  const int bh = blockIdx.y;
  const int sub = sub0 + (int)blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* Kb = K + (size_t)bh * N_cap * D;
  uint16_t* Pb = P + (size_t)bh * geo.nodes * D;
  const int M1 = geo.M[1];
  const int col = (lane % LPR) * 8;

  for (int li = warp; li < LPB; li += THREADS / 32) {
    const int leaf = sub * LPB + li;
    if (leaf >= M1) break;
    const int r0 = leaf * 64, r1 = min(N, r0 + 64);
    float hi[8], lo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hi[k] = lo[k] = 0.f;
#pragma unroll 8
    for (int r = r0 + lane / LPR; r < r1; r += RPI) {
      uint4 v = ldg16(Kb + (size_t)r * D + col);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float s, e;
        two_sum(hi[2 * k], bf16_lo(w[k]), s, e);
        hi[2 * k] = s;
        lo[2 * k] += e;
        two_sum(hi[2 * k + 1], bf16_hi(w[k]), s, e);
        hi[2 * k + 1] = s;
        lo[2 * k + 1] += e;
      }
    }
    // combine the partial sums of lanes that share a column
#pragma unroll
    for (int m = LPR; m < 32; m <<= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float oh = __shfl_xor_sync(0xffffffffu, hi[k], m);
        float ol = __shfl_xor_sync(0xffffffffu, lo[k], m);
        float s, e;
        two_sum(hi[k], oh, s, e);
        hi[k] = s;
        lo[k] = lo[k] + ol + e;
      }
    }
    if (lane < LPR) {
      const int cnt = r1 - r0;
      uint32_t packed[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint16_t a = bf16_mean(hi[2 * k], lo[2 * k], cnt);
        uint16_t b = bf16_mean(hi[2 * k + 1], lo[2 * k + 1], cnt);
        packed[k] = (uint32_t)a | ((uint32_t)b << 16);
      }
      uint4 out = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      // nodes below the range are exact already (and may be read meanwhile): not rewritten
      if ((long long)(leaf + 1) * 64 > key_lo) *reinterpret_cast<uint4*>(Pb + (size_t)(geo.off[1] + leaf) * D + col) = out;
      *reinterpret_cast<uint4*>(&buf[0][li][col]) = out;
    }
  }
  __syncthreads();

  // levels 2..top_level of this subtree, from shared memory
  int cur = 0;
  for (int l = 2; l <= top_level; ++l) {
    const int per = LPB >> (l - 1);                  // nodes of this subtree at level l
    const int first = (sub * LPB) >> (l - 1);        // global index of the first one
    const int first_child = (sub * LPB) >> (l - 2);
    for (int idx = threadIdx.x; idx < per * D; idx += THREADS) {
      const int i = idx / D, e = idx % D;
      const int node = first + i;
      if (node >= geo.M[l]) continue;
      const int c0 = 2 * node, c1 = min(2 * node + 2, geo.M[l - 1]);
      const float a = bf16_to_f32(buf[cur][c0 - first_child][e]);
      const float b = c1 - c0 > 1 ? bf16_to_f32(buf[cur][c0 + 1 - first_child][e]) : 0.f;
      float s, err;
      two_sum(a, b, s, err);
      const uint16_t v = bf16_mean(s, err, c1 - c0);
      if (((long long)(node + 1) << (l + 5)) > key_lo) Pb[(size_t)(geo.off[l] + node) * D + e] = v;
      buf[cur ^ 1][i][e] = v;
    }
    __syncthreads();
    cur ^= 1;
  }
}

// Levels first_level..L for one (b, h_kv), each from the level below it in P.  A thread takes
// 16-byte chunks (8 values of one row) in batches: all loads of a batch are issued before its
// stores, so a level costs about one memory round trip per batch instead of one per value.
template <int D>
__global__ void __launch_bounds__(THREADS) pyramid_upper_kernel(uint16_t* __restrict__ P, Geometry geo,
                                                                int first_level, long long key_lo, long long key_hi) {
  constexpr int CH = D / 8;   // chunks per row
  constexpr int BATCH = 8;
  uint16_t* Pb = P + (size_t)blockIdx.x * geo.nodes * D;
  for (int l = first_level; l <= geo.L; ++l) {
    const int m = geo.M[l], mc = geo.M[l - 1];
    // the nodes whose span (2^(l+5) keys) meets [key_lo, key_hi)
    const int n0 = (int)(key_lo >> (l + 5));
    const int n1 = (int)min((long long)m, ((key_hi - 1) >> (l + 5)) + 1);
    const int total = (n1 - n0) * CH;
    const uint16_t* src = Pb + (size_t)geo.off[l - 1] * D;
    uint16_t* dst = Pb + (size_t)geo.off[l] * D;
    for (int base = threadIdx.x; base < total; base += THREADS * BATCH) {
      uint4 va[BATCH], vb[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        va[u] = vb[u] = make_uint4(0, 0, 0, 0);
        if (idx < total) {
          const int node = n0 + idx / CH, c = idx - (idx / CH) * CH;
          va[u] = *reinterpret_cast<const uint4*>(src + (size_t)(2 * node) * D + 8 * c);
          if (2 * node + 1 < mc) vb[u] = *reinterpret_cast<const uint4*>(src + (size_t)(2 * node + 1) * D + 8 * c);
        }
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        if (idx >= total) continue;
        const int node = n0 + idx / CH, c = idx - (idx / CH) * CH;
        const int cnt = 2 * node + 1 < mc ? 2 : 1;
        const uint32_t wa[4] = {va[u].x, va[u].y, va[u].z, va[u].w}, wb[4] = {vb[u].x, vb[u].y, vb[u].z, vb[u].w};
        uint32_t packed[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float s0, e0, s1, e1;
          two_sum(bf16_lo(wa[k]), cnt > 1 ? bf16_lo(wb[k]) : 0.f, s0, e0);
          two_sum(bf16_hi(wa[k]), cnt > 1 ? bf16_hi(wb[k]) : 0.f, s1, e1);
          packed[k] = (uint32_t)bf16_mean(s0, e0, cnt) | ((uint32_t)bf16_mean(s1, e1, cnt) << 16);
        }
        *reinterpret_cast<uint4*>(dst + (size_t)node * D + 8 * c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
    __syncthreads();
  }
}

template <int D>
cudaError_t launch_pyramid_d(const uint16_t* K, uint16_t* P, const Problem& p, const Geometry& geo, long long key_lo,
                             long long key_hi, cudaStream_t s) {
  if (geo.L == 0 || key_hi <= key_lo) return cudaSuccess;
  const int top = geo.L < SUB_LEVELS ? geo.L : SUB_LEVELS;
  // the 16-leaf subtrees (1024 keys) that meet the range
  const int sub0 = (int)(key_lo / (64 * LPB)), sub1 = (int)((key_hi - 1) / (64 * LPB)) + 1;
  dim3 grid(sub1 - sub0, p.B * p.H_kv);
  pyramid_leaves_kernel<D><<<grid, THREADS, 0, s>>>(K, P, p.N, p.N_cap, geo, top, sub0, key_lo);
  if (geo.L > top) pyramid_upper_kernel<D><<<p.B * p.H_kv, THREADS, 0, s>>>(P, geo, top + 1, key_lo, key_hi);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pyramid_range(const uint16_t* K, uint16_t* P, const Problem& p, const Geometry& geo, long long key_lo,
                                 long long key_hi, cudaStream_t s) {
  if (key_hi > p.N) key_hi = p.N;
  if (p.d == 128) return launch_pyramid_d<128>(K, P, p, geo, key_lo, key_hi, s);
  return launch_pyramid_d<64>(K, P, p, geo, key_lo, key_hi, s);
}

cudaError_t launch_pyramid(const uint16_t* K, uint16_t* P, const Problem& p, const Geometry& geo, cudaStream_t s) {
  return launch_pyramid_range(K, P, p, geo, 0, p.N, s);
}

}  // namespace pisa
