// Backward of step 4 (the attention over the selected blocks; summary page of "Block Sparse
// Attention with Log-Linear Complexity", section "Method step details", step 4; the softmax
// covers the connected positions only, blog post of the same title, section 3.3).  The pages
// give no backward: this is the gradient of the forward function.  For query t, head h and
// the visible keys c of its selected blocks, with the forward's LSE:
//   P_c = exp(scale q.k_c - LSE),  D = dO . O,  dP_c = dO . v_c,  dS_c = P_c (dP_c - D)
//   dq = scale sum_c dS_c k_c,   dk_c += scale dS_c q,   dv_c += P_c dO
// (dk_c and dv_c summed over every query head of the group that selected c's block).
//
// Kernels: (1) D per (b, t, h) from the stored O and dO; (2) an inverse index, block ->
// the queries that selected it, each list sorted by position and cut into chunks of at most QC
// queries, the chunks ordered by their first position; then for d = 128 and G_Q of 8 or 16:
// (4') dK and dV on tcgen05, the chunk's queries in tiles of 128 query-head rows, which also
// writes dS of every (query, block) pair, and (3') dQ = scale dS K, one warp per query;
// otherwise (3) dQ, one warp per query over its selected blocks in 32-key halves (the
// forward's structure, with dP = dO V^T and dQ += dS K in place of P V) and (4) dK and dV, one
// 4-warp CTA per chunk, each warp owning 16 keys of the block and accumulating over the chunk's
// queries by mma.sync (their Q and dO rows staged three ahead in a 4-buffer ring).  dK and dV
// are added into fp32 (a block selected by many queries spans several chunks).
#include "kernels.cuh"
#include "pdl.cuh"

namespace pisa {
namespace {

constexpr int QC = 256;     // queries per dK/dV chunk
constexpr int HK = 32;      // keys per half block (dQ kernel)
constexpr int DQ_WARPS = 8;
constexpr int KV_WARPS = 4;
constexpr int KV_NBUF = 4;  // staged queries per dK/dV CTA (three prefetched ahead)
constexpr int SORT_CAP = 16384;   // block lists up to this length are sorted by query position
constexpr int NBUCKETS = 1024;    // position buckets for the chunk order

struct BwdParams {
  const uint16_t *Q, *K, *V, *O, *dO;
  const int32_t* idx;
  const float* LSE;
  float *dQ, *dK, *dV, *Dsum;
  uint16_t* dS;  // tcgen05 path: dS of every (query, selected block) by entry, [entries][G_Q][64] bf16,
                 // 16-byte chunks swizzled by head (chunk c of head h at c ^ (h & 7))
  int32_t* epos;  // tcgen05 path: entry of (b, h_kv, t, selection slot)
  int32_t *counts, *offsets, *entries;  // entries: (t << 5) | selection slot
  int32_t* rank;  // each selection entry's place in its block's list (from the counting atomics)
  int4* chunks;
  int32_t* nchunks;
  int4* chunks_by_t;            // the chunks reordered by their first query position
  int32_t *bucket_count, *bucket_start, *bucket_cursor;
  int bucket_shift;             // position bucket = t >> bucket_shift (< NBUCKETS)
  int B, N, N_cap, H_q, H_kv, GQ, Ksel, M1, causal;
  int tc;  // dK and dV on tcgen05 (with dS written out when dS is not null)
  float scale, sl2;
};

// swizzled [half][rows][64] bf16 tile: byte offset of row k, 16-byte chunk c (8 columns)
__device__ __forceinline__ uint32_t swz(int half_bytes, int k, int c) {
  return (c >> 3) * half_bytes + k * 128 + ((((c & 7) ^ (k & 7))) << 4);
}

// (1) D[b][h][t] = sum_e dO[b,t,h,e] O[b,t,h,e]: D / 8 lanes per row, 16 bytes of dO and of O
// each (coalesced: a warp reads 32 x 16 contiguous bytes of each), a shuffle tree per row
template <int D>
__global__ void bwd_dsum_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  constexpr int LPR = D / 8, RPW = 32 / LPR;  // lanes per row (16 at d = 128), rows per warp
  const long long rows = (long long)p.B * p.N * p.H_q;
  const int lane = threadIdx.x & 31, sub = lane % LPR;
  const long long nwarps = (long long)gridDim.x * (blockDim.x / 32);
  // warp-uniform loop (the shuffles need every lane): rows RPW w .. RPW w + RPW - 1
  for (long long w = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); w * RPW < rows; w += nwarps) {
    const long long i = w * RPW + lane / LPR;
    const bool ok = i < rows;
    float s = 0.f;
    if (ok) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(p.dO + i * D) + sub);
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(p.O + i * D) + sub);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) s += bf16_lo(xs[u]) * bf16_lo(ys[u]) + bf16_hi(xs[u]) * bf16_hi(ys[u]);
    }
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (ok && sub == 0) {
      const long long h = i % p.H_q, bt = i / p.H_q, t = bt % p.N, b = bt / p.N;
      p.Dsum[(b * p.H_q + h) * p.N + t] = s;
    }
  }
}

__device__ __forceinline__ bool valid_block(const BwdParams& p, int blk, int t) {
  return blk >= 0 && blk < p.M1 && (!p.causal || blk * 64 <= t);
}

// (2a) per (bh, block): how many queries selected it; the value each atomic returns is the
// entry's place in the block's list
__global__ void bwd_count_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  const long long total = (long long)p.B * p.H_kv * p.N * p.Ksel;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const long long item = i / p.Ksel;
    const int t = (int)(item % p.N), bh = (int)(item / p.N);
    const int blk = p.idx[i];
    if (valid_block(p, blk, t)) p.rank[i] = atomicAdd(&p.counts[(long long)bh * p.M1 + blk], 1);
  }
}

// (2b) exclusive scans of the counts and of the per-block chunk counts (one CTA)
__global__ void bwd_scan_kernel(BwdParams p, int nkeys, int32_t* chunk_off) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  __shared__ int32_t carry_s[2];
  __shared__ int32_t warp_s[2][32];
  if (threadIdx.x == 0) carry_s[0] = carry_s[1] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < nkeys; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int c = i < nkeys ? p.counts[i] : 0;
    const int ch = (c + QC - 1) / QC;
    int a = c, b = ch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) {
        a += ya;
        b += yb;
      }
    }
    if (lane == 31) {
      warp_s[0][warp] = a;
      warp_s[1][warp] = b;
    }
    __syncthreads();
    int pa = 0, pb = 0;
    for (int w = 0; w < warp; ++w) {
      pa += warp_s[0][w];
      pb += warp_s[1][w];
    }
    const int ca = carry_s[0], cb = carry_s[1];
    if (i < nkeys) {
      p.offsets[i] = ca + pa + a - c;
      chunk_off[i] = cb + pb + b - ch;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      carry_s[0] = ca + pa + a;
      carry_s[1] = cb + pb + b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.offsets[nkeys] = carry_s[0];
    *p.nchunks = carry_s[1];
  }
}

// (2c) each selection entry's query position into its block's list
__global__ void bwd_scatter_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  const long long total = (long long)p.B * p.H_kv * p.N * p.Ksel;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const long long item = i / p.Ksel;
    const int t = (int)(item % p.N), bh = (int)(item / p.N);
    const int blk = p.idx[i];
    if (!valid_block(p, blk, t)) continue;
    const long long key = (long long)bh * p.M1 + blk;
    p.entries[p.offsets[key] + p.rank[i]] = (t << 5) | (int)(i - item * p.Ksel);
  }
}

// (2d) chunk records {bh, block, first entry, count}
__global__ void bwd_chunks_kernel(BwdParams p, int nkeys, const int32_t* chunk_off) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  for (int key = blockIdx.x * blockDim.x + threadIdx.x; key < nkeys; key += gridDim.x * blockDim.x) {
    const int c = p.counts[key];
    const int bh = key / p.M1, blk = key - bh * p.M1;
    for (int j = 0; j * QC < c; ++j)
      p.chunks[chunk_off[key] + j] = make_int4(bh, blk, p.offsets[key] + j * QC, min(QC, c - j * QC));
  }
}

// (2e) each block's query list in increasing position (a list longer than SORT_CAP keeps its
// order), so that a chunk covers a narrow band of positions: one CTA per list, bitonic sort in
// shared memory.  The entries (t << 5 | slot) are distinct, so the order is unique.
__global__ void __launch_bounds__(512) bwd_sort_lists_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  extern __shared__ int32_t sbuf[];
  const int key = blockIdx.x;
  const int lo = p.offsets[key], n = p.offsets[key + 1] - lo;
  const long long bh = key / p.M1;
  auto place = [&](int i, int e) {  // where entry lo + i (= e) sits, for the dQ kernel
    if (p.epos) p.epos[((long long)bh * p.N + (e >> 5)) * p.Ksel + (e & 31)] = lo + i;
  };
  if (n <= 1 || n > SORT_CAP) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) place(i, p.entries[lo + i]);
    return;
  }
  int np = 2;
  while (np < n) np <<= 1;
  for (int i = threadIdx.x; i < np; i += blockDim.x) sbuf[i] = i < n ? p.entries[lo + i] : INT_MAX;
  __syncthreads();
  for (int k = 2; k <= np; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < np; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const int a = sbuf[i], b = sbuf[l];
          if ((a > b) == ((i & k) == 0)) {
            sbuf[i] = b;
            sbuf[l] = a;
          }
        }
      }
      __syncthreads();
    }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    p.entries[lo + i] = sbuf[i];
    place(i, sbuf[i]);
  }
}

// (2f) the chunks in order of their first query position (counting sort by position bucket;
// order inside a bucket arbitrary): the persistent dK/dV CTAs then work on chunks whose
// queries lie close together, and their Q and dO rows are re-read from the L2
__device__ __forceinline__ int chunk_bucket(const BwdParams& p, int ci) {
  return (p.entries[p.chunks[ci].z] >> 5) >> p.bucket_shift;
}

__global__ void bwd_bucket_count_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  const int n = *p.nchunks;
  for (int ci = blockIdx.x * blockDim.x + threadIdx.x; ci < n; ci += gridDim.x * blockDim.x)
    atomicAdd(&p.bucket_count[chunk_bucket(p, ci)], 1);
}

__global__ void __launch_bounds__(NBUCKETS) bwd_bucket_scan_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  __shared__ int32_t ws[NBUCKETS / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = p.bucket_count[threadIdx.x];
  int a = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, a, o);
    if (lane >= o) a += y;
  }
  if (lane == 31) ws[warp] = a;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += ws[w];
  p.bucket_start[threadIdx.x] = base + a - c;
}

__global__ void bwd_bucket_scatter_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  const int n = *p.nchunks;
  for (int ci = blockIdx.x * blockDim.x + threadIdx.x; ci < n; ci += gridDim.x * blockDim.x) {
    const int b = chunk_bucket(p, ci);
    p.chunks_by_t[p.bucket_start[b] + atomicAdd(&p.bucket_cursor[b], 1)] = p.chunks[ci];
  }
}

// (3) dQ: one warp per (b, h_kv, t)
template <int D>
__global__ void __launch_bounds__(32 * DQ_WARPS) bwd_dq_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  constexpr int KST = D / 16, NDT = D / 8, CPR = D / 8;
  constexpr int HALF = HK * 128;             // bytes of one 64-column half of a slot
  constexpr int SLOT = HK * D * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  uint8_t* ks = smem + (size_t)warp * 2 * SLOT;
  uint8_t* vs = ks + SLOT;
  const uint32_t kb = smem_u32(ks), vb = smem_u32(vs);
  const long long total = (long long)p.B * p.H_kv * p.N;
  for (long long item = (long long)blockIdx.x * DQ_WARPS + warp; item < total; item += (long long)gridDim.x * DQ_WARPS) {
    const int bh = (int)(item / p.N), t = (int)(item - (long long)bh * p.N);
    const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
    const int last = p.causal ? min(t, p.N - 1) : p.N - 1;
    int v = lane < p.Ksel ? p.idx[item * p.Ksel + lane] : -1;
    if (!valid_block(p, v, t)) v = -1;
    unsigned mask = __ballot_sync(0xffffffffu, v >= 0);
    // A fragments of Q and dO (rows r, r+8 of the group; zero past G_Q)
    const size_t row0 = ((size_t)b * p.N + t) * p.H_q + (size_t)hk * p.GQ;
    uint32_t qa[KST][4], da[KST][4];
#pragma unroll
    for (int s = 0; s < KST; ++s) {
      const int c0 = 16 * s + 2 * q;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rr = r + 8 * (u & 1), cc = c0 + 8 * (u >> 1);
        const bool in = rr < p.GQ;
        qa[s][u] = in ? *reinterpret_cast<const uint32_t*>(p.Q + (row0 + rr) * D + cc) : 0u;
        da[s][u] = in ? *reinterpret_cast<const uint32_t*>(p.dO + (row0 + rr) * D + cc) : 0u;
      }
    }
    // per row: log2-domain LSE (+inf zeroes P on padded or empty rows) and D
    float lse2[2], dsum[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int rr = r + 8 * u;
      const size_t li = ((size_t)b * p.H_q + (size_t)hk * p.GQ + rr) * p.N + t;
      const float l = rr < p.GQ ? p.LSE[li] : NEG_INF;
      lse2[u] = l == NEG_INF ? POS_INF : l * LOG2E;
      dsum[u] = rr < p.GQ ? p.Dsum[li] : 0.f;
    }
    float dq[NDT][4];
#pragma unroll
    for (int i = 0; i < NDT; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
    for (; mask; mask &= mask - 1) {
      const int blk = __shfl_sync(0xffffffffu, v, __ffs(mask) - 1);
#pragma unroll 1
      for (int hb = 0; hb < 2; ++hb) {
        const int kbase = blk * 64 + HK * hb;
        if (kbase > last) break;
        // K and V rows kbase .. kbase + 31 (rows past the last visible key become zero)
        const uint16_t* Kg = p.K + ((size_t)bh * p.N_cap) * D;
        const uint16_t* Vg = p.V + ((size_t)bh * p.N_cap) * D;
        for (int i = lane; i < HK * CPR; i += 32) {
          const int k = i / CPR, c = i - k * CPR;
          const int key = kbase + k;
          const bool in = key <= last;
          const size_t off = (size_t)(in ? key : kbase) * D + 8 * c;
          cp_async16(ks + swz(HALF, k, c), Kg + off, in ? 16 : 0);
          cp_async16(vs + swz(HALF, k, c), Vg + off, in ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncwarp();
        // S = Q K^T and dP = dO V^T over 32 keys (4 n-tiles)
        float sacc[4][4], pacc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int u = 0; u < 4; ++u) sacc[nt][u] = pacc[nt][u] = 0.f;
#pragma unroll
        for (int kp = 0; kp < KST / 2; ++kp) {
          const int d0 = 32 * kp + 8 * (lane >> 3);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            const int key = 8 * nt + (lane & 7);
            const uint32_t off = (d0 >> 6) * HALF + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kb + off, b0, b1, b2, b3);
            mma_bf16_16816(sacc[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b0, b1);
            mma_bf16_16816(sacc[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2], qa[2 * kp + 1][3], b2, b3);
            ldmatrix_x4(vb + off, b0, b1, b2, b3);
            mma_bf16_16816(pacc[nt], da[2 * kp][0], da[2 * kp][1], da[2 * kp][2], da[2 * kp][3], b0, b1);
            mma_bf16_16816(pacc[nt], da[2 * kp + 1][0], da[2 * kp + 1][1], da[2 * kp + 1][2], da[2 * kp + 1][3], b2, b3);
          }
        }
        // dS = P (dP - D), packed as bf16 A fragments (keys are the k index of dQ += dS K)
        uint32_t sa[2][4];
        if (kbase + 31 <= last) {  // every key of the half block visible: packed fp32 pairs
          const unsigned long long sl2x2 = pack_f32x2(p.sl2, p.sl2);
          const unsigned long long nl0 = pack_f32x2(-lse2[0], -lse2[0]), nl1 = pack_f32x2(-lse2[1], -lse2[1]);
          const unsigned long long nd0 = pack_f32x2(-dsum[0], -dsum[0]), nd1 = pack_f32x2(-dsum[1], -dsum[1]);
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            float x0, x1, x2, x3;
            unpack_f32x2(fma_f32x2(pack_f32x2(sacc[nt][0], sacc[nt][1]), sl2x2, nl0), x0, x1);
            unpack_f32x2(fma_f32x2(pack_f32x2(sacc[nt][2], sacc[nt][3]), sl2x2, nl1), x2, x3);
            float d0, d1, d2, d3;
            unpack_f32x2(mul_f32x2(pack_f32x2(fast_exp2(x0), fast_exp2(x1)),
                                   add_f32x2(pack_f32x2(pacc[nt][0], pacc[nt][1]), nd0)), d0, d1);
            unpack_f32x2(mul_f32x2(pack_f32x2(fast_exp2(x2), fast_exp2(x3)),
                                   add_f32x2(pack_f32x2(pacc[nt][2], pacc[nt][3]), nd1)), d2, d3);
            const int kk = nt >> 1, hi = nt & 1;
            sa[kk][hi ? 2 : 0] = pack_bf16x2(d0, d1);
            sa[kk][hi ? 3 : 1] = pack_bf16x2(d2, d3);
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            float ds[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int key = kbase + 8 * nt + 2 * q + (u & 1);
              const int rr = u >> 1;
              const float pr = key <= last ? fast_exp2(fmaf(sacc[nt][u], p.sl2, -lse2[rr])) : 0.f;
              ds[u] = pr * (pacc[nt][u] - dsum[rr]);
            }
            const int kk = nt >> 1, hi = nt & 1;
            sa[kk][hi ? 2 : 0] = pack_bf16x2(ds[0], ds[1]);
            sa[kk][hi ? 3 : 1] = pack_bf16x2(ds[2], ds[3]);
          }
        }
        // dQ += dS K (K^T fragments by ldmatrix.trans on the K slot)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int key = 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
          for (int np = 0; np < NDT / 2; ++np) {
            const int d0 = 8 * (2 * np + (lane >> 4));
            const uint32_t addr = kb + (d0 >> 6) * HALF + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(addr, b0, b1, b2, b3);
            mma_bf16_16816(dq[2 * np], sa[kk][0], sa[kk][1], sa[kk][2], sa[kk][3], b0, b1);
            mma_bf16_16816(dq[2 * np + 1], sa[kk][0], sa[kk][1], sa[kk][2], sa[kk][3], b2, b3);
          }
        }
        __syncwarp();  // every lane is done with the slots before the next copy
      }
    }
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = 8 * i + 2 * q;
      if (r < p.GQ)
        *reinterpret_cast<float2*>(p.dQ + (row0 + r) * D + col) = make_float2(dq[i][0] * p.scale, dq[i][1] * p.scale);
      if (r + 8 < p.GQ)
        *reinterpret_cast<float2*>(p.dQ + (row0 + r + 8) * D + col) =
            make_float2(dq[i][2] * p.scale, dq[i][3] * p.scale);
    }
  }
}

// (3') dQ from the dS rows the tcgen05 dK/dV kernel wrote (d = 128): one warp per (b, h_kv, t)
// over its selected blocks in 32-key halves, dQ += dS K.  Each warp streams its queries'
// selections through a ring of shared-memory slots: per half block, the K rows by TMA (one box:
// 32 rows x both 64-column halves of d, 128-byte swizzle, rows past N read as zero) and the
// (query, block) pair's dS rows by a bulk copy (stored by entry, swizzled as the dK/dV kernel's
// tile was; found through the (query, slot) -> entry map), on one barrier.  A cursor walks the
// same sequence of half blocks DQS_SLOTS - 1 ahead of the multiplications, across query
// boundaries, so the dS reads from DRAM are off the path.  All waits are bounded.
constexpr int DQS_WARPS = 11, DQS_SLOTS = 2;

struct DqCursor {
  long long item;  // (bh, t) as bh * N + t; >= total once exhausted
  unsigned mask;   // selection positions of the item not yet passed (the current block first)
  int val;         // this lane's selection entry of the item (-1 if not a valid block)
  int ent;         // the dS entry of this lane's selection slot
  int hb;          // half of the current block
  int last;        // last visible key of the item's query
};

// positions the cursor on the first visible half block of item `it` or of a later item
__device__ __forceinline__ void dq_seek(DqCursor& c, const BwdParams& p, long long it, long long total, long long stride) {
  const int lane = threadIdx.x & 31;
  for (; it < total; it += stride) {
    const int t = (int)(it % p.N);
    int v = lane < p.Ksel ? p.idx[it * p.Ksel + lane] : -1;
    if (!valid_block(p, v, t)) v = -1;
    const unsigned m = __ballot_sync(0xffffffffu, v >= 0);
    if (m) {
      c.item = it;
      c.mask = m;
      c.val = v;
      c.ent = v >= 0 ? p.epos[it * p.Ksel + lane] : 0;
      c.hb = 0;
      c.last = p.causal ? min(t, p.N - 1) : p.N - 1;
      return;
    }
  }
  c.item = total;
}

__device__ __forceinline__ int dq_block(const DqCursor& c) { return __shfl_sync(0xffffffffu, c.val, __ffs(c.mask) - 1); }

__device__ __forceinline__ void dq_next(DqCursor& c, const BwdParams& p, long long total, long long stride) {
  if (c.hb == 0 && dq_block(c) * 64 + HK <= c.last) {
    c.hb = 1;
    return;
  }
  c.hb = 0;
  c.mask &= c.mask - 1;
  if (!c.mask) dq_seek(c, p, c.item + stride, total, stride);
}

__global__ void __launch_bounds__(32 * DQS_WARPS, 1) bwd_dq_ds_kernel(const __grid_constant__ CUtensorMap mapK, BwdParams p,
                                                                    uint32_t* err) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  constexpr int D = 128, NDT = D / 8;
  constexpr int HALF = HK * 128;             // bytes of one 64-column half of a slot
  constexpr int SLOT = HK * D * 2;
  constexpr int SLOT_ALL = SLOT + 16 * 128;  // the K half block, then the pair's dS rows (up to 16 x 64)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar[DQS_WARPS][DQS_SLOTS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  uint8_t* slots = smem + (size_t)warp * DQS_SLOTS * SLOT_ALL;
  if (lane == 0) {
    for (int i = 0; i < DQS_SLOTS; ++i) mbar_init(&bar[warp][i], 1);
    mbar_fence_init();
  }
  __syncwarp();
  const long long total = (long long)p.B * p.H_kv * p.N;
  const long long stride = (long long)gridDim.x * DQS_WARPS;
  const long long first = (long long)blockIdx.x * DQS_WARPS + warp;
  // the copy of one K half block into a slot (its previous contents were read by ldmatrix whose
  // results fed MMAs issued before this point, so those reads are complete)
  auto issue = [&](const DqCursor& c, int slot) {
    const int bh = (int)(c.item / p.N);
    const int row = dq_block(c) * 64 + HK * c.hb;
    const int ent = __shfl_sync(0xffffffffu, c.ent, __ffs(c.mask) - 1);
    const uint32_t ds_bytes = (uint32_t)(p.GQ * 128);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[warp][slot], SLOT + ds_bytes);
      tma_load_4d(slots + slot * SLOT_ALL, &mapK, &bar[warp][slot], 0, row, 0, bh);
      asm volatile(  // the pair's dS rows (swizzled as stored)
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(slots + slot * SLOT_ALL + SLOT)),
          "l"(p.dS + (size_t)ent * (size_t)(p.GQ * 64)), "r"(ds_bytes), "r"(smem_u32(&bar[warp][slot]))
          : "memory");
    }
  };
  DqCursor ck;  // the next K half block to load
  dq_seek(ck, p, first, total, stride);
  long long nk = 0, h = 0;  // half blocks issued, half blocks consumed
  for (; nk < DQS_SLOTS - 1 && ck.item < total; ++nk) {
    issue(ck, (int)(nk % DQS_SLOTS));
    dq_next(ck, p, total, stride);
  }

  bool ok = true;
  for (long long item = first; item < total && ok; item += stride) {
    const int bh = (int)(item / p.N), t = (int)(item - (long long)bh * p.N);
    const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
    const int last = p.causal ? min(t, p.N - 1) : p.N - 1;
    int v = lane < p.Ksel ? p.idx[item * p.Ksel + lane] : -1;
    if (!valid_block(p, v, t)) v = -1;
    unsigned mask = __ballot_sync(0xffffffffu, v >= 0);
    const size_t row0 = ((size_t)b * p.N + t) * p.H_q + (size_t)hk * p.GQ;
    float dq[NDT][4];
#pragma unroll
    for (int i = 0; i < NDT; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;
    for (; mask && ok; mask &= mask - 1) {
      const int sl = __ffs(mask) - 1;
      const int blk = __shfl_sync(0xffffffffu, v, sl);
#pragma unroll 1
      for (int hb = 0; hb < 2; ++hb) {
        if (blk * 64 + HK * hb > last) break;
        // keep DQS_SLOTS - 1 half blocks in flight beyond this one
        if (ck.item < total) {
          issue(ck, (int)(nk % DQS_SLOTS));
          dq_next(ck, p, total, stride);
          ++nk;
        }
        const int slot = (int)(h % DQS_SLOTS);
        if (!mbar_wait_warp(&bar[warp][slot], (uint32_t)(h / DQS_SLOTS) & 1u, err)) {
          ok = false;
          break;
        }
        // dS as bf16 A fragments from the slot's dS rows: rows r, r+8 (heads; zero past G_Q), keys
        // 32 hb + 16 kk + {2q, 2q + 8}: chunk 4 hb + 2 kk (+1) at its swizzled place (h & 7 = r)
        const uint8_t* dsm = slots + slot * SLOT_ALL + SLOT;
        uint32_t sa[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int o0 = (((4 * hb + 2 * kk) ^ r) << 4) + 4 * q, o1 = (((4 * hb + 2 * kk + 1) ^ r) << 4) + 4 * q;
          sa[kk][0] = r < p.GQ ? *reinterpret_cast<const uint32_t*>(dsm + r * 128 + o0) : 0u;
          sa[kk][1] = r + 8 < p.GQ ? *reinterpret_cast<const uint32_t*>(dsm + (r + 8) * 128 + o0) : 0u;
          sa[kk][2] = r < p.GQ ? *reinterpret_cast<const uint32_t*>(dsm + r * 128 + o1) : 0u;
          sa[kk][3] = r + 8 < p.GQ ? *reinterpret_cast<const uint32_t*>(dsm + (r + 8) * 128 + o1) : 0u;
        }
        // dQ += dS K (K^T fragments by ldmatrix.trans on the slot)
        const uint32_t kb = smem_u32(slots + slot * SLOT_ALL);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const int key = 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
          for (int np = 0; np < NDT / 2; ++np) {
            const int d0 = 8 * (2 * np + (lane >> 4));
            const uint32_t addr = kb + (d0 >> 6) * HALF + key * 128 + ((((d0 & 63) >> 3) ^ (key & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(addr, b0, b1, b2, b3);
            mma_bf16_16816(dq[2 * np], sa[kk][0], sa[kk][1], sa[kk][2], sa[kk][3], b0, b1);
            mma_bf16_16816(dq[2 * np + 1], sa[kk][0], sa[kk][1], sa[kk][2], sa[kk][3], b2, b3);
          }
        }
        ++h;
      }
    }
    if (!ok) break;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = 8 * i + 2 * q;
      if (r < p.GQ)
        *reinterpret_cast<float2*>(p.dQ + (row0 + r) * D + col) = make_float2(dq[i][0] * p.scale, dq[i][1] * p.scale);
      if (r + 8 < p.GQ)
        *reinterpret_cast<float2*>(p.dQ + (row0 + r + 8) * D + col) =
            make_float2(dq[i][2] * p.scale, dq[i][3] * p.scale);
    }
  }
  // after a timeout, copies still in flight land before shared memory goes away (bounded)
  if (!ok)
    for (long long u = h; u < nk; ++u)
      mbar_wait_warp(&bar[warp][u % DQS_SLOTS], (uint32_t)(u / DQS_SLOTS) & 1u, err, 100000000ull);
}

// Bulk copy shared -> global of `bytes` (a multiple of 16; both addresses 16-byte aligned),
// tracked in the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the thread's committed bulk copies have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and finished writing global memory
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void red_add(float* a, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(a), "f"(v) : "memory");
}

// (4) dK, dV: one CTA of 4 warps per chunk; warp w owns keys 16w .. 16w + 15 of the block
template <int D>
// 3 CTAs per SM (<= 168 registers): the per-query chain is latency-bound, more warps hide it
__global__ void __launch_bounds__(32 * KV_WARPS, 3) bwd_dkv_kernel(BwdParams p) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  constexpr int KST = D / 16, NDT = D / 8, CPR = D / 8;
  constexpr int KHALF = 64 * 128;            // K/V tiles: [half][64 keys][64]
  constexpr int QHALF = 16 * 128;            // Q/dO tiles: [half][16 heads][64]
  constexpr int KTILE = 64 * D * 2, QTILE = 16 * D * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* Ks = smem;
  uint8_t* Vs = Ks + KTILE;
  uint8_t* Qs = Vs + KTILE;                  // [KV_NBUF][QTILE]
  uint8_t* dOs = Qs + KV_NBUF * QTILE;       // [KV_NBUF][QTILE]
  __shared__ float lse2_s[KV_NBUF][16], dsum_s[KV_NBUF][16];
  __shared__ int t_s[KV_NBUF];
  if (blockIdx.x >= *p.nchunks) return;
  const int4 ch = p.chunks[blockIdx.x];
  const int bh = ch.x, blk = ch.y, first = ch.z, cnt = ch.w;
  const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, r = lane >> 2, q = lane & 3;
  const int key0 = blk * 64;
  // the block's K and V (rows past N become zero)
  {
    const uint16_t* Kg = p.K + ((size_t)bh * p.N_cap) * D;
    const uint16_t* Vg = p.V + ((size_t)bh * p.N_cap) * D;
    for (int i = threadIdx.x; i < 64 * CPR; i += blockDim.x) {
      const int k = i / CPR, c = i - k * CPR;
      const bool in = key0 + k < p.N;
      const size_t off = (size_t)(in ? key0 + k : key0) * D + 8 * c;
      cp_async16(Ks + swz(KHALF, k, c), Kg + off, in ? 16 : 0);
      cp_async16(Vs + swz(KHALF, k, c), Vg + off, in ? 16 : 0);
    }
  }
  // one query's Q and dO rows (heads past G_Q become zero), log2 LSE and D, into buffer bf
  auto stage = [&](int i, int bf) {
    const int t = p.entries[first + i] >> 5;
    const size_t row0 = ((size_t)b * p.N + t) * p.H_q + (size_t)hk * p.GQ;
    for (int j = threadIdx.x; j < 16 * CPR; j += blockDim.x) {
      const int h = j / CPR, c = j - h * CPR;
      const bool in = h < p.GQ;
      const size_t off = (row0 + (in ? h : 0)) * D + 8 * c;
      cp_async16(Qs + bf * QTILE + swz(QHALF, h, c), p.Q + off, in ? 16 : 0);
      cp_async16(dOs + bf * QTILE + swz(QHALF, h, c), p.dO + off, in ? 16 : 0);
    }
    if (threadIdx.x < 16) {
      const int h = threadIdx.x;
      const size_t li = ((size_t)b * p.H_q + (size_t)hk * p.GQ + h) * p.N + t;
      const float l = h < p.GQ ? p.LSE[li] : NEG_INF;
      lse2_s[bf][h] = l == NEG_INF ? POS_INF : l * LOG2E;
      dsum_s[bf][h] = h < p.GQ ? p.Dsum[li] : 0.f;
    }
    if (threadIdx.x == 0) t_s[bf] = t;
  };
  // the K/V copies join the first group; every iteration commits one (possibly empty) group,
  // so waiting until KV_NBUF - 1 groups remain in flight completes the current query's
  for (int j = 0; j < KV_NBUF - 1; ++j) {
    if (j < cnt) stage(j, j);
    cp_async_commit();
  }
  float dk[NDT][4], dv[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i)
#pragma unroll
    for (int u = 0; u < 4; ++u) dk[i][u] = dv[i][u] = 0.f;
  const uint32_t ksa = smem_u32(Ks), vsa = smem_u32(Vs);
  for (int i = 0; i < cnt; ++i) {
    const int bf = i % KV_NBUF;
    if (i + KV_NBUF - 1 < cnt) stage(i + KV_NBUF - 1, (i + KV_NBUF - 1) % KV_NBUF);
    cp_async_commit();
    asm volatile("cp.async.wait_group %0;" ::"n"(KV_NBUF - 1) : "memory");
    __syncthreads();
    const int t = t_s[bf];
    const int last = p.causal ? min(t, p.N - 1) : p.N - 1;
    const uint32_t qsa = smem_u32(Qs + bf * QTILE), dsa = smem_u32(dOs + bf * QTILE);
    // S^T [16 keys x 16 heads] = K_w Q^T and dP^T = V_w dO^T
    float sacc[2][4], pacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int u = 0; u < 4; ++u) sacc[nt][u] = pacc[nt][u] = 0.f;
#pragma unroll
    for (int s = 0; s < KST; ++s) {
      const int m = lane >> 3;
      // A: rows 16w + 8 (m & 1) + (lane & 7), columns 16 s + 8 (m >> 1)
      const int ak = 16 * warp + 8 * (m & 1) + (lane & 7), ac = 2 * s + (m >> 1);
      uint32_t k0, k1, k2, k3, v0, v1, v2, v3;
      ldmatrix_x4(ksa + swz(KHALF, ak, ac), k0, k1, k2, k3);
      ldmatrix_x4(vsa + swz(KHALF, ak, ac), v0, v1, v2, v3);
      // B: heads 8 (m >> 1) + (lane & 7), columns 16 s + 8 (m & 1)
      const int bh8 = 8 * (m >> 1) + (lane & 7), bc = 2 * s + (m & 1);
      uint32_t q0, q1, q2, q3, o0, o1, o2, o3;
      ldmatrix_x4(qsa + swz(QHALF, bh8, bc), q0, q1, q2, q3);
      ldmatrix_x4(dsa + swz(QHALF, bh8, bc), o0, o1, o2, o3);
      mma_bf16_16816(sacc[0], k0, k1, k2, k3, q0, q1);
      mma_bf16_16816(sacc[1], k0, k1, k2, k3, q2, q3);
      mma_bf16_16816(pacc[0], v0, v1, v2, v3, o0, o1);
      mma_bf16_16816(pacc[1], v0, v1, v2, v3, o2, o3);
    }
    // P^T and dS^T (rows: keys 16w + r, + 8; columns: heads 8 nt + 2q + {0, 1})
    uint32_t pa[4], sa[4];
    if (key0 + 16 * warp + 15 <= last) {  // all of this warp's keys visible: packed fp32 pairs
      const unsigned long long sl2x2 = pack_f32x2(p.sl2, p.sl2);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int h0 = 8 * nt + 2 * q;
        const unsigned long long nl = pack_f32x2(-lse2_s[bf][h0], -lse2_s[bf][h0 + 1]);
        const unsigned long long nd = pack_f32x2(-dsum_s[bf][h0], -dsum_s[bf][h0 + 1]);
        float x0, x1, x2, x3;
        unpack_f32x2(fma_f32x2(pack_f32x2(sacc[nt][0], sacc[nt][1]), sl2x2, nl), x0, x1);
        unpack_f32x2(fma_f32x2(pack_f32x2(sacc[nt][2], sacc[nt][3]), sl2x2, nl), x2, x3);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2), p3 = fast_exp2(x3);
        float d0, d1, d2, d3;
        unpack_f32x2(mul_f32x2(pack_f32x2(p0, p1), add_f32x2(pack_f32x2(pacc[nt][0], pacc[nt][1]), nd)), d0, d1);
        unpack_f32x2(mul_f32x2(pack_f32x2(p2, p3), add_f32x2(pack_f32x2(pacc[nt][2], pacc[nt][3]), nd)), d2, d3);
        pa[nt ? 2 : 0] = pack_bf16x2(p0, p1);
        pa[nt ? 3 : 1] = pack_bf16x2(p2, p3);
        sa[nt ? 2 : 0] = pack_bf16x2(d0, d1);
        sa[nt ? 3 : 1] = pack_bf16x2(d2, d3);
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float pv[4], dsv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int key = key0 + 16 * warp + r + 8 * (u >> 1);
          const int h = 8 * nt + 2 * q + (u & 1);
          const float pr = key <= last ? fast_exp2(fmaf(sacc[nt][u], p.sl2, -lse2_s[bf][h])) : 0.f;
          pv[u] = pr;
          dsv[u] = pr * (pacc[nt][u] - dsum_s[bf][h]);
        }
        pa[nt ? 2 : 0] = pack_bf16x2(pv[0], pv[1]);
        pa[nt ? 3 : 1] = pack_bf16x2(pv[2], pv[3]);
        sa[nt ? 2 : 0] = pack_bf16x2(dsv[0], dsv[1]);
        sa[nt ? 3 : 1] = pack_bf16x2(dsv[2], dsv[3]);
      }
    }
    // dV_w += P^T dO and dK_w += dS^T Q (B fragments by ldmatrix.trans: k = head, n = d)
#pragma unroll
    for (int np = 0; np < NDT / 2; ++np) {
      const int h = 8 * ((lane >> 3) & 1) + (lane & 7);
      const int c = 2 * np + (lane >> 4);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(dsa + swz(QHALF, h, c), b0, b1, b2, b3);
      mma_bf16_16816(dv[2 * np], pa[0], pa[1], pa[2], pa[3], b0, b1);
      mma_bf16_16816(dv[2 * np + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
      ldmatrix_x4_trans(qsa + swz(QHALF, h, c), b0, b1, b2, b3);
      mma_bf16_16816(dk[2 * np], sa[0], sa[1], sa[2], sa[3], b0, b1);
      mma_bf16_16816(dk[2 * np + 1], sa[0], sa[1], sa[2], sa[3], b2, b3);
    }
    __syncthreads();  // the buffer is restaged KV_NBUF - 1 queries later
  }
  cp_async_wait_all();
  // add this chunk's contribution (keys past N carry none)
  float* dKg = p.dK + ((size_t)bh * p.N_cap) * D;
  float* dVg = p.dV + ((size_t)bh * p.N_cap) * D;
#pragma unroll
  for (int u2 = 0; u2 < 2; ++u2) {
    const int key = key0 + 16 * warp + r + 8 * u2;
    if (key >= p.N) continue;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = 8 * i + 2 * q;
      red_add(dKg + (size_t)key * D + col, dk[i][2 * u2] * p.scale);
      red_add(dKg + (size_t)key * D + col + 1, dk[i][2 * u2 + 1] * p.scale);
      red_add(dVg + (size_t)key * D + col, dv[i][2 * u2]);
      red_add(dVg + (size_t)key * D + col + 1, dv[i][2 * u2 + 1]);
    }
  }
}

// (4') dK, dV on tcgen05 (d = 128, G_Q of 8 or 16).  Persistent CTAs take the chunks with a
// stride.  Per chunk: the block's K and V by TMA; per tile of 128 query-head rows (the next
// 128 / G_Q queries of the chunk, their Q rows and their dO rows by one 4-D TMA box each, on
// separate barriers so that S starts on the Q rows while the dO rows land):
//   S = Q K^T, dP = dO V^T       M 128 rows x N 64 keys x K = d, fp32 in TMEM
//   epilogue (one row a thread): P = exp2(S sl2 - LSE2), dS = P (dP - D), written as bf16 rows
//     of 64 keys to shared memory (keys past t or N, and rows of absent queries, 0)
//   dK^T += Q^T dS, dV^T += dO^T P   M 128 (d) x N 64 keys x K = rows: the Q / dO tile read
//     as a d-major A operand and dS / P as a key-major B operand (both MN-major); dK^T first,
//     so that the stage's Q rows are free for the next tile before its dO rows
// After the chunk's last tile, TMEM lane = d, dV^T is added into dV and scale x dK^T into dK.
// Roles: a producer warp (TMA), one thread issuing every tile's S and dP, another issuing the
// dK and dV products, and two epilogue groups of eight warps taking alternate tiles (two warps
// a TMEM lane quarter, 32 keys each), so that one tile's S and dP run on the tensor pipe while
// the other group turns the previous tile's into P and dS.  Stages are double-buffered (Q/dO
// tiles, S/dP accumulators and P/dS tiles; stage = tile parity = epilogue group) and so are
// the dV/dK accumulators (set = chunk parity; the group of that parity adds a chunk's set into
// dV and dK while the other chunk's tiles go on).  Every wait is bounded.
namespace tcb {
constexpr int THREADS = 608;                    // warp 0 producer, warps 1-2 MMA issuers, 3-18 epilogue
constexpr int EPI_WARP0 = 3, EPI_GROUP_WARPS = 8;
constexpr int ROWS = 128, KEYS = 64;
constexpr uint32_t QT_BYTES = ROWS * 128 * 2;   // a Q or dO tile, 32 KB
constexpr uint32_t KV_BYTES = KEYS * 128 * 2;   // a K or V block, 16 KB
constexpr uint32_t PS_BYTES = ROWS * KEYS * 2;  // a P or dS tile, 16 KB
constexpr size_t SMEM = 4 * QT_BYTES + 2 * KV_BYTES + 4 * PS_BYTES + 1024;
// TMEM columns: S of stage b at 128 b, dP at 128 b + 64; dV^T of set a at 256 + 128 a, dK^T 64 further
constexpr uint32_t COL_ACC = 256;
}  // namespace tcb

__global__ void __launch_bounds__(tcb::THREADS, 1) bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                     const __grid_constant__ CUtensorMap mapO,
                                                                     const __grid_constant__ CUtensorMap mapK,
                                                                     const __grid_constant__ CUtensorMap mapV,
                                                                     BwdParams p, uint32_t* err) {
  pdl_trigger();
  pdl_wait();  // the kernel before on the stream has completed
  using namespace tcb;
  constexpr int D = 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;                        // stage st: Q at 2 st, dO at 2 st + 1 (QT_BYTES each)
  uint8_t* sK = smem + 4 * QT_BYTES;
  uint8_t* sV = sK + KV_BYTES;
  uint8_t* sP = sV + KV_BYTES;               // stage st: P at 2 st, dS at 2 st + 1 (PS_BYTES each)
  // q_full / o_full[st]: the stage's Q / dO rows landed; q_empty / o_empty[st]: no longer read
  __shared__ uint64_t kv_full, kv_empty, q_full[2], o_full[2], q_empty[2], o_empty[2], s_full[2], s_empty[2],
      p_full[2], p_empty[2], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunks = *p.nchunks;
  const int RPQ = p.GQ, QPT = ROWS / p.GQ;  // rows per query, queries per tile

  // stale rows of a partial tile must be finite: zero both Q/dO stages once
  for (uint32_t i = threadIdx.x; i < 4 * QT_BYTES / 16; i += THREADS)
    reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    mbar_init(&drain, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], EPI_GROUP_WARPS);
      mbar_init(&p_full[i], EPI_GROUP_WARPS);
      mbar_init(&p_empty[i], p.dS ? 2 : 1);  // the dK/dV products done (and the dS tile copied out)
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], EPI_GROUP_WARPS);
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    bool failed = false;
    uint32_t tt = 0, cc = 0;
    for (int ci = blockIdx.x; ci < nchunks && !failed; ci += gridDim.x, ++cc) {
      const int4 ch = p.chunks[ci];
      const int bh = ch.x, blk = ch.y, first = ch.z, cnt = ch.w;
      const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
      if (!mbar_wait_warp(&kv_empty, (cc & 1) ^ 1, err)) {
        failed = true;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&kv_full, 2 * KV_BYTES);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_load_3d(sK + h * (KEYS * 128), &mapK, &kv_full, 64 * h, blk * KEYS, bh);
          tma_load_3d(sV + h * (KEYS * 128), &mapV, &kv_full, 64 * h, blk * KEYS, bh);
        }
        if (ci + (int)gridDim.x < nchunks) {  // the next chunk's block towards L2
          const int4 nx = p.chunks[ci + gridDim.x];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_prefetch_3d(&mapK, 64 * h, nx.y * KEYS, nx.x);
            tma_prefetch_3d(&mapV, 64 * h, nx.y * KEYS, nx.x);
          }
        }
      }
      // lane l's query of the tile starting at entry kk (-1 past the chunk); a tile's queries
      // are read two tiles ahead, when its rows are prefetched towards L2
      auto entry = [&](int kk) -> int {
        return (kk < cnt && lane < min(QPT, cnt - kk)) ? p.entries[first + kk + lane] >> 5 : -1;
      };
      auto q_row = [&](int t) -> int { return (int)((((long long)b * p.N + t) * p.H_q + (long long)hk * p.GQ) >> 3); };
      auto prefetch_rows = [&](int t) {
        if (t >= 0) {
          tma_prefetch_4d(&mapQ, 0, 0, 0, q_row(t));
          tma_prefetch_4d(&mapO, 0, 0, 0, q_row(t));
        }
      };
      int t_cur = entry(0), t_next = entry(QPT);
      prefetch_rows(t_cur);
      prefetch_rows(t_next);
      for (int k0 = 0; k0 < cnt; k0 += QPT, ++tt) {
        const int st = tt & 1;
        const int t_after = entry(k0 + 2 * QPT);  // in flight while the stage frees
        const int nq = min(QPT, cnt - k0);
        // the Q rows as soon as the previous tile's dK products are done (S starts on them),
        // the dO rows once its dV products are
        if (!mbar_wait_warp(&q_empty[st], ((tt >> 1) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&q_full[st], (uint32_t)nq * RPQ * 256);
        __syncwarp();
        if (lane < nq) tma_load_4d(sQ + (2 * st) * QT_BYTES + lane * RPQ * 256, &mapQ, &q_full[st], 0, 0, 0, q_row(t_cur));
        if (!mbar_wait_warp(&o_empty[st], ((tt >> 1) & 1) ^ 1, err)) {
          if (lane == 0) mbar_wait(&q_full[st], (tt >> 1) & 1, err, 100000000ull);  // this tile's Q rows
          failed = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&o_full[st], (uint32_t)nq * RPQ * 256);
        __syncwarp();
        if (lane < nq) tma_load_4d(sQ + (2 * st + 1) * QT_BYTES + lane * RPQ * 256, &mapO, &o_full[st], 0, 0, 0, q_row(t_cur));
        prefetch_rows(t_after);
        t_cur = t_next;
        t_next = t_after;
      }
    }
    // after a timeout, copies still in flight land before shared memory goes away (bounded)
    if (failed && lane == 0) {
      if (cc > 0) mbar_wait(&kv_full, (cc - 1) & 1, err, 100000000ull);
      for (uint32_t u = tt > 2 ? tt - 2 : 0; u < tt; ++u) {
        mbar_wait(&q_full[u & 1], (u >> 1) & 1, err, 100000000ull);
        mbar_wait(&o_full[u & 1], (u >> 1) & 1, err, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------- MMA issuer: S = Q K^T and dP = dO V^T -------------------
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(ROWS, KEYS);
      uint32_t tt = 0, cc = 0;
      bool failed = false;
      for (int ci = blockIdx.x; ci < nchunks && !failed; ci += gridDim.x, ++cc) {
        const int cnt = p.chunks[ci].w;
        if (!mbar_wait(&kv_full, cc & 1, err)) {
          failed = true;
          break;
        }
        const uint32_t kb = smem_u32(sK), vb = smem_u32(sV);
        for (int k0 = 0; k0 < cnt; k0 += QPT, ++tt) {
          const int st = tt & 1;
          if (!mbar_wait(&q_full[st], (tt >> 1) & 1, err) || !mbar_wait(&s_empty[st], ((tt >> 1) & 1) ^ 1, err)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t qb = smem_u32(sQ + (2 * st) * QT_BYTES), ob = smem_u32(sQ + (2 * st + 1) * QT_BYTES);
          // K = d; grouped rows: d half h of 8-row group g at g 2048 + h 1024
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            umma_bf16(tmem_base + st * 128, smem_desc_sw128(qb + (s >> 2) * 1024 + (s & 3) * 32, 16, 2048),
                      smem_desc_sw128(kb + (s >> 2) * (KEYS * 128) + (s & 3) * 32, 16, 1024), id_kk, s > 0 ? 1u : 0u);
          if (!mbar_wait(&o_full[st], (tt >> 1) & 1, err)) {
            failed = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            umma_bf16(tmem_base + st * 128 + 64, smem_desc_sw128(ob + (s >> 2) * 1024 + (s & 3) * 32, 16, 2048),
                      smem_desc_sw128(vb + (s >> 2) * (KEYS * 128) + (s & 3) * 32, 16, 1024), id_kk, s > 0 ? 1u : 0u);
          umma_commit(&s_full[st]);
          if (k0 + QPT >= cnt) umma_commit(&kv_empty);  // the block's K and V are no longer read
        }
      }
      // every MMA issued has completed before the tensor memory is released (bounded)
      umma_commit(&drain);
      mbar_wait(&drain, 0, err);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------ MMA issuer: dV^T += dO^T P and dK^T += Q^T dS ------------------
    if (lane == 0) {
      constexpr uint32_t id_mn = idesc_bf16_f32(ROWS, KEYS) | (1u << 15) | (1u << 16);  // A and B MN-major
      uint32_t tt = 0, cc = 0;
      bool failed = false;
      for (int ci = blockIdx.x; ci < nchunks && !failed; ci += gridDim.x, ++cc) {
        const int first = p.chunks[ci].z, cnt = p.chunks[ci].w;
        const int a = cc & 1;
        const uint32_t col = tmem_base + COL_ACC + 128 * a;
        for (int k0 = 0; k0 < cnt; k0 += QPT, ++tt) {
          const int st = tt & 1;
          if (!mbar_wait(&p_full[st], (tt >> 1) & 1, err) ||
              (k0 == 0 && !mbar_wait(&acc_empty[a], ((cc >> 1) & 1) ^ 1, err))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t qb = smem_u32(sQ + (2 * st) * QT_BYTES), ob = smem_u32(sQ + (2 * st + 1) * QT_BYTES);
          const uint32_t pb = smem_u32(sP + (2 * st) * PS_BYTES), db = smem_u32(sP + (2 * st + 1) * PS_BYTES);
          // K = rows: 16 rows = two 8-row groups per step; dK^T first, so that the Q rows free early
#pragma unroll
          for (int s = 0; s < ROWS / 16; ++s)
            umma_bf16(col + 64, smem_desc_sw128(qb + s * 4096, 1024, 2048), smem_desc_sw128(db + s * 2048, 8192, 1024),
                      id_mn, (k0 == 0 && s == 0) ? 0u : 1u);
          umma_commit(&q_empty[st]);
#pragma unroll
          for (int s = 0; s < ROWS / 16; ++s)
            umma_bf16(col, smem_desc_sw128(ob + s * 4096, 1024, 2048), smem_desc_sw128(pb + s * 2048, 8192, 1024), id_mn,
                      (k0 == 0 && s == 0) ? 0u : 1u);
          umma_commit(&o_empty[st]);
          umma_commit(&p_empty[st]);
          if (p.dS) {  // the tile's dS rows (the first nq queries' rows, in the entries' order) out
            const int nq = min(QPT, cnt - k0);
            bulk_store(p.dS + (size_t)(first + k0) * (size_t)(RPQ * 64), sP + (2 * st + 1) * PS_BYTES,
                       (uint32_t)(nq * RPQ * 128));
            bulk_commit();
            bulk_wait_read();
            mbar_arrive(&p_empty[st]);
          }
          if (k0 + QPT >= cnt) umma_commit(&acc_full[a]);
        }
      }
      bulk_wait();  // the dS tiles are in global memory
      umma_commit(&drain);
      mbar_wait(&drain, 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int g = (warp - EPI_WARP0) / EPI_GROUP_WARPS;  // group: the tiles (and the stage) of parity g
    const int kh = ((warp - EPI_WARP0) % EPI_GROUP_WARPS) >> 2;  // keys 32 kh .. 32 kh + 31 of the block
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;       // TMEM lane: query-head row for S / dP, d for dV^T / dK^T
    const int qi = row / RPQ, h = row - qi * RPQ;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const int st = g;
    uint32_t tt = 0, cc = 0;
    bool failed = false;
    for (int ci = blockIdx.x; ci < nchunks && !failed; ci += gridDim.x, ++cc) {
      const int4 ch = p.chunks[ci];
      const int bh = ch.x, blk = ch.y, first = ch.z, cnt = ch.w;
      const int b = bh / p.H_kv, hk = bh - b * p.H_kv;
      const int key0 = blk * KEYS;
      for (int k0 = 0; k0 < cnt; k0 += QPT, ++tt) {
        if ((int)(tt & 1) != g) continue;
        const bool vq = k0 + qi < cnt;
        const int t = vq ? p.entries[first + k0 + qi] >> 5 : 0;
        float lse2 = POS_INF, dsum = 0.f;
        if (vq) {
          const size_t li = ((size_t)b * p.H_q + (size_t)hk * p.GQ + h) * p.N + t;
          const float l = p.LSE[li];
          lse2 = l == NEG_INF ? POS_INF : l * LOG2E;
          dsum = p.Dsum[li];
        }
        const int last = vq ? (p.causal ? min(t, p.N - 1) : p.N - 1) - key0 : -1;  // visible keys j <= last
        if (!mbar_wait_warp(&s_full[st], (tt >> 1) & 1, err)) {
          failed = true;
          break;
        }
        tc_fence_after();
        // P and dS go to this stage's tiles once the previous tile of the stage has been consumed
        if (!mbar_wait_warp(&p_empty[st], ((tt >> 1) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        uint8_t* prow = sP + (2 * st) * PS_BYTES + row * 128;
        uint8_t* drow = sP + (2 * st + 1) * PS_BYTES + row * 128;
        // this warp's 32 keys, 16 at a time: S and dP in one round trip, then P and dS = P (dP - D)
        // as bf16 into two 16-byte chunks of each row (128-byte swizzle)
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const int j0 = 32 * kh + 16 * hf;  // first key of the step
          uint32_t sr[16], dr[16];
          tmem_ld16(lane_base + st * 128 + j0, sr);
          tmem_ld16(lane_base + st * 128 + 64 + j0, dr);
          tmem_wait_ld();
          if (hf == 1) {  // S and dP are read out: the MMA may reuse this buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[st]);
          }
          uint32_t pk[8], dk2[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float p0 = (j0 + j <= last) ? fast_exp2(fmaf(__uint_as_float(sr[j]), p.sl2, -lse2)) : 0.f;
            const float p1 = (j0 + j + 1 <= last) ? fast_exp2(fmaf(__uint_as_float(sr[j + 1]), p.sl2, -lse2)) : 0.f;
            pk[j / 2] = pack_bf16x2(p0, p1);
            dk2[j / 2] = pack_bf16x2(p0 * (__uint_as_float(dr[j]) - dsum), p1 * (__uint_as_float(dr[j + 1]) - dsum));
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {  // 16-byte chunk j0 / 8 + c of the row
            const uint32_t off = (uint32_t)(((j0 / 8 + c) ^ (row & 7)) << 4);
            *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            *reinterpret_cast<uint4*>(drow + off) = make_uint4(dk2[4 * c], dk2[4 * c + 1], dk2[4 * c + 2], dk2[4 * c + 3]);
          }
        }
        fence_proxy_async();  // the MMA reads the tiles through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[st]);
      }
      if (failed) break;
      if ((int)(cc & 1) != g) continue;
      // the chunk's dV^T and dK^T (lane = d): add into dV and scale x dK (keys past N carry none)
      if (!mbar_wait_warp(&acc_full[g], (cc >> 1) & 1, err)) {
        failed = true;
        break;
      }
      tc_fence_after();
      float* dKg = p.dK + ((size_t)bh * p.N_cap) * D;
      float* dVg = p.dV + ((size_t)bh * p.N_cap) * D;
      const uint32_t col = lane_base + COL_ACC + 128 * g;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {  // this warp's 32 keys, 16 at a time
        const int j0 = 32 * kh + 16 * c;
        uint32_t vr[16], kr[16];
        tmem_ld16(col + j0, vr);
        tmem_ld16(col + 64 + j0, kr);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int key = key0 + j0 + j;
          if (key < p.N) {
            red_add(dVg + (size_t)key * D + row, __uint_as_float(vr[j]));
            red_add(dKg + (size_t)key * D + row, __uint_as_float(kr[j]) * p.scale);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[g]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

cudaError_t launch_dkv_tc(BwdParams& p, long long max_chunks, int num_sms, uint32_t* err, cudaStream_t s) {
  constexpr int D = 128;
  CUtensorMap mapQ, mapO, mapK, mapV;
  const long long rows = (long long)p.B * p.N * p.H_q;
  {
    // one box per query: (64 columns, 8 rows, 2 d halves, G_Q / 8 row groups), lands as
    // [row group][half][8 rows][64]
    const uint64_t dims[4] = {64, 8, 2, (uint64_t)(rows / 8)};
    const uint64_t strides[3] = {(uint64_t)D * 2, 128, (uint64_t)8 * D * 2};
    const uint32_t box[4] = {64, 8, 2, (uint32_t)(p.GQ / 8)};
    if (!encode_tensor_map(&mapQ, p.Q, 4, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_tensor_map(&mapO, p.dO, 4, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.N, (uint64_t)p.B * p.H_kv};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.N_cap * D * 2};
    const uint32_t box[3] = {64, (uint32_t)tcb::KEYS, 1};
    if (!encode_tensor_map(&mapK, p.K, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!encode_tensor_map(&mapV, p.V, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcb::SMEM);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, bwd_dkv_tc_kernel)) != cudaSuccess) return e;
  if (fa.maxThreadsPerBlock < tcb::THREADS) return cudaErrorLaunchOutOfResources;  // registers x threads
  const int grid = (int)std::min<long long>(max_chunks, (long long)num_sms);
  if (grid > 0)
    return launch_pdl(bwd_dkv_tc_kernel, dim3(grid), dim3(tcb::THREADS), tcb::SMEM, s, mapQ, mapO, mapK, mapV, p, err);
  return cudaSuccess;
}

template <int D>
cudaError_t launch_d(BwdParams& p, int nkeys, int32_t* chunk_off, long long max_chunks, int num_sms, uint32_t* err,
                     cudaStream_t s) {
  cudaError_t e;
  const long long rows = (long long)p.B * p.N * p.H_q;
  const long long ents = (long long)p.B * p.H_kv * p.N * p.Ksel;
  const int g1 = (int)std::min<long long>((rows * (D / 8) + 255) / 256, (long long)num_sms * 32);
  const int g2 = (int)std::min<long long>((ents + 255) / 256, (long long)num_sms * 16);
  // after the first, every kernel is a programmatic dependent of the one before (each waits for
  // it to complete before its first access)
  bwd_dsum_kernel<D><<<g1 > 0 ? g1 : 1, 256, 0, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_count_kernel, dim3(g2 > 0 ? g2 : 1), dim3(256), 0, s, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_scan_kernel, dim3(1), dim3(1024), 0, s, p, nkeys, chunk_off)) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_scatter_kernel, dim3(g2 > 0 ? g2 : 1), dim3(256), 0, s, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_chunks_kernel, dim3((nkeys + 255) / 256), dim3(256), 0, s, p, nkeys, chunk_off)) != cudaSuccess)
    return e;
  // lists by position, chunks by their first position
  if ((e = cudaFuncSetAttribute(bwd_sort_lists_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(SORT_CAP * sizeof(int32_t)))) != cudaSuccess)
    return e;
  if (nkeys > 0 &&
      (e = launch_pdl(bwd_sort_lists_kernel, dim3(nkeys), dim3(512), SORT_CAP * sizeof(int32_t), s, p)) != cudaSuccess)
    return e;
  const int gc = (int)std::min<long long>((max_chunks + 255) / 256, (long long)num_sms * 8);
  if ((e = launch_pdl(bwd_bucket_count_kernel, dim3(gc > 0 ? gc : 1), dim3(256), 0, s, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_bucket_scan_kernel, dim3(1), dim3(NBUCKETS), 0, s, p)) != cudaSuccess) return e;
  if ((e = launch_pdl(bwd_bucket_scatter_kernel, dim3(gc > 0 ? gc : 1), dim3(256), 0, s, p)) != cudaSuccess) return e;
  p.chunks = p.chunks_by_t;
  const long long items = (long long)p.B * p.H_kv * p.N;
  if (p.tc && (e = launch_dkv_tc(p, max_chunks, num_sms, err, s)) != cudaSuccess) return e;
  if (p.dS) {  // the tcgen05 dK/dV kernel wrote dS: dQ = scale dS K
    // K half blocks by TMA: dims (64 columns, rows, d half, b*h_kv), both d halves in one box
    CUtensorMap mapK;
    {
      const uint64_t dims[4] = {64, (uint64_t)p.N, 2, (uint64_t)p.B * p.H_kv};
      const uint64_t strides[3] = {128 * 2, 128, (uint64_t)p.N_cap * 128 * 2};
      const uint32_t box[4] = {64, (uint32_t)HK, 2, 1};
      if (!encode_tensor_map(&mapK, p.K, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const size_t smem_ds = (size_t)DQS_WARPS * DQS_SLOTS * (HK * 128 * 2 + 16 * 128) + 1024;
    if ((e = cudaFuncSetAttribute(bwd_dq_ds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_ds)) !=
        cudaSuccess)
      return e;
    const long long gds = std::min<long long>((items + DQS_WARPS - 1) / DQS_WARPS, (long long)num_sms);
    return launch_pdl(bwd_dq_ds_kernel, dim3((unsigned)gds), dim3(32 * DQS_WARPS), smem_ds, s, mapK, p, err);
  }
  const size_t smem_q = (size_t)DQ_WARPS * 2 * HK * D * 2 + 1024;
  if ((e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q)) != cudaSuccess)
    return e;
  const long long gq = std::min<long long>((items + DQ_WARPS - 1) / DQ_WARPS, (long long)num_sms);
  if ((e = launch_pdl(bwd_dq_kernel<D>, dim3((unsigned)gq), dim3(32 * DQ_WARPS), smem_q, s, p)) != cudaSuccess) return e;
  if (p.tc) return cudaSuccess;
  const size_t smem_kv = (size_t)2 * 64 * D * 2 + (size_t)2 * KV_NBUF * 16 * D * 2 + 1024;
  if ((e = cudaFuncSetAttribute(bwd_dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv)) !=
      cudaSuccess)
    return e;
  if (max_chunks > 0 &&
      (e = launch_pdl(bwd_dkv_kernel<D>, dim3((unsigned)max_chunks), dim3(32 * KV_WARPS), smem_kv, s, p)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace

// dK and dV on tcgen05 (and dQ from the dS rows it writes) for d = 128 and G_Q of 8 or 16
bool bwd_tc_path(const Problem& p) { return p.d == 128 && (p.GQ == 8 || p.GQ == 16) && p.H_q % 8 == 0; }

// dS of every (query, block) pair, written by the tcgen05 dK/dV kernel for the dQ kernel, up to
// 64 GB of scratch; above that the dQ kernel forms S and dP again instead
constexpr size_t DS_MAX_BYTES = (size_t)1 << 36;
size_t bwd_ds_bytes(const Problem& p) {
  const size_t b = (size_t)p.B * p.H_kv * p.N * p.K * p.GQ * 64 * 2;
  return bwd_tc_path(p) && b <= DS_MAX_BYTES ? b : 0;
}

size_t attn_backward_workspace_bytes(const Problem& p, bool with_ds) {
  const size_t ds = with_ds ? bwd_ds_bytes(p) : 0;
  const long long M1 = (p.N + 63) / 64;
  const long long nkeys = (long long)p.B * p.H_kv * M1;
  const long long ents = (long long)p.B * p.H_kv * p.N * p.K;
  const long long max_chunks = nkeys + ents / QC + 1;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return up((size_t)p.B * p.H_q * p.N * 4) + 3 * up((size_t)(nkeys + 1) * 4) + 2 * up((size_t)ents * 4) +
         up((size_t)max_chunks * 16) + up(4) + up(ds) + up((size_t)max_chunks * 16) + 3 * up((size_t)NBUCKETS * 4) +
         (ds ? up((size_t)ents * 4) : 0);
}

cudaError_t launch_attn_backward(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                 const uint16_t* O, const float* LSE, const uint16_t* dO, float* dQ, float* dK,
                                 float* dV, void* ws, bool with_ds, const Problem& pr, int num_sms, uint32_t* err,
                                 cudaStream_t s) {
  BwdParams p;
  p.Q = Q;
  p.K = K;
  p.V = V;
  p.O = O;
  p.dO = dO;
  p.idx = idx;
  p.LSE = LSE;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.B = pr.B;
  p.N = pr.N;
  p.N_cap = pr.N_cap;
  p.H_q = pr.H_q;
  p.H_kv = pr.H_kv;
  p.GQ = pr.GQ;
  p.Ksel = pr.K;
  p.M1 = (pr.N + 63) / 64;
  p.causal = pr.causal;
  p.scale = pr.scale;
  p.sl2 = pr.scale * LOG2E;
  const long long nkeys = (long long)pr.B * pr.H_kv * p.M1;
  const long long ents = (long long)pr.B * pr.H_kv * pr.N * pr.K;
  const long long max_chunks = nkeys + ents / QC + 1;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.Dsum = reinterpret_cast<float*>(w);
  w += up((size_t)pr.B * pr.H_q * pr.N * 4);
  p.counts = reinterpret_cast<int32_t*>(w);
  w += up((size_t)(nkeys + 1) * 4);
  p.rank = reinterpret_cast<int32_t*>(w);
  w += up((size_t)ents * 4);
  p.offsets = reinterpret_cast<int32_t*>(w);
  w += up((size_t)(nkeys + 1) * 4);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(w);
  w += up((size_t)(nkeys + 1) * 4);
  p.entries = reinterpret_cast<int32_t*>(w);
  w += up((size_t)ents * 4);
  p.chunks = reinterpret_cast<int4*>(w);
  w += up((size_t)max_chunks * 16);
  p.nchunks = reinterpret_cast<int32_t*>(w);
  w += up(4);
  p.tc = bwd_tc_path(pr) ? 1 : 0;
  const size_t ds = with_ds ? bwd_ds_bytes(pr) : 0;
  p.dS = ds ? reinterpret_cast<uint16_t*>(w) : nullptr;
  w += up(ds);
  p.chunks_by_t = reinterpret_cast<int4*>(w);
  w += up((size_t)max_chunks * 16);
  p.bucket_count = reinterpret_cast<int32_t*>(w);
  w += up((size_t)NBUCKETS * 4);
  p.bucket_start = reinterpret_cast<int32_t*>(w);
  w += up((size_t)NBUCKETS * 4);
  p.bucket_cursor = reinterpret_cast<int32_t*>(w);
  w += up((size_t)NBUCKETS * 4);
  p.epos = p.dS ? reinterpret_cast<int32_t*>(w) : nullptr;
  p.bucket_shift = 0;
  while ((((long long)pr.N - 1) >> p.bucket_shift) >= NBUCKETS) ++p.bucket_shift;
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.counts, 0, (size_t)(nkeys + 1) * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.bucket_count, 0, (size_t)NBUCKETS * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.bucket_cursor, 0, (size_t)NBUCKETS * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dK, 0, (size_t)pr.B * pr.H_kv * pr.N_cap * pr.d * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dV, 0, (size_t)pr.B * pr.H_kv * pr.N_cap * pr.d * 4, s)) != cudaSuccess) return e;
  if (pr.d == 128) return launch_d<128>(p, (int)nkeys, chunk_off, max_chunks, num_sms, err, s);
  return launch_d<64>(p, (int)nkeys, chunk_off, max_chunks, num_sms, err, s);
}

}  // namespace pisa
