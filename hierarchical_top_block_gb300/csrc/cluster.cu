// Clustering for Stage 2 (summary page of "Block Sparse Attention with Log-Linear
// Complexity", section "Method step details", step 2: queries that must score the same
// leaf block are gathered and cut into Q tiles so that each key block is loaded once per
// tile).  Here the unit is a level-2 survivor (a pair of sibling leaves, 128 keys): every
// (query t, survivor slot i) becomes an entry in the list of key (b, h_kv, window, node).
// Windows of consecutive queries keep the Q rows a tile gathers resident in L2.
//
//   count   : histogram of entries per key (atomics; accumulated by the Stage 1 walk as it
//             writes each query's survivors, into counts zeroed before it; the value each
//             atomic returned is the entry's place k in its list, kept in cb.rank)
//   scan    : exclusive scans of counts and of ceil(count / qt) (three small kernels; the
//             second also zeroes Stage 2's tile counter)
//   scatter : entries[offset[key] + k] = (t << 6) | slot   (order within a key arbitrary)
//   tiles   : {bh, node, first entry, entry count <= qt} for every tile
//             (scatter and tiles are independent: one launch, split by block)
// Each kernel is launched as a programmatic dependent of the one before it on the stream.
// The order of entries inside a list does not change any result: each entry is scored
// on its own and written to its own (t, slot) location.
#include "kernels.cuh"
#include "pdl.cuh"

namespace pisa {
namespace {

constexpr int THREADS = 256;
constexpr int SCAN_THREADS = 1024;
constexpr int SCAN_PER_THREAD = 4;
constexpr int SCAN_CHUNK = SCAN_THREADS * SCAN_PER_THREAD;

__device__ __forceinline__ long long key_of(int bh, int t, int node, const ClusterBuffers& cb) {
  return ((long long)bh * cb.nwin + t / cb.win) * cb.M2 + node;
}

// block-local exclusive scan of (count, tiles) pairs; writes block totals
__device__ __forceinline__ int2 warp_incl_scan(int2 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, v.x, o), b = __shfl_up_sync(0xffffffffu, v.y, o);
    if (lane >= o) {
      v.x += a;
      v.y += b;
    }
  }
  return v;
}

__device__ int2 block_excl_scan(int2 v, int2* total) {
  __shared__ int2 warp_sums[SCAN_THREADS / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int2 inc = warp_incl_scan(v);
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int2 w = lane < SCAN_THREADS / 32 ? warp_sums[lane] : make_int2(0, 0);
    w = warp_incl_scan(w);
    if (lane < SCAN_THREADS / 32) warp_sums[lane] = w;
  }
  __syncthreads();
  int2 base = warp > 0 ? warp_sums[warp - 1] : make_int2(0, 0);
  *total = warp_sums[SCAN_THREADS / 32 - 1];
  __syncthreads();
  return make_int2(base.x + inc.x - v.x, base.y + inc.y - v.y);
}

__global__ void __launch_bounds__(SCAN_THREADS) scan_local_kernel(ClusterBuffers cb) {
  pdl_trigger();
  pdl_wait();
  const long long base = (long long)blockIdx.x * SCAN_CHUNK + (long long)threadIdx.x * SCAN_PER_THREAD;
  int2 vals[SCAN_PER_THREAD];
  int2 sum = make_int2(0, 0);
#pragma unroll
  for (int i = 0; i < SCAN_PER_THREAD; ++i) {
    const long long k = base + i;
    const int c = k < cb.nkeys ? cb.counts[k] : 0;
    vals[i] = make_int2(c, (c + cb.qt - 1) / cb.qt);
    sum.x += vals[i].x;
    sum.y += vals[i].y;
  }
  int2 tot;
  int2 off = block_excl_scan(sum, &tot);
#pragma unroll
  for (int i = 0; i < SCAN_PER_THREAD; ++i) {
    const long long k = base + i;
    if (k < cb.nkeys) {
      cb.offsets[k] = off.x;
      cb.tile_off[k] = off.y;
    }
    off.x += vals[i].x;
    off.y += vals[i].y;
  }
  if (threadIdx.x == 0) {
    cb.block_sums[2 * blockIdx.x] = tot.x;
    cb.block_sums[2 * blockIdx.x + 1] = tot.y;
  }
}

__global__ void __launch_bounds__(SCAN_THREADS) scan_blocks_kernel(ClusterBuffers cb) {
  pdl_trigger();
  pdl_wait();
  // single block: exclusive scan of the block totals in chunks, carrying the running sum
  int2 carry = make_int2(0, 0);
  for (int base = 0; base < cb.nblocks; base += SCAN_THREADS) {
    const int i = base + threadIdx.x;
    int2 v = i < cb.nblocks ? make_int2(cb.block_sums[2 * i], cb.block_sums[2 * i + 1]) : make_int2(0, 0);
    int2 tot;
    int2 ex = block_excl_scan(v, &tot);
    if (i < cb.nblocks) {
      cb.block_sums[2 * i] = ex.x + carry.x;
      cb.block_sums[2 * i + 1] = ex.y + carry.y;
    }
    carry.x += tot.x;
    carry.y += tot.y;
  }
  if (threadIdx.x == 0) {
    cb.totals[0] = carry.x;
    cb.totals[1] = carry.y;
    cb.totals[2] = 0;  // Stage 2's tile counter
    cb.totals[3] = 0;
  }
}

__global__ void __launch_bounds__(SCAN_THREADS) scan_add_kernel(ClusterBuffers cb) {
  pdl_trigger();
  pdl_wait();
  const int bx = blockIdx.x;
  const int ax = cb.block_sums[2 * bx], ay = cb.block_sums[2 * bx + 1];
  const long long base = (long long)bx * SCAN_CHUNK;
  for (int i = threadIdx.x; i < SCAN_CHUNK; i += SCAN_THREADS) {
    const long long k = base + i;
    if (k < cb.nkeys) {
      cb.offsets[k] += ax;
      cb.tile_off[k] += ay;
    }
  }
}

// blocks [0, nb_scatter) place the entries, the others write the tile list
__global__ void scatter_tiles_kernel(const int32_t* __restrict__ S2, ClusterBuffers cb, int N, int t_lo, int nq, int Ksel,
                                     long long total, int nb_scatter) {
  pdl_trigger();
  pdl_wait();
  if ((int)blockIdx.x >= nb_scatter) {
    // a warp takes 32 keys at a time (one per lane) and writes the tiles of each of them with all
    // its lanes, so a key that many queries of a window selected (hundreds of tiles) costs no
    // more than a few stores per lane
    const int lane = threadIdx.x & 31;
    const long long nw = ((long long)gridDim.x - nb_scatter) * (blockDim.x / 32);
    const long long gw = ((long long)blockIdx.x - nb_scatter) * (blockDim.x / 32) + (threadIdx.x >> 5);
    for (long long k0 = gw * 32; k0 < cb.nkeys; k0 += nw * 32) {
      const long long k = k0 + lane;
      const int n = k < cb.nkeys ? cb.counts[k] : 0;
      const int e0 = n ? cb.offsets[k] : 0, t0 = n ? cb.tile_off[k] : 0;
      unsigned busy = __ballot_sync(0xffffffffu, n > 0);
      while (busy) {
        const int j = __ffs(busy) - 1;
        busy &= busy - 1;
        const int nj = __shfl_sync(0xffffffffu, n, j), ej = __shfl_sync(0xffffffffu, e0, j);
        const int tj = __shfl_sync(0xffffffffu, t0, j);
        const long long kj = k0 + j;
        const int node = (int)(kj % cb.M2);
        const int bh = (int)(kj / ((long long)cb.nwin * cb.M2));
        for (int i = lane; i * cb.qt < nj; i += 32) {
          const int s = i * cb.qt;
          cb.tiles[tj + i] = make_int4(bh, node, ej + s, min(cb.qt, nj - s));
        }
      }
    }
    return;
  }
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total * Ksel;
       e += (long long)nb_scatter * blockDim.x) {
    const long long item = e / Ksel;
    const int slot = (int)(e - item * Ksel);
    const int bh = (int)(item / nq), t = t_lo + (int)(item % nq);
    const int node = S2[((long long)bh * N + t) * Ksel + slot];
    if (node < 0) continue;
    const long long key = key_of(bh, t, node, cb);
    const int pos = cb.offsets[key] + cb.rank[((long long)bh * N + t) * (2 * Ksel) + slot];
    cb.entries[pos] = (t << 6) | slot;
  }
}

inline int grid_for(long long work, int threads, int cap = 4096) {
  long long b = (work + threads - 1) / threads;
  if (b < 1) b = 1;
  return (int)(b < cap ? b : cap);
}

}  // namespace

cudaError_t launch_cluster(const int32_t* S2, const ClusterBuffers& cb, const Problem& p, cudaStream_t s) {
  const int nq = p.t_hi - p.t_lo;
  const long long total = (long long)p.B * p.H_kv * (nq > 0 ? nq : 0);
  cudaError_t e;
  if ((e = launch_pdl(scan_local_kernel, dim3(cb.nblocks), dim3(SCAN_THREADS), 0, s, cb)) != cudaSuccess) return e;
  if ((e = launch_pdl(scan_blocks_kernel, dim3(1), dim3(SCAN_THREADS), 0, s, cb)) != cudaSuccess) return e;
  if ((e = launch_pdl(scan_add_kernel, dim3(cb.nblocks), dim3(SCAN_THREADS), 0, s, cb)) != cudaSuccess) return e;
  const int nb_scatter = grid_for(total * p.K, THREADS), nb_tiles = grid_for((cb.nkeys + 31) / 32, THREADS / 32);
  return launch_pdl(scatter_tiles_kernel, dim3(nb_scatter + nb_tiles), dim3(THREADS), 0, s, S2, cb, p.N, p.t_lo, nq,
                    p.K, total, nb_scatter);
}

}  // namespace pisa
