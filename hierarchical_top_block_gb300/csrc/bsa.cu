// BSA flat block selection, the single-level baseline the paper's selection-speed figure
// compares PISA with (summary page of "Block Sparse Attention with Log-Linear Complexity",
// section "Prerequisites": block sparse attention keeps K blocks per query, ranked by the
// dot product of the query with every block summary, q . kbar_j / sqrt(d), over all
// M = ceil(N / C) blocks; GQA: the G_Q heads of a group share one selection, their scores
// summed; section "Experimental results", item 5, Fig. 3).  The summaries are the level-1
// nodes of the mean-pooled pyramid (step 1); causal eligibility, the forced own block and the
// tie rule are those of the PISA selection.
//
// The score is linear in q, so the group's head sum folds into the query:
//   u_{t,j} = scale * sum_h q_{t,h} . kbar_j = scale * (sum_h q_{t,h}) . kbar_j.
// bsa_qsum_kernel sums the G_Q heads of every query in fp32 and splits the sum into two bf16
// parts hi + lo (hi = bf16(x), lo = bf16(x - hi); |x - hi - lo| <= 2^-18 |x|), so that the
// products run on the bf16 tensor cores with a score error far below the 1e-3 tie tolerance.
//
// bsa_select_kernel: persistent, warp-specialised, one CTA per SM.  A work tile is 128
// consecutive queries of one (b, h_kv), heaviest (latest) tiles first, handed out round-robin.
//   warp 0      TMA producer: the tile's query parts [2][128][d] into a 2-stage A ring, then
//               the 128-leaf summary tiles [128][d] of every block tile into a 2-stage B ring
//               (rows past the leaves belong to upper levels or read as zero; they are masked).
//   warp 1      owns TMEM (2 x 128 fp32 columns); one thread issues D = hi.B^T + lo.B^T
//               (M 128 queries x N 128 blocks x K 2d) per block tile and commits.
//   warps 2-5   epilogue: one TMEM lane (one query) per thread; each block tile's 128 scores
//               are compared with the running K-th best and the rare winners inserted into a
//               sorted list in registers (score desc, index asc); at the end the own block is
//               added and the set sorted ascending.
// Every wait is bounded; on timeout the error word is set, the MMAs and TMA loads still in
// flight are waited for (bounded) and the CTA returns.
#include "kernels.cuh"

namespace pisa {
namespace {

constexpr int BQ = 128;        // queries per tile (MMA M)
constexpr int BN = 128;        // leaf blocks per block tile (MMA N)
constexpr int NA = 2, NB = 2, NACC = 2;
constexpr int THREADS = 192;
constexpr int BIG = 0x7fffffff;

struct BsaParams {
  int32_t* idx;
  int BH, N, M1, Ksel, Kp, causal;  // Kp: ranked places (K - 1 with the forced own block)
  int ntq;                          // query tiles per (b, h_kv)
  long long ntiles;                 // BH * ntq
  long long nodes;                  // pyramid rows per (b, h_kv)
};

// ---- head sum ---------------------------------------------------------------------------
// One warp per (b, h_kv, t); lane l owns d values [E l, E l + E).  Qs: [BH][2][N][D] bf16.
template <int D>
__global__ void __launch_bounds__(256) bsa_qsum_kernel(const uint16_t* __restrict__ Q, uint16_t* __restrict__ Qs, int N,
                                                       int H_q, int H_kv, int GQ, long long total) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < total; it += nwarps) {
    const int bh = (int)(it / N), t = (int)(it - (long long)bh * N);
    const int b = bh / H_kv, hk = bh - b * H_kv;
    const uint16_t* q = Q + (((size_t)b * N + t) * H_q + (size_t)hk * GQ) * D + lane * E;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int h = 0; h < GQ; ++h) {  // heads in a fixed order
      if constexpr (E == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(q + (size_t)h * D);
        acc[0] += bf16_lo(v.x);
        acc[1] += bf16_hi(v.x);
        acc[2] += bf16_lo(v.y);
        acc[3] += bf16_hi(v.y);
      } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(q + (size_t)h * D);
        acc[0] += bf16_lo(v);
        acc[1] += bf16_hi(v);
      }
    }
    uint32_t hi[E / 2], lo[E / 2];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const uint16_t h0 = f32_to_bf16_rne(acc[e]), h1 = f32_to_bf16_rne(acc[e + 1]);
      hi[e / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
      lo[e / 2] = pack_bf16x2(acc[e] - bf16_to_f32(h0), acc[e + 1] - bf16_to_f32(h1));
    }
    uint16_t* o0 = Qs + (((size_t)bh * 2 + 0) * N + t) * D + lane * E;
    uint16_t* o1 = Qs + (((size_t)bh * 2 + 1) * N + t) * D + lane * E;
    if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(o0) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(o1) = make_uint2(lo[0], lo[1]);
    } else {
      *reinterpret_cast<uint32_t*>(o0) = hi[0];
      *reinterpret_cast<uint32_t*>(o1) = lo[0];
    }
  }
}

// ---- the scoring GEMM and the per-query top-K ------------------------------------------------
__device__ __forceinline__ void tile_of(const BsaParams& p, long long i, int& bh, int& t0, int& nbt) {
  const int qt = p.ntq - 1 - (int)(i / p.BH);  // latest (heaviest) query tiles first
  bh = (int)(i % p.BH);
  t0 = qt * BQ;
  int nblk = p.M1;
  if (p.causal) {
    const int last = min(t0 + BQ - 1, p.N - 1);
    nblk = min(p.M1, (last >> 6) + 1);
  }
  nbt = (nblk + BN - 1) / BN;
}

// Inserts (s, j) into the list sorted by (score desc, index asc), dropping the last entry.
// The list's last Kp slots hold the ranked blocks; the slots before them hold +inf sentinels
// that always rank first, so the K-th best is always the last slot.  Blocks arrive in
// ascending index order, so every listed block ranks above an equal score of the new one; the
// list shifts down by one from the insertion point with fixed indices only (each new entry i
// is chosen from the old entries i and i - 1), so it stays in registers.
template <int KM>
__device__ __forceinline__ void list_insert(float (&sv)[KM], int (&si)[KM], float s, int j) {
#pragma unroll
  for (int i = KM - 1; i >= 1; --i) {
    const bool stay = sv[i] >= s, prev_stay = sv[i - 1] >= s;
    const float ns = stay ? sv[i] : (prev_stay ? s : sv[i - 1]);
    const int ni = stay ? si[i] : (prev_stay ? j : si[i - 1]);
    sv[i] = ns;
    si[i] = ni;
  }
  if (!(sv[0] >= s)) {
    sv[0] = s;
    si[0] = j;
  }
}

template <int D, int KM>
__global__ void __launch_bounds__(THREADS, 1) bsa_select_kernel(const __grid_constant__ CUtensorMap mapA,
                                                                const __grid_constant__ CUtensorMap mapB, BsaParams p,
                                                                uint32_t* err) {
  constexpr int HALVES = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t PART_BYTES = BQ * D * 2;  // one bf16 part of the tile's queries
  constexpr uint32_t A_BYTES = 2 * PART_BYTES;
  constexpr uint32_t B_BYTES = BN * D * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + NA * A_BYTES;
  float* spill = reinterpret_cast<float*>(sB + NB * B_BYTES);  // [32][128] slow-path scores

  __shared__ uint64_t a_full[NA], a_empty[NA], b_full[NB], b_empty[NB], acc_full[NACC], acc_empty[NACC], drain;
  __shared__ uint32_t tmem_base_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(&drain, 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, NACC * BN);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      long long a_it = 0, b_it = 0;
      bool ok = true;
      for (long long i = blockIdx.x; i < p.ntiles && ok; i += gridDim.x) {
        int bh, t0, nbt;
        tile_of(p, i, bh, t0, nbt);
        const int as = (int)(a_it % NA);
        if (!mbar_wait(&a_empty[as], (uint32_t)((a_it / NA) & 1) ^ 1u, err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&a_full[as], A_BYTES);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            tma_load_2d(sA + as * A_BYTES + part * PART_BYTES + h * (BQ * 128), &mapA, &a_full[as], 64 * h,
                        (bh * 2 + part) * p.N + t0);
        ++a_it;
        for (int jt = 0; jt < nbt; ++jt) {
          const int bs = (int)(b_it % NB);
          if (!mbar_wait(&b_empty[bs], (uint32_t)((b_it / NB) & 1) ^ 1u, err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], B_BYTES);
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            tma_load_2d(sB + bs * B_BYTES + h * (BN * 128), &mapB, &b_full[bs], 64 * h,
                        (int)((long long)bh * p.nodes + (long long)jt * BN));
          ++b_it;
        }
      }
      // after a timeout, loads still in flight land before the CTA's shared memory goes away
      // (bounded): the latest load of each stage completes its barrier's current phase
      for (long long k = a_it - NA; !ok && k < a_it; ++k)
        if (k >= 0) mbar_wait(&a_full[k % NA], (uint32_t)((k / NA) & 1), err);
      for (long long k = b_it - NB; !ok && k < b_it; ++k)
        if (k >= 0) mbar_wait(&b_full[k % NB], (uint32_t)((k / NB) & 1), err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BQ, BN);
      long long a_it = 0, b_it = 0, acc_it = 0;
      bool ok = true;
      for (long long i = blockIdx.x; i < p.ntiles && ok; i += gridDim.x) {
        int bh, t0, nbt;
        tile_of(p, i, bh, t0, nbt);
        const int as = (int)(a_it % NA);
        if (!mbar_wait(&a_full[as], (uint32_t)((a_it / NA) & 1), err)) {
          ok = false;
          break;
        }
        for (int jt = 0; jt < nbt; ++jt) {
          const int bs = (int)(b_it % NB), ac = (int)(acc_it % NACC);
          if (!mbar_wait(&b_full[bs], (uint32_t)((b_it / NB) & 1), err) ||
              !mbar_wait(&acc_empty[ac], (uint32_t)((acc_it / NACC) & 1) ^ 1u, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t abase = smem_u32(sA + as * A_BYTES), bbase = smem_u32(sB + bs * B_BYTES);
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int s = 0; s < KSTEPS; ++s) {
              const uint32_t koff = (s >> 2) * (BQ * 128) + (s & 3) * 32;
              umma_bf16(tmem_base + ac * BN, smem_desc_sw128(abase + part * PART_BYTES + koff, 16, 1024),
                        smem_desc_sw128(bbase + koff, 16, 1024), idesc, (part | s) ? 1u : 0u);
            }
          umma_commit(&b_empty[bs]);
          umma_commit(&acc_full[ac]);
          ++b_it;
          ++acc_it;
        }
        if (!ok) break;
        umma_commit(&a_empty[as]);
        ++a_it;
      }
      // every MMA issued has completed before TMEM is released (bounded)
      umma_commit(&drain);
      mbar_wait(&drain, 0, err);
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    float* my_spill = spill + row;  // column k of this thread at my_spill[k * 128]
    long long acc_it = 0;
    bool ok = true;
    for (long long i = blockIdx.x; i < p.ntiles && ok; i += gridDim.x) {
      int bh, t0, nbt;
      tile_of(p, i, bh, t0, nbt);
      const int t = t0 + row;
      const bool valid = t < p.N;
      // a warp's 32 queries lie in one block of 64 keys, so the own block and the causal limit
      // are the same for all its lanes (lanes past N are never written)
      const int own = p.causal ? (t >> 6) : -1;
      const int jlim = p.causal ? min(p.M1, (t >> 6) + 1) : p.M1;
      float sv[KM];
      int si[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        const bool sentinel = k < KM - p.Kp;
        sv[k] = sentinel ? POS_INF : NEG_INF;
        si[k] = sentinel ? -1 : BIG;
      }
      float thr = sv[KM - 1];  // +inf when no place is ranked: nothing is inserted
      for (int jt = 0; jt < nbt; ++jt) {
        const int ac = (int)(acc_it % NACC);
        if (!mbar_wait_warp(&acc_full[ac], (uint32_t)((acc_it / NACC) & 1), err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int j0 = jt * BN + c * 32;
          if (j0 >= jlim) break;  // the rest of the tile is past the eligible blocks
          uint32_t v[32];
          tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + ac * BN + c * 32, v);
          tmem_wait_ld();
          // bit k: block j0 + k beats the current K-th best (masks only where a chunk reaches past
          // the eligible blocks or holds the own block)
          uint32_t cand = 0;
          if (j0 + 32 <= jlim && (own < j0 || own >= j0 + 32)) {
#pragma unroll
            for (int k = 0; k < 32; ++k) cand |= (__uint_as_float(v[k]) > thr ? 1u : 0u) << k;
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int j = j0 + k;
              cand |= ((j < jlim && j != own && __uint_as_float(v[k]) > thr) ? 1u : 0u) << k;
            }
          }
          if (__any_sync(0xffffffffu, cand != 0)) {
            // the winners, in block order, through shared memory (a register array cannot be
            // indexed by a runtime bit position)
#pragma unroll
            for (int k = 0; k < 32; ++k) my_spill[k * BQ] = __uint_as_float(v[k]);
            while (cand) {
              const int k = __ffs(cand) - 1;
              cand &= cand - 1;
              const float s = my_spill[k * BQ];
              if (s > thr) {
                list_insert(sv, si, s, j0 + k);
                thr = sv[KM - 1];
              }
            }
          }
          __syncwarp();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[ac]);
        ++acc_it;
      }
      if (!ok) break;
      if (valid) {
        // the own block (causal) joins the ranked blocks; the set is written ascending,
        // -1 padded (odd-even transposition sort over fixed positions)
        int e[KM + 1];
#pragma unroll
        for (int k = 0; k < KM; ++k) e[k] = si[k] < 0 ? BIG : si[k];  // sentinels and empty places
        e[KM] = p.causal ? own : BIG;
#pragma unroll
        for (int pass = 0; pass < KM + 1; ++pass)
#pragma unroll
          for (int k = pass & 1; k + 1 < KM + 1; k += 2) {
            const int a = min(e[k], e[k + 1]), b = max(e[k], e[k + 1]);
            e[k] = a;
            e[k + 1] = b;
          }
        int32_t* out = p.idx + ((size_t)bh * p.N + t) * p.Ksel;
#pragma unroll
        for (int k = 0; k < KM; ++k)
          if (k < p.Ksel) out[k] = e[k] == BIG ? -1 : e[k];
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, NACC * BN);
  }
}

template <int D>
cudaError_t launch_d(const uint16_t* Q, const uint16_t* P, int32_t* idx, uint16_t* Qs, const Problem& p,
                     const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s) {
  const long long BH = (long long)p.B * p.H_kv;
  const long long total = BH * p.N;
  if (total == 0) return cudaSuccess;
  {
    long long blocks = (total + 7) / 8;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    bsa_qsum_kernel<D><<<(int)blocks, 256, 0, s>>>(Q, Qs, p.N, p.H_q, p.H_kv, p.GQ, total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mapA, mapB;
  {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)(BH * 2 * p.N)};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)BQ};
    if (!encode_tensor_map(&mapA, Qs, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)(BH * geo.nodes)};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)BN};
    if (!encode_tensor_map(&mapB, P, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  BsaParams prm;
  prm.idx = idx;
  prm.BH = (int)BH;
  prm.N = p.N;
  prm.M1 = geo.M[1];
  prm.Ksel = p.K;
  prm.Kp = p.causal ? p.K - 1 : p.K;
  prm.causal = p.causal;
  prm.ntq = (p.N + BQ - 1) / BQ;
  prm.ntiles = BH * prm.ntq;
  prm.nodes = geo.nodes;
  const size_t smem = (size_t)NA * 2 * BQ * D * 2 + (size_t)NB * BN * D * 2 + 32 * BQ * 4 + 1024;
  const long long grid = prm.ntiles < num_sms ? prm.ntiles : num_sms;
  // the register list holds K entries (with the own block: K places for K - 1 ranked blocks)
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(int)grid, THREADS, smem, s>>>(mapA, mapB, prm, err);
    return cudaGetLastError();
  };
  if (p.K <= 8) return go(bsa_select_kernel<D, 8>);
  if (p.K <= 16) return go(bsa_select_kernel<D, 16>);
  return go(bsa_select_kernel<D, 32>);
}

}  // namespace

size_t bsa_workspace_bytes(const Problem& p) { return (size_t)p.B * p.H_kv * 2 * (size_t)p.N * p.d * 2; }

cudaError_t launch_bsa_select(const uint16_t* Q, const uint16_t* P, int32_t* idx, void* ws, const Problem& p,
                              const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s) {
  uint16_t* Qs = static_cast<uint16_t*>(ws);
  if (p.d == 128) return launch_d<128>(Q, P, idx, Qs, p, geo, num_sms, err, s);
  return launch_d<64>(Q, P, idx, Qs, p, geo, num_sms, err, s);
}

}  // namespace pisa
