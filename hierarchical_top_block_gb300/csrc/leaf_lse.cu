// Stage 2 of the two-stage selection (summary page of "Block Sparse Attention with
// Log-Linear Complexity", section "Method step details", step 2; section "Core method",
// eq. 21 at the leaf level): the exact LSE of every leaf candidate over its raw keys,
// summed over the query heads of the GQA group.
//
// Work unit: a tile = up to qt queries (qt * max(G_Q, 8) = 128 rows) that all need the
// same level-2 survivor, i.e. the same pair of sibling leaves (128 contiguous keys).
//   D[128 rows, 128 keys] = Q_tile[128, d] . K_pair[128, d]^T   on tcgen05, fp32 in TMEM
// then each epilogue thread owns one TMEM lane (one query head row) and reduces the 64 keys
// per leaf to log-sum-exp (causal mask inside the query's own block), and the G_Q rows of
// a query are summed with lane shuffles in a fixed order.
//
// Persistent, warp-specialised CTA (one per SM, 17 warps):
//   warp 0      scheduler: tiles come in runs of consecutive tiles from an atomic counter
//               (a run's tile records and entries are staged in shared memory in one round
//               trip); it publishes each tile's record and query list into a 16-slot ring
//               that runs ahead of the Q stages, and loads each new K pair by TMA (3-D map,
//               rows past N read as zero) into a 2-stage ring, reused across consecutive
//               tiles of the same pair.
//   warps 2-3   Q loaders: once a tile's record is out and its Q stage (4-stage ring) is
//               free, the tile's query rows by TMA, the queries split over the two warps.
//               For d = 128 and G_Q a multiple of 8 one 4-D box per query (8-row groups with
//               both d halves), else one 2-D box of RPQ rows per d half; 128-byte swizzle.
//   warp 1, 16  MMA issuers: lane 0 of each issues the d/16 MMAs of alternate tiles (an
//               issuing thread stalls while the tensor pipe's queue is full, so the other
//               prepares its next tile meanwhile) and commits to mbarriers; warp 1 owns TMEM
//               (3 x 128 columns of accumulators, one per epilogue group).
//   warps 4-15  epilogue: three groups of four (one warp per TMEM lane quarter), group g
//               taking tiles g, g+3, ... in its own accumulator; each warp reduces both
//               leaves of its rows.
// Every wait is bounded; on timeout the error word is set, the MMAs and TMA loads still in
// flight are waited for (bounded) and the CTA exits.  Launched as a programmatic dependent of
// the clustering's last kernel.
#include "kernels.cuh"
#include "pdl.cuh"

namespace pisa {
namespace {

constexpr int NQS = 4;            // Q stages
constexpr int NREC = 16;          // tile records, published ahead of the Q stages and read by the epilogue
constexpr int NKS = 2;            // K-pair stages
constexpr int ROWS = 128;         // MMA M (query-head rows)
constexpr int KEYS = 128;         // MMA N (two leaves of 64 keys)
constexpr int NACC = 3;           // accumulator buffers = epilogue groups
constexpr int EPI_WARPS = 4 * NACC;
constexpr int LOAD_WARPS = 2;
constexpr int LOAD_WARP0 = 2;
constexpr int EPI_WARP0 = 4;      // a warpgroup boundary, so warp & 3 is the TMEM lane quarter
constexpr int MMA2_WARP = EPI_WARP0 + EPI_WARPS;  // the second MMA issuer (the first is warp 1)
constexpr int THREADS = 32 * (MMA2_WARP + 1);     // 544: 96 registers a thread

// Accumulator buffer a = t % NACC holds tile t; MMA issuer t & 1 issues it.  Use m = t / NACC
// of buffer a waits for the release of use m - 1, which the epilogue group signals on the
// empty barrier of the issuer of use m, so each issuer waits every phase of its own barriers
// in order (a parity wait never runs two phases ahead of its barrier).  Returns the phase
// index of that release among the releases on the barrier, or -1 when no wait is needed.
__device__ __forceinline__ int acc_release_phase(int t) {
  const int a = t % NACC, m = t / NACC;
  if (m == 0) return -1;
  if (NACC % 2 == 0) return m - 1;            // every use of the buffer has the same issuer
  const int j0 = ((t & 1) + a + 1) & 1;        // first earlier use whose successor is t's issuer
  return (m - 1 - j0) >> 1;
}
constexpr uint32_t TMEM_COLS = 512;
constexpr int QT_MAX = ROWS / 8;  // queries per tile (G_Q rows each, padded to 8)



struct TileInfo {
  int4 tile;   // bh, node, first entry, count
  int ks;      // K stage holding the pair
  int newk;    // 1 if the pair was loaded for this tile
};

constexpr int SCHED_CHUNK = 8;    // tiles handed to a CTA per grab (consecutive: mostly one K pair)

struct Params {
  const int4* tiles;
  const int32_t* entries;
  const int32_t* totals;
  int32_t* sched;      // tile counter, zero at launch
  float* leaf_score;
  int N, H_q, H_kv, GQ, RPQ, Ksel, M1, causal;
  int qgrp;   // 1: one 4-D box per query, stage layout [query][8-row group][d half][8][64]
  int scoring;  // 0 LSE, 1 log m + mean, 2 log m + mean + variance / 2
  float sl2;  // scale * log2(e)
  int32_t* counts;     // the clustering histogram and Stage 1's item counter: zeroed here
  long long ncounts;
};

// SC >= 0: the block score fixed at compile time (else prm.scoring); R > 0: G_Q = RPQ = R
template <int D, int SC, int R>
__global__ void __launch_bounds__(THREADS, 1) leaf_lse_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                              const __grid_constant__ CUtensorMap mapK, Params prm,
                                                              uint32_t* err) {
  pdl_trigger();
  pdl_wait();  // the tile list and its counts come from the kernel before
  // nothing reads the histogram (or Stage 1's item counter) after the tile list: left zeroed,
  // so a next selection over the same scratch may skip its memset
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < prm.ncounts;
       i += (long long)gridDim.x * blockDim.x)
    prm.counts[i] = 0;
  constexpr int HALVES = D / 64;
  constexpr uint32_t STAGE_BYTES = ROWS * D * 2;   // also the K-pair stage size (KEYS == ROWS)
  constexpr int KSTEPS = D / 16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + NQS * STAGE_BYTES;

  __shared__ uint64_t rec_full[NREC], rec_empty[NREC], q_full[NQS], q_empty[NQS], k_full[NKS], k_empty[NKS],
      acc_full[NACC], acc_empty[NACC][2], drain;
  __shared__ TileInfo rec[NREC];
  __shared__ int32_t rec_ent[NREC][QT_MAX];
  __shared__ uint32_t tmem_base_s;
  __shared__ int done_it_s;  // iteration index of the end marker
  __shared__ int4 chunk_tiles[SCHED_CHUNK];        // producer staging of the current chunk
  __shared__ int32_t chunk_ent[SCHED_CHUNK * ROWS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    done_it_s = 0x7fffffff;
    for (int i = 0; i < NREC; ++i) {
      mbar_init(&rec_full[i], 1);
      mbar_init(&rec_empty[i], LOAD_WARPS + 4 + 2);  // read by the Q loaders, an epilogue group, both MMA issuers
    }
    for (int i = 0; i < NQS; ++i) {
      mbar_init(&q_full[i], LOAD_WARPS);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < NKS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 2);  // both MMA issuers
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i][0], 4);  // released for the next use by issuer 0 / 1
      mbar_init(&acc_empty[i][1], 4);
    }
    mbar_init(&drain, 2);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, TMEM_COLS);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  const int ntiles = prm.totals[1];

  // ------------------------------ MMA issuers ------------------------------
  // Two threads (lane 0 of warp 1 and of the last warp) issue the MMAs of alternate tiles, so
  // one waits for its next tile's Q stage, K pair and accumulator while the other's MMAs run
  // (an issuing thread stalls while the tensor pipe's queue is full).  Each reads every tile
  // record, so both follow the K-stage sequence, and commits its own MMAs on k_empty when the
  // pair changes (k_empty counts both).  A tile's MMAs complete -> its Q stage is free and
  // its accumulator goes to the epilogue group; the record stays in its ring slot until the
  // loaders, both issuers and the group have read it.
  auto mma_issuer = [&](const int par) {
    constexpr uint32_t idesc = idesc_bf16_f32(ROWS, KEYS);
    uint32_t kload = 0;
    int cur_ks = -1;
    bool kwait = false;  // the current K pair has not been waited for by this thread
    // Every K load is waited for in order, also those of pairs without a tile of this thread,
    // so no parity wait runs two phases ahead of k_full (the scheduler publishes a record
    // before the stage it names is free).
    auto wait_k = [&]() -> bool {
      if (!kwait) return true;
      kwait = false;
      return mbar_wait(&k_full[cur_ks], ((kload - 1) / NKS) & 1, err);
    };
    auto wait_acc = [&](int t) -> bool {
      const int ph = acc_release_phase(t);
      return ph < 0 || mbar_wait(&acc_empty[t % NACC][par], (ph & 1), err);
    };
    for (int it = 0;; ++it) {
      const int qs = it % NQS, rs = it % NREC;
      if (!mbar_wait(&rec_full[rs], (it / NREC) & 1, err)) break;
      const TileInfo ti = rec[rs];
      if (ti.tile.w < 0) {  // end marker: tell the groups of this thread's parity once their buffers are free
        done_it_s = it;     // both issuers write the same value
        __threadfence_block();
        for (int k = 0; k < NACC; ++k) {
          const int i2 = it + k;
          if ((i2 & 1) != par) continue;
          if (!wait_acc(i2)) break;
          mbar_arrive(&acc_full[i2 % NACC]);
        }
        break;
      }
      mbar_arrive(&rec_empty[rs]);
      if (ti.newk) {
        if (!wait_k()) break;
        if (cur_ks >= 0) umma_commit(&k_empty[cur_ks]);
        ++kload;
        cur_ks = ti.ks;
        kwait = true;
      }
      if ((it & 1) != par) continue;
      if (!wait_k() || !mbar_wait(&q_full[qs], (it / NQS) & 1, err) || !wait_acc(it)) break;
      const int a = it % NACC;
      tc_fence_after();
      const uint32_t qbase = smem_u32(sQ + qs * STAGE_BYTES);
      const uint32_t kbase = smem_u32(sK + ti.ks * STAGE_BYTES);
#pragma unroll
      for (int s = 0; s < KSTEPS; ++s) {
        const uint32_t off = (s >> 2) * (ROWS * 128) + (s & 3) * 32;
        // grouped Q: d half h of 8-row group g at g * 2048 + h * 1024
        const uint32_t qoff = prm.qgrp ? (s >> 2) * 1024 + (s & 3) * 32 : off;
        umma_bf16(tmem_base + a * KEYS, smem_desc_sw128(qbase + qoff, 16, prm.qgrp ? 2048 : 1024),
                  smem_desc_sw128(kbase + off, 16, 1024), idesc, s > 0 ? 1u : 0u);
      }
      umma_commit(&acc_full[a]);
      umma_commit(&q_empty[qs]);
    }
    // every MMA issued by either thread has completed before the tensor memory is released
    // (bounded)
    umma_commit(&drain);
    mbar_wait(&drain, 0, err);
  };

  if (warp == 0) {
    // ------------------------------ scheduler ------------------------------
    // Publishes tile records into a ring that runs up to NREC tiles ahead of the Q stages,
    // and loads each new K pair.
    const uint64_t keep_policy = l2_evict_last_policy();  // K pairs are reused by later windows
    uint32_t kload = 0;
    int prev_bh = -1, prev_node = -1, ks = 0;
    int next_tile = 0, chunk_end = 0, chunk_base = 0, chunk_e0 = 0;
    bool failed = false;
    for (int it = 0;; ++it) {
      const int rs = it % NREC;
      if (next_tile >= chunk_end) {
        // grab the next run of consecutive tiles (mostly one K pair) and stage their tile
        // records and entries in shared memory with one round trip each
        int base = 0;
        if (lane == 0) base = atomicAdd(prm.sched, SCHED_CHUNK);
        base = __shfl_sync(0xffffffffu, base, 0);
        next_tile = chunk_base = base;
        chunk_end = min(base + SCHED_CHUNK, ntiles);
        if (base < ntiles) {
          if (lane < chunk_end - base) chunk_tiles[lane] = prm.tiles[base + lane];
          __syncwarp();
          const int4 first = chunk_tiles[0], last = chunk_tiles[chunk_end - base - 1];
          chunk_e0 = first.z;
          const int ne = last.z + last.w - first.z;
          for (int i = lane; i < ne; i += 32) chunk_ent[i] = prm.entries[chunk_e0 + i];
          __syncwarp();
        }
      }
      if (!mbar_wait_warp(&rec_empty[rs], ((it / NREC) & 1) ^ 1, err)) {
        failed = true;
        break;
      }
      if (next_tile >= ntiles) {  // no work left: pass an end marker down the pipeline
        if (lane == 0) {
          rec[rs].tile = make_int4(0, 0, 0, -1);
          mbar_arrive(&rec_full[rs]);
        }
        break;
      }
      const int4 tl = chunk_tiles[next_tile - chunk_base];
      ++next_tile;
      const int bh = tl.x, node = tl.y, start = tl.z, cnt = tl.w;
      const int newk = (bh != prev_bh || node != prev_node) ? 1 : 0;
      if (newk) ks = kload % NKS;
      // publish the tile first: its Q loads need not wait for a free K stage
      if (lane < cnt) rec_ent[rs][lane] = chunk_ent[start - chunk_e0 + lane];
      __syncwarp();
      if (lane == 0) {
        rec[rs].tile = tl;
        rec[rs].ks = ks;
        rec[rs].newk = newk;
        mbar_arrive(&rec_full[rs]);  // release: the record is visible to whoever waits
      }
      __syncwarp();
      if (newk) {
        if (!mbar_wait_warp(&k_empty[ks], ((kload / NKS) & 1) ^ 1, err)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&k_full[ks], STAGE_BYTES);
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            tma_load_3d_hint(sK + ks * STAGE_BYTES + h * (KEYS * 128), &mapK, &k_full[ks], 64 * h, node * KEYS, bh,
                             keep_policy);
        }
        ++kload;
        prev_bh = bh;
        prev_node = node;
      }
    }
    // after a timeout, K pairs still in flight land before shared memory goes away (bounded):
    // the latest load of each stage completes its barrier's current phase
    if (failed && lane == 0)
      for (uint32_t k = kload > NKS ? kload - NKS : 0; k < kload; ++k) mbar_wait(&k_full[k % NKS], (k / NKS) & 1, err);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) mma_issuer(0);
    __syncwarp();
  } else if (warp == MMA2_WARP) {
    if (lane == 0) mma_issuer(1);
    __syncwarp();
  } else if (warp >= LOAD_WARP0 && warp < LOAD_WARP0 + LOAD_WARPS) {
    // ------------------------------ Q loaders ------------------------------
    // Each loader waits for the tile's record and for the Q stage to be free, then issues
    // the TMA boxes (one per query, or RPQ rows x 64 columns per d half) of the tile's
    // queries w, w + LOAD_WARPS, ...; each warp arrives on the stage's barrier with the
    // bytes it expects, so the MMA issuer sees the stage full once every box has landed.
    const int lw = warp - LOAD_WARP0;
    int issued = 0;  // iterations whose loads this warp has issued
    bool failed = false;
    for (int it = 0;; ++it) {
      const int qs = it % NQS, rs = it % NREC;
      if (!mbar_wait_warp(&rec_full[rs], (it / NREC) & 1, err) ||
          !mbar_wait_warp(&q_empty[qs], ((it / NQS) & 1) ^ 1, err)) {
        failed = true;
        break;
      }
      const int4 tl = rec[rs].tile;
      if (tl.w < 0) {  // end marker: pass it to the MMA issuer
        if (lane == 0) mbar_arrive(&q_full[qs]);
        break;
      }
      const int bh = tl.x, cnt = tl.w;
      const int b = bh / prm.H_kv, hk = bh - b * prm.H_kv;
      const int mine = cnt > lw ? (cnt - lw + LOAD_WARPS - 1) / LOAD_WARPS : 0;  // queries of this warp
      int t_mine = 0;
      if (lane < mine) t_mine = rec_ent[rs][lw + LOAD_WARPS * lane] >> 6;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&rec_empty[rs]);
        mbar_arrive_expect_tx(&q_full[qs], (uint32_t)mine * prm.RPQ * D * 2);
      }
      __syncwarp();
      if (prm.qgrp) {  // the query's 8-row groups with both d halves in one box
        if (lane < mine) {
          const int i = lw + LOAD_WARPS * lane;
          const long long row = ((long long)b * prm.N + t_mine) * prm.H_q + (long long)hk * prm.GQ;
          tma_load_4d(sQ + qs * STAGE_BYTES + i * prm.RPQ * 256, &mapQ, &q_full[qs], 0, 0, 0, (int)(row >> 3));
        }
      } else {
        // lane j of the first mine * HALVES issues d half j % HALVES of query j / HALVES
        const int src = lane / HALVES, h = lane % HALVES;
        const int t = __shfl_sync(0xffffffffu, t_mine, src < 32 ? src : 0);
        if (lane < mine * HALVES) {
          const int i = lw + LOAD_WARPS * src;
          const int row = (int)(((long long)b * prm.N + t) * prm.H_q + (long long)hk * prm.GQ);
          tma_load_2d(sQ + qs * STAGE_BYTES + h * (ROWS * 128) + i * prm.RPQ * 128, &mapQ, &q_full[qs], 64 * h,
                      row);
        }
      }
      issued = it + 1;
    }
    // after a timeout, Q rows still in flight land before shared memory goes away (bounded);
    // on the normal path every stage was consumed, and the end marker has reused one of them
    if (failed && lane == 0)
      for (int k = issued > NQS ? issued - NQS : 0; k < issued; ++k) mbar_wait(&q_full[k % NQS], (k / NQS) & 1, err);
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    // NACC groups of four warps, one warp per TMEM lane quarter: group g takes the tiles
    // g, g + NACC, ... (accumulator buffer g) and reduces both leaves of each, so the epilogue
    // warps sharing a scheduler partition work on different tiles and hide each other's
    // TMEM loads, shuffles and stores.
    const int ew = warp - EPI_WARP0;
    const int grp = ew >> 2;
    const int quarter = warp & 3;
    const int RPQ = R > 0 ? R : prm.RPQ, GQ = R > 0 ? R : prm.GQ;
    const int scoring = SC >= 0 ? SC : prm.scoring;
    const int row = quarter * 32 + lane;
    const int qi = row / RPQ, h = row - qi * RPQ;
    const int twoK = 2 * prm.Ksel;
    for (int it = grp;; it += NACC) {
      const int a = grp, rs = it % NREC;
      if (!mbar_wait_warp(&acc_full[a], (it / NACC) & 1, err)) break;
      if (it >= *(volatile int*)&done_it_s) break;
      tc_fence_after();
      // the record's publication, acquired directly (it completed before the MMAs were issued,
      // and the slot cannot be reused before this group frees it, so this returns at once)
      if (!mbar_wait_warp(&rec_full[rs], (it / NREC) & 1, err)) break;
      const int4 tl = rec[rs].tile;
      const bool vq = qi < tl.w;
      const int e = vq ? rec_ent[rs][qi] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&rec_empty[rs]);
      const int t = e >> 6, slot = e & 63;
      const int bh = tl.x, node = tl.y;
#pragma unroll 1
      for (int leaf_c = 0; leaf_c < 2; ++leaf_c) {
        uint32_t v[64];
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + a * KEYS + leaf_c * 64;
        tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_wait_ld();
        if (leaf_c == 1) {  // the accumulator is read out: the MMA may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a][(it + NACC) & 1]);  // for the issuer of the next use
        }
        const int leaf = 2 * node + leaf_c;
        const long long key0 = (long long)leaf * 64;
        const bool leaf_ok = vq && leaf < prm.M1 && (!prm.causal || key0 <= t);
        // keys j <= lim of this leaf are visible (causal: key <= t; always: key < N)
        long long lim64 = (long long)prm.N - 1 - key0;
        if (prm.causal && (long long)t - key0 < lim64) lim64 = (long long)t - key0;
        const int lim = (int)(lim64 < 63 ? lim64 : 63);
        float lse2 = NEG_INF;
        if (leaf_ok && h < GQ && scoring != 0) {
          // truncated forms over the m = lim + 1 visible keys, log2 units: log2 m + mean(x),
          // plus ln2/2 * Var(x) for the second order; x = logit * sl2, so the sums run on the
          // raw logits and are scaled once (Var by sl2^2)
          const float m = (float)(lim + 1);
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
          if (lim >= 63) {
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              a0 += __uint_as_float(v[j]);
              a1 += __uint_as_float(v[j + 1]);
              a2 += __uint_as_float(v[j + 2]);
              a3 += __uint_as_float(v[j + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              a0 += (j <= lim) ? __uint_as_float(v[j]) : 0.f;
              a1 += (j + 1 <= lim) ? __uint_as_float(v[j + 1]) : 0.f;
            }
          }
          const float mean = ((a0 + a1) + (a2 + a3)) / m;  // raw logits
          lse2 = fast_log2(m) + mean * prm.sl2;
          if (scoring == 2) {
            float q0 = 0.f, q1 = 0.f, q2 = 0.f, q3 = 0.f;
            if (lim >= 63) {
#pragma unroll
              for (int j = 0; j < 64; j += 4) {
                const float d0 = __uint_as_float(v[j]) - mean, d1 = __uint_as_float(v[j + 1]) - mean;
                const float d2 = __uint_as_float(v[j + 2]) - mean, d3 = __uint_as_float(v[j + 3]) - mean;
                q0 = fmaf(d0, d0, q0);
                q1 = fmaf(d1, d1, q1);
                q2 = fmaf(d2, d2, q2);
                q3 = fmaf(d3, d3, q3);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 64; j += 2) {
                const float d0 = __uint_as_float(v[j]) - mean, d1 = __uint_as_float(v[j + 1]) - mean;
                q0 += (j <= lim) ? d0 * d0 : 0.f;
                q1 += (j + 1 <= lim) ? d1 * d1 : 0.f;
              }
            }
            lse2 += 0.5f * LN2 * prm.sl2 * prm.sl2 * ((q0 + q1) + (q2 + q3)) / m;
          }
        } else if (leaf_ok && h < GQ) {
          // four independent partial sums; the mask is only needed inside the own block
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
          if (lim >= 63) {
            // the scaling and the sums two lanes per instruction (packed fp32: same roundings
            // and the same four partial sums as the scalar form)
            const unsigned long long s2 = pack_f32x2(prm.sl2, prm.sl2);
            unsigned long long acc01 = 0ull, acc23 = 0ull;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              float a, b, c, d;
              unpack_f32x2(mul_f32x2(pack_u32x2(v[j], v[j + 1]), s2), a, b);
              unpack_f32x2(mul_f32x2(pack_u32x2(v[j + 2], v[j + 3]), s2), c, d);
              acc01 = add_f32x2(acc01, pack_f32x2(fast_exp2(a), fast_exp2(b)));
              acc23 = add_f32x2(acc23, pack_f32x2(fast_exp2(c), fast_exp2(d)));
            }
            unpack_f32x2(acc01, p0, p1);
            unpack_f32x2(acc23, p2, p3);
          } else {
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              p0 += (j <= lim) ? fast_exp2(__uint_as_float(v[j]) * prm.sl2) : 0.f;
              p1 += (j + 1 <= lim) ? fast_exp2(__uint_as_float(v[j + 1]) * prm.sl2) : 0.f;
            }
          }
          const float s = (p0 + p1) + (p2 + p3);
          if (s > 0.f && s < POS_INF) {
            lse2 = fast_log2(s);
          } else {  // logits beyond the fp32 exponent range: subtract the max first
            float m = NEG_INF;
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (j <= lim) m = fmaxf(m, __uint_as_float(v[j]) * prm.sl2);
            float s2 = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (j <= lim) s2 += fast_exp2(__uint_as_float(v[j]) * prm.sl2 - m);
            lse2 = m + fast_log2(s2);
          }
        }
        // sum over the G_Q head rows of each query (lanes of one query are contiguous)
        float part = (leaf_ok && h < GQ) ? lse2 : 0.f;
        for (int o = 1; o < RPQ; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (vq && h == 0)
          prm.leaf_score[((size_t)bh * prm.N + t) * twoK + 2 * slot + leaf_c] = leaf_ok ? part * LN2 : NEG_INF;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const uint16_t* Q, const uint16_t* K, const ClusterBuffers& cb, float* leaf_score,
                     const Problem& p, const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s) {
  const int RPQ = p.GQ < 8 ? 8 : p.GQ;
  CUtensorMap mapQ, mapK;
  Params prm;
  // d = 128 with G_Q a multiple of 8: one box per query, (64 columns, 8 rows, 2 d halves,
  // G_Q / 8 row groups), lands as [row group][half][8 rows][64]: per d half the 8-row groups
  // are 2 KB apart, a valid 128-byte-swizzled K-major operand; otherwise one 2-D box of RPQ
  // rows per d half
  const long long rows = (long long)p.B * p.N * p.H_q;
  prm.qgrp = (D == 128 && p.GQ % 8 == 0 && p.H_q % 8 == 0) ? 1 : 0;
  if (prm.qgrp) {
    const uint64_t dims[4] = {64, 8, 2, (uint64_t)(rows / 8)};
    const uint64_t strides[3] = {(uint64_t)D * 2, 128, (uint64_t)8 * D * 2};
    const uint32_t box[4] = {64, 8, 2, (uint32_t)(p.GQ / 8)};
    if (!encode_tensor_map(&mapQ, Q, 4, dims, strides, box)) return cudaErrorInvalidValue;
  } else {
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, (uint32_t)RPQ};
    if (!encode_tensor_map(&mapQ, Q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.N, (uint64_t)p.B * p.H_kv};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.N * D * 2};
    const uint32_t box[3] = {64, (uint32_t)KEYS, 1};
    if (!encode_tensor_map(&mapK, K, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  prm.tiles = cb.tiles;
  prm.entries = cb.entries;
  prm.totals = cb.totals;
  prm.sched = cb.totals + 2;
  prm.leaf_score = leaf_score;
  prm.N = p.N;
  prm.H_q = p.H_q;
  prm.H_kv = p.H_kv;
  prm.GQ = p.GQ;
  prm.RPQ = RPQ;
  prm.Ksel = p.K;
  prm.M1 = geo.M[1];
  prm.causal = p.causal;
  prm.scoring = p.scoring;
  prm.sl2 = p.scale * LOG2E;
  prm.counts = cb.counts;
  prm.ncounts = cb.nkeys + 1;
  const size_t smem = (size_t)(NQS + NKS) * ROWS * D * 2 + 1024;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.maxThreadsPerBlock < THREADS) return cudaErrorLaunchOutOfResources;  // registers x threads
    return launch_pdl(kern, dim3(num_sms), dim3(THREADS), smem, s, mapQ, mapK, prm, err);
  };
  if (p.GQ == 16 && RPQ == 16) return p.scoring == 0 ? go(leaf_lse_kernel<D, 0, 16>) : go(leaf_lse_kernel<D, -1, 16>);
  return p.scoring == 0 ? go(leaf_lse_kernel<D, 0, 0>) : go(leaf_lse_kernel<D, -1, 0>);
}

}  // namespace

cudaError_t launch_leaf_lse(const uint16_t* Q, const uint16_t* K, const ClusterBuffers& cb, float* leaf_score,
                            const Problem& p, const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s) {
  if (p.d == 128) return launch_d<128>(Q, K, cb, leaf_score, p, geo, num_sms, err, s);
  return launch_d<64>(Q, K, cb, leaf_score, p, geo, num_sms, err, s);
}

}  // namespace pisa
