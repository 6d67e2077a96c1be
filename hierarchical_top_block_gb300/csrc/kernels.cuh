// Internal launchers of the PISA kernels (one per translation unit), called by api.cu.
#pragma once

#include "common.cuh"

namespace pisa {

struct Problem {
  int B, N, N_cap, H_q, H_kv, d;
  int C, g, K, causal;
  int scoring;  // 0 LSE, 1 log m + mean, 2 log m + mean + variance / 2
  float scale;  // logit scale (already resolved; > 0)
  int GQ;       // H_q / H_kv
  // queries processed by the per-query kernels (Stage 1, clustering, top-K, attention):
  // t in [t_lo, t_hi); every buffer keeps its full-length layout and is indexed by t
  int t_lo, t_hi;
};

// Builds pyramid levels 1..geo.L from the first N rows of K (layout capacity N_cap).
cudaError_t launch_pyramid(const uint16_t* K, uint16_t* P, const Problem& p, const Geometry& geo, cudaStream_t s);
// Rewrites the nodes whose span meets keys [key_lo, key_hi); builds over consecutive ranges,
// each run once the keys below its key_hi are in place, leave the nodes below the last key_hi exact.
cudaError_t launch_pyramid_range(const uint16_t* K, uint16_t* P, const Problem& p, const Geometry& geo, long long key_lo,
                                 long long key_hi, cudaStream_t s);

// Clustering of (query, level-2 survivor) entries into per-(b, h_kv, window, node) lists
// and Q tiles for Stage 2.
struct ClusterBuffers {
  int32_t* counts;      // [nkeys]
  int32_t* rank;        // [B * H_kv * N * 2K]  place of entry (t, slot) in its key's list, at
                        // [(bh * N + t) * 2K + slot] (the leaf-score buffer, before Stage 2 fills it)
  int32_t* offsets;     // [nkeys]  exclusive scan of counts
  int32_t* tile_off;    // [nkeys]  exclusive scan of ceil(counts / qt)
  int32_t* block_sums;  // [2 * nblocks]
  int32_t* entries;     // [B * H_kv * N * K]   (t << 6) | slot
  int4* tiles;          // [max_tiles]          {bh, node, entry start, entry count}
  int32_t* totals;      // [4] {entries, tiles, ...}
  int32_t* sched;       // [1] Stage 1 item counter, zeroed with counts
  long long nkeys;
  int nwin, win, M2, qt, nblocks;
  long long max_tiles;
};
// Stage 1: level walk for every (b, h_kv, t); writes the level-2 survivors S2 [.., K] and adds
// each survivor to the clustering histogram cb.counts (zeroed by the caller, with cb.sched).
cudaError_t launch_stage1(const uint16_t* Q, const uint16_t* P, int32_t* S2, const ClusterBuffers& cb, const Problem& p,
                          const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s);

// The rest of the clustering: scans of the histogram, scatter of the entries, tile list.
cudaError_t launch_cluster(const int32_t* S2, const ClusterBuffers& cb, const Problem& p, cudaStream_t s);

// Stage 2: exact leaf LSE of the candidate leaf pairs with tcgen05, head-summed.
cudaError_t launch_leaf_lse(const uint16_t* Q, const uint16_t* K, const ClusterBuffers& cb, float* leaf_score,
                            const Problem& p, const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s);

// Final top-K with the own block kept; idx rows ascending, -1 padded.
// Also writes -inf into the leaf-score slots of absent survivors.
cudaError_t launch_topk(const int32_t* S2, float* leaf_score, int32_t* idx, const Problem& p,
                        const Geometry& geo, int num_sms, cudaStream_t s);

// BSA flat selection: head-summed query parts into ws (bsa_workspace_bytes), then the scoring
// GEMM with a per-query top-K over every eligible leaf summary; idx rows ascending, -1 padded.
size_t bsa_workspace_bytes(const Problem& p);
cudaError_t launch_bsa_select(const uint16_t* Q, const uint16_t* P, int32_t* idx, void* ws, const Problem& p,
                              const Geometry& geo, int num_sms, uint32_t* err, cudaStream_t s);

// Block-sparse attention over idx.
cudaError_t launch_sparse_attn(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                               uint16_t* O, float* LSE, const Problem& p, int num_sms, uint32_t* err, cudaStream_t s);

// Backward of the attention over the selected blocks (dQ, dK, dV).
// with_ds: room for dS of every (query, block) pair (where the tcgen05 path writes it), which
// spares the dQ kernel forming S and dP again
size_t attn_backward_workspace_bytes(const Problem& p, bool with_ds);
cudaError_t launch_attn_backward(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                 const uint16_t* O, const float* LSE, const uint16_t* dO, float* dQ, float* dK,
                                 float* dV, void* ws, bool with_ds, const Problem& p, int num_sms, uint32_t* err,
                                 cudaStream_t s);

// Fused decode step.  logits (nullable, decode_logits_bytes(p) bytes) keeps the leaf
// candidates' logits for the attention, which then reads no K rows of the selected blocks.
size_t decode_logits_bytes(const Problem& p);
cudaError_t launch_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                          uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out, float* logits,
                          const Problem& p, const Geometry& geo_cap, uint32_t* err, cudaStream_t s);

// One CTA whose bounded waits run out after limit_ns (checks the timeout path).
cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* err, cudaStream_t s);

// Tensor-map encoding through the driver entry point (no link-time libcuda dependency).
bool encode_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace pisa
