/*
 * pisa.h - C ABI of the GB300 (sm_103a) library for log-linear block-sparse attention
 * with pyramid-LSE block selection.
 *
 * Method: "Block Sparse Attention with Log-Linear Complexity" (Tang, Qin, Pan, Li, Liu),
 * as described on its summary page:
 *   - section "Prerequisites", BSA: keys/values are cut into contiguous blocks of C keys,
 *     each query keeps K blocks and attends only to their raw K/V;
 *   - section "Core method", eq. 21: a candidate block's score is the log-sum-exp of its
 *     children's logits q.k/sqrt(d) (raw keys at the leaf level);
 *   - section "Method step details": step 1 the mean-pooled key pyramid (eqs 10-15);
 *     step 2 the coarse-to-fine walk that scores at most gK candidates per level, sums the
 *     score over the GQA group (eq. 22), keeps K (SelectK), expands survivors to their
 *     children, scores the leaf candidates exactly and takes a final top-K; step 3 the
 *     decode step that updates the new token's leaf and ancestors and walks all levels in
 *     one kernel; step 4 attention over the selected blocks.
 * The softmax runs over the connected positions only (blog post of the same title, 3.3).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, unless a name ends in
 *     _host.  The library allocates nothing: scratch memory is passed in as `ws`.
 *   - bf16 tensors are passed as uint16_t bit patterns; every tensor is row-major with
 *     the last dimension contiguous and a 16-byte aligned base.
 *   - Layouts: Q, O [B][N][H_q][d];  K, V [B][H_kv][N_cap][d];
 *              P (pyramid) [B][H_kv][pisa_pyramid_nodes(N_cap)][d], level l (1 = leaves)
 *              starting at node offset sum_{l'<l} M_l'(N_cap);
 *              idx [B][H_kv][N][K] int32; LSE [B][H_q][N] fp32 (natural log).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Argument errors are reported synchronously, before anything is launched.
 *   - Supported: d in {64, 128}; C = 64; g = 2; 1 <= K <= 32; H_q % H_kv == 0 and
 *     G_Q = H_q / H_kv in {1, 2, 4, 8, 16}.  Other values return PISA_ERR_UNSUPPORTED.
 *   - Sizes: N_cap < 2^25 and B * N_cap * H_q < 2^31 everywhere; the selection entry points
 *     (pisa_select_prefill, pisa_select_prefill_noalloc, pisa_prefill_host) and the backward
 *     also need B * H_kv * N * K < 2^31 (their per-block lists use 32-bit offsets).  Larger
 *     shapes return PISA_ERR_UNSUPPORTED, and their workspace queries return 0.
 *   - Selected index rows are sorted ascending and padded with -1 at the end.
 *   - Kernels never trap: waits are bounded and out-of-range indices are skipped; either
 *     event sets a device error word that pisa_get_last_device_error() returns.
 */
#ifndef PISA_H
#define PISA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PISA_API __attribute__((visibility("default")))
#else
#define PISA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PISA_OK = 0,
  PISA_ERR_INVALID_ARG = 1,  /* NULL or misaligned pointer, bad size */
  PISA_ERR_UNSUPPORTED = 2,  /* valid but not implemented shape or parameter */
  PISA_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  PISA_ERR_TIMEOUT = 4,      /* a bounded device wait gave up (device error word) */
  PISA_ERR_BAD_INDEX = 5,    /* a selected block index was out of range (device error word) */
  PISA_ERR_WORKSPACE = 6     /* ws_bytes smaller than the *_workspace_bytes query */
} pisa_status;

/* Method parameters (summary page, "Reproducibility": C = 64, g = 2, K = 8 or 32). */
typedef struct {
  int C;        /* leaf block size in keys; must be 64 */
  int g;        /* pooling factor per pyramid level; must be 2 */
  int K;        /* blocks kept per query (SelectK and the final top-K) */
  int causal;   /* 1: query t sees keys <= t and blocks starting <= t; own block kept */
  float scale;  /* logit scale; <= 0 selects 1/sqrt(d) */
  int scoring;  /* block score from a block's m eligible child logits z (summary page,
                   "Core method", eq. 21 and its expansion, eqs. 32-34): 0 = PISA, the LSE;
                   1 = PISA-1, log m + mean(z); 2 = PISA-2, log m + mean(z) + Var(z)/2
                   (population variance).  Used at every scored level and at the leaf level;
                   the head sum, SelectK and the final top-K are the same for all three. */
} pisa_params;

typedef struct {
  int B;        /* batch (sequences) */
  int N;        /* tokens per sequence (prefill) */
  int H_q;      /* query heads */
  int H_kv;     /* key/value heads; each serves G_Q = H_q / H_kv query heads */
  int d;        /* head dimension */
  int N_cap;    /* row capacity of the K/V/P layouts (>= N); 0 means N */
} pisa_shape;

typedef void* pisa_stream; /* cudaStream_t */

/* ---- geometry --------------------------------------------------------------------- */

/* Number of pyramid levels for N tokens: M_1 = ceil(N/C) leaves, M_{l+1} = ceil(M_l/g),
 * up to the single root (summary page, step 1).  0 for N = 0. */
PISA_API int pisa_pyramid_levels(long long N, int C, int g);

/* Total pyramid nodes sum_l M_l for N tokens: the P row count per (b, h_kv). */
PISA_API long long pisa_pyramid_nodes(long long N, int C, int g);

/* Scratch bytes pisa_select_prefill needs for this shape (a multiple of 256). */
PISA_API size_t pisa_select_workspace_bytes(pisa_shape shape, pisa_params params);

/* ---- step 1: key pyramid ------------------------------------------------------------ */

/* Builds levels 1..L(N) of P from the first N rows of K (summary page, step 1,
 * eqs 10-15): leaf j = mean of keys [jC, min(jC+C, N)); node i of level l+1 = mean of
 * its <= g children.  Sums are exact to well below bf16 resolution; each node is rounded
 * once to bf16 (nearest even).  K: [B][H_kv][N_cap][d]; P: [B][H_kv][nodes(N_cap)][d]. */
PISA_API pisa_status pisa_build_pyramid(const uint16_t* K, uint16_t* P, pisa_shape shape, pisa_params params,
                               pisa_stream stream);

/* ---- step 2: block selection for prefill ---------------------------------------------- */

/* For every (b, h_kv, t): the coarse-to-fine level walk (scores <= gK candidates per level
 * with eq. 21, sums over the G_Q heads of the group, eq. 22, keeps K), exact leaf LSE of
 * the <= gK leaf candidates, and the final top-K (own block kept in causal mode; ties go
 * to the lower block index).  Q, K, P as above (N_cap must equal N).
 *   idx        [B][H_kv][N][K]   int32 out: selected leaf blocks, ascending, -1 padded.
 *   leaf_score [B][H_kv][N][g*K] fp32 out, nullable: head-summed leaf LSE per candidate
 *              slot (slot g*i + c = child c of the i-th level-2 survivor; -inf if empty).
 *   s2         [B][H_kv][N][K]   int32 out, nullable: level-2 survivors, ascending.
 *   ws         device scratch of at least pisa_select_workspace_bytes(); 256-B aligned. */
PISA_API pisa_status pisa_select_prefill(const uint16_t* Q, const uint16_t* K, const uint16_t* P, int32_t* idx,
                                float* leaf_score, int32_t* s2, void* ws, size_t ws_bytes, pisa_shape shape,
                                pisa_params params, pisa_stream stream);

/* pisa_select_prefill for callers that cannot allocate device memory (a host that owns
 * the allocator, a pool they may not grow, a loop that must not call cudaMalloc).  The
 * paper has no counterpart: this is a library convenience, not part of the method.
 * Same arguments and results as pisa_select_prefill minus ws/ws_bytes: the scratch is one
 * fixed 32 MiB array in device memory that every GPU loading the library holds until the
 * process exits.  Shapes whose pisa_select_workspace_bytes() exceeds 32 MiB return
 * PISA_ERR_WORKSPACE before any launch.  The first call on a device looks up the array's
 * address with that device current, so make it before any stream capture.  All calls share
 * the array (the selection clears what must start at zero): calls that overlap on the GPU
 * race and must be serialised by the caller.  Allocates nothing. */
PISA_API pisa_status pisa_select_prefill_noalloc(const uint16_t* Q, const uint16_t* K, const uint16_t* P,
                                                 int32_t* idx, float* leaf_score, int32_t* s2, pisa_shape shape,
                                                 pisa_params params, pisa_stream stream);

/* ---- baseline: BSA flat selection ----------------------------------------------------- */

/* The single-level selection PISA is compared with (summary page, "Prerequisites": block
 * sparse attention ranks every block by the dot product of the query with the block's
 * summary, q . kbar_j / sqrt(d), over all M = ceil(N / C) blocks, the G_Q heads of a group
 * sharing one selection with their scores summed; "Experimental results", item 5, Fig. 3
 * times this selection against PISA's).  The summaries are the leaf level of P (the mean of
 * each block's keys, as built by pisa_build_pyramid).  In causal mode block j is eligible for
 * query t iff j C <= t and the own block t / C always belongs to the set, counting toward K;
 * ties go to the lower block index; non-causal mode is a plain top-K.  The head sum is taken
 * in fp32 and the products on the tensor cores from a two-part bf16 split of it (score error
 * below 1e-4 at the workloads' sizes).  Only params.K, causal and scale are used; the result
 * does not depend on the scale's value (> 0).  Q, P as for pisa_select_prefill (N_cap must
 * equal N).
 *   idx  [B][H_kv][N][K] int32 out: ascending, -1 padded.
 *   ws   device scratch of at least pisa_select_bsa_workspace_bytes(); 256-B aligned.
 * Shapes with B * H_kv * 2 * N or B * H_kv * nodes(N) >= 2^31 return PISA_ERR_UNSUPPORTED
 * (their workspace query returns 0). */
PISA_API size_t pisa_select_bsa_workspace_bytes(pisa_shape shape, pisa_params params);
PISA_API pisa_status pisa_select_bsa(const uint16_t* Q, const uint16_t* P, int32_t* idx, void* ws, size_t ws_bytes,
                                     pisa_shape shape, pisa_params params, pisa_stream stream);

/* ---- step 4: attention over the selected blocks --------------------------------------- */

/* o_{t,h} = sum over keys c of the selected blocks of head h's group (c <= t if causal) of
 * softmax(scale q.k_c) v_c, with the softmax over those positions only; LSE = log of the
 * softmax denominator.  Entries of idx < 0 are skipped; entries >= ceil(N/C) are skipped
 * and flag PISA_ERR_BAD_INDEX.  A row with no position gives o = 0 and LSE = -inf.
 *   O [B][N][H_q][d] bf16 (nearest even);  LSE [B][H_q][N] fp32, nullable. */
PISA_API pisa_status pisa_sparse_attn_prefill(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                     uint16_t* O, float* LSE, pisa_shape shape, pisa_params params,
                                     pisa_stream stream);

/* Backward of the attention over the selected blocks: the gradient of pisa_sparse_attn_prefill
 * with respect to Q, K and V for an upstream gradient dO (the pages give no backward; this is
 * the derivative of the forward).  With the forward's LSE, for the visible keys c of the
 * selected blocks: P_c = exp(scale q.k_c - LSE), D = dO.O, dS_c = P_c (dO.v_c - D);
 * dq = scale sum dS_c k_c, dk_c += scale dS_c q, dv_c += P_c dO, the last two summed over
 * every query head of the group that selected c's block.  idx, causal and scale as in the
 * forward; only params.K, causal and scale are used.
 *   O, dO [B][N][H_q][d] bf16 (O and LSE from the forward);  LSE [B][H_q][N] fp32.
 *   dQ [B][N][H_q][d] fp32 out;  dK, dV [B][H_kv][N_cap][d] fp32 out (rows >= N are zero).
 *   ws  device scratch, 256-B aligned, of ws_bytes >= pisa_attn_backward_min_workspace_bytes()
 *       (else PISA_ERR_WORKSPACE).  With ws_bytes >= pisa_attn_backward_workspace_bytes(), and
 *       for d = 128 and G_Q of 8 or 16, it also holds dS of every (query, selected block) in
 *       bf16 (B * H_kv * N * K * G_Q * 64 * 2 bytes, 8.6 GB at N = 262144, H_kv = 1,
 *       G_Q = K = 16; up to 64 GB): the dK/dV kernel writes it and the dQ kernel reads it
 *       instead of forming S and dP again.  The results are the same either way up to the
 *       rounding order of the fp32 sums.
 * dK and dV accumulate with fp32 atomic adds, so their last bits may vary between runs. */
PISA_API size_t pisa_attn_backward_workspace_bytes(pisa_shape shape, pisa_params params);
/* The least scratch pisa_sparse_attn_backward runs with (no dS scratch); 0 where it refuses. */
PISA_API size_t pisa_attn_backward_min_workspace_bytes(pisa_shape shape, pisa_params params);
PISA_API pisa_status pisa_sparse_attn_backward(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                                               const int32_t* idx, const uint16_t* O, const float* LSE,
                                               const uint16_t* dO, float* dQ, float* dK, float* dV, void* ws,
                                               size_t ws_bytes, pisa_shape shape, pisa_params params,
                                               pisa_stream stream);

/* ---- full prefill from host buffers (end-to-end path) --------------------------------- */

/* Copies Q, K, V host -> device, builds the pyramid, selects, attends and copies O (and
 * LSE, idx when non-NULL) device -> host; returns when all of it has finished.  The work runs
 * in query chunks (at most 11: doubling from N/32 positions, at least 8192, up to N/4 and
 * halving again towards the end, equal chunks of at most N/4 between) so that the host -> device copy of the next
 * chunk's Q, the device -> host copy of the previous chunk's O and the attention of one chunk
 * overlap the selection of the next.  In causal mode each chunk's K rows go first: the keys
 * its selection can read (the summaries of the levels where more than K candidates can be
 * eligible, and the leaf pairs and blocks that start at or before its last position), with
 * the pyramid nodes over them built on a stream of their own while earlier chunks are
 * computed; V follows in the same chunks as Q, each extended to the end of the 64-key block of
 * its last position, since a chunk's attention reads no later block.  Otherwise K is copied
 * first and whole, and V whole after the first chunk's Q.  Selection runs on `stream`;
 * attention, the copies and the pyramid on four streams of the library's own (ordered after
 * the work queued on `stream` before the call), and all of them are idle again on return.  Results equal those of pisa_build_pyramid + pisa_select_prefill +
 * pisa_sparse_attn_prefill on the same inputs.  One call at a time per device (calls from
 * several threads are serialised).  Host buffers should be pinned for full copy bandwidth
 * and concurrent copies.  dev_ws is device scratch of at least
 * pisa_prefill_host_workspace_bytes().  N_cap must equal N. */
PISA_API size_t pisa_prefill_host_workspace_bytes(pisa_shape shape, pisa_params params);
/* The query chunks pisa_prefill_host uses for a sequence of N positions (host only, no device
 * work): writes the chunk bounds 0 = bounds[0] < bounds[1] < ... < bounds[n] = N into
 * bounds[0..n] and returns n (0 for N = 0, at most 16).  Returns -1, writing nothing, when
 * bounds is NULL, N < 0 or max_bounds < n + 1. */
PISA_API int pisa_prefill_host_chunks(long long N, long long* bounds, int max_bounds);
PISA_API pisa_status pisa_prefill_host(const uint16_t* Q_host, const uint16_t* K_host, const uint16_t* V_host,
                              uint16_t* O_host, float* LSE_host, int32_t* idx_host, void* dev_ws, size_t ws_bytes,
                              pisa_shape shape, pisa_params params, pisa_stream stream);

/* ---- step 3: decode ------------------------------------------------------------------- */

/* One decode step for every sequence b, in one fused kernel (summary page, step 3):
 * T = seq_len[b]; writes k, v at row T of the caches; recomputes leaf T/C from its raw
 * keys and every ancestor from its children (so Pc equals pisa_build_pyramid of the first
 * T+1 keys); selects for the query at T over T+1 tokens (level walk, exact leaf LSE,
 * top-K with the own block); attends; and advances seq_len[b] by one.
 *   q [B][H_q][d], k, v [B][H_kv][d] bf16 in;  Kc, Vc [B][H_kv][N_cap][d] and
 *   Pc [B][H_kv][nodes(N_cap)][d] bf16 in/out;  seq_len [B] int32 in/out (device), each
 *   entry < N_cap;  o [B][H_q][d] bf16 out;  lse [B][H_q] fp32 out, nullable;
 *   idx_out [B][H_kv][K] int32 out, nullable.  shape.N is ignored; shape.N_cap is required.
 * Causal mode only. */
PISA_API pisa_status pisa_decode_step(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                             uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out,
                             pisa_shape shape, pisa_params params, pisa_stream stream);
/* The same step with device scratch: ws (256-byte aligned, at least
 * pisa_decode_workspace_bytes() bytes, owned by the caller, not to be used by other work
 * until the step has run) keeps the exact leaf scoring's logits of every candidate block,
 * B * H_kv * 2K * 64 keys * G' heads fp32 (G' = G_Q up to 8, 16 above), and the attention takes the selected
 * blocks' logits from there instead of reading their K rows again.  The logits are the same
 * products in the same order, so o, lse and idx equal pisa_decode_step's bit for bit.
 * ws = NULL runs pisa_decode_step; ws_bytes below the size returns PISA_ERR_WORKSPACE.
 * pisa_decode_workspace_bytes returns 0 for arguments pisa_decode_step refuses. */
PISA_API size_t pisa_decode_workspace_bytes(pisa_shape shape, pisa_params params);
PISA_API pisa_status pisa_decode_step_ws(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc,
                                         uint16_t* Vc, uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse,
                                         int32_t* idx_out, void* ws, size_t ws_bytes, pisa_shape shape,
                                         pisa_params params, pisa_stream stream);

/* ---- status ---------------------------------------------------------------------------- */

PISA_API const char* pisa_status_string(pisa_status status);

/* Waits for `stream`, then returns and clears the current device's error word:
 * PISA_ERR_TIMEOUT if a bounded wait gave up, PISA_ERR_BAD_INDEX if an index was out of
 * range, PISA_OK otherwise (PISA_ERR_CUDA if the CUDA calls themselves fail). */
PISA_API pisa_status pisa_get_last_device_error(pisa_stream stream);

/* ---- per-phase device time (a profiling aid; the paper has no counterpart) --------------- */

/* While enabled, every compute entry point records a CUDA event on its stream when its work
 * starts and after each of its kernel phases: pyramid, Stage 1 (with the clustering histogram),
 * clustering, Stage 2 leaf LSE, top-K, sparse attention, BSA selection, decode step, attention
 * backward.  The records cost a few microseconds per call and add no ordering beyond the
 * stream's own.  Events are recorded on the device current at the call.
 * pisa_phase_timing(1) enables recording and clears the current device's totals; (0) disables
 * it (the totals are kept).  Returns PISA_ERR_CUDA if resolving earlier records failed.
 * pisa_phase_times waits for the current device's recorded events and writes, for each phase
 * i < n, the total milliseconds into ms[i] and the number of timed launches into count[i]
 * (either may be NULL).  Returns the number of phases, or -1 on a CUDA error.
 * pisa_phase_name returns a phase's name ("stage1", ...), or NULL past the last phase. */
PISA_API pisa_status pisa_phase_timing(int enable);
PISA_API int pisa_phase_times(double* ms, long long* count, int n);
PISA_API const char* pisa_phase_name(int phase);

/* ---- a check of the timeout path (no counterpart in the paper) ---------------------------- */

/* Launches one CTA that holds tensor memory and waits, through the same bounded waits every
 * kernel of the library uses, on an mbarrier that nothing completes.  Each wait gives up after
 * limit_ns (1 us to 10 s; otherwise PISA_ERR_INVALID_ARG, nothing launched), sets the device
 * error word, and the CTA frees its tensor memory and returns: pisa_get_last_device_error()
 * then reports PISA_ERR_TIMEOUT and the device stays usable.  Lets a caller or a test exercise
 * the timeout path without hanging a GPU.  Asynchronous on `stream`. */
PISA_API pisa_status pisa_check_wait_timeout(unsigned long long limit_ns, pisa_stream stream);

/* Library version string. */
PISA_API const char* pisa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PISA_H */
