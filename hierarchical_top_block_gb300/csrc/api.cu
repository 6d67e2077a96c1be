// C ABI of the PISA library (declared in include/pisa.h): argument checks, workspace
// carving, per-device state and the launch sequence of each entry point.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "../../include/pisa.h"
#include "kernels.cuh"

namespace pisa {

// One error word per device: kernels OR ERR_* bits into it; the host reads and clears it.
static __device__ uint32_t g_device_error;

namespace {

constexpr int MAX_DEVICES = 64;

// Streams and events of the host-buffer prefill pipeline (created on first use).
constexpr int PIPE_MAX_CHUNKS = 16;
constexpr int PIPE_EVENTS = 4 + 6 * PIPE_MAX_CHUNKS;

struct HostPipe {
  bool ready = false;
  std::mutex run;                                    // one host-buffer prefill at a time per device
  cudaStream_t in = nullptr, out = nullptr;          // host->device and device->host copies
  cudaStream_t attn = nullptr;                       // attention of chunk j beside selection of j+1
  cudaStream_t pyr = nullptr;                        // pyramid over each chunk's key slice (causal)
  cudaEvent_t ev[PIPE_EVENTS] = {};
};

// Query chunks of the host-buffer prefill.  The chunks double from N/32 (at least 8192
// queries) up to a quarter of the sequence and halve again at the end, with equal chunks of at
// most N/4 between: a short first chunk shortens the copy-in that precedes any compute, and
// the halving tail keeps each chunk's copy-out shorter than the compute of the chunks after
// it, so only the last, small copy-out trails the compute.  Bounds are multiples of 64 except
// where the remainder of a ragged N falls; at most 11 chunks.
int plan_chunks(long long N, long long* bounds) {
  long long lo = N / 32 / 64 * 64;
  if (lo < 8192) lo = 8192;
  long long cap = N / 4 / 64 * 64;
  if (cap < lo) cap = lo;
  long long ramp[8];
  int nr = 0;
  long long used = 0;
  for (long long c = lo; c < cap && used + 2 * c <= N && nr < 6; c *= 2) {
    ramp[nr++] = c;
    used += 2 * c;
  }
  const long long mid = N - used;
  long long nm = mid > 0 ? (mid + cap - 1) / cap : 0;
  if (nm > PIPE_MAX_CHUNKS - 2 * nr) nm = PIPE_MAX_CHUNKS - 2 * nr;
  int n = 0;
  long long t = 0;
  bounds[0] = 0;
  for (int i = 0; i < nr; ++i) bounds[++n] = (t += ramp[i]);
  for (long long i = 1; i < nm; ++i) bounds[++n] = t + mid * i / nm / 64 * 64;
  t += mid;
  if (nm > 0) bounds[++n] = t;
  for (int i = nr - 1; i >= 0; --i) bounds[++n] = (t += ramp[i]);
  return n;
}

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  uint32_t* err = nullptr;  // device address of g_device_error on this device
  HostPipe pipe;
};

std::mutex g_mutex;
DeviceState g_dev[MAX_DEVICES];

// ---- per-phase device time (profiling aid) ------------------------------------------------
// While enabled, each entry point records a CUDA event on its stream at the start of its work
// and after each kernel phase; pisa_phase_times() resolves the events and sums the phases.
enum Phase { PH_PYRAMID, PH_STAGE1, PH_CLUSTER, PH_LEAF_LSE, PH_TOPK, PH_ATTN, PH_BSA, PH_DECODE, PH_BACKWARD, NPHASE };
const char* const PHASE_NAMES[NPHASE] = {"pyramid", "stage1", "cluster", "leaf_lse", "topk",
                                         "sparse_attn", "bsa_select", "decode", "attn_backward"};

std::atomic<bool> g_timing{false};

struct PhaseRec {
  int phase;
  cudaEvent_t a, b;
  bool own_a;  // a opens a chain (else it is the previous record's b)
};
struct PhaseLog {
  std::vector<cudaEvent_t> pool;
  std::vector<PhaseRec> pending;
  double ms[NPHASE] = {};
  long long count[NPHASE] = {};
};
PhaseLog g_phase[MAX_DEVICES];  // guarded by g_mutex

cudaEvent_t take_event(PhaseLog& log) {
  if (!log.pool.empty()) {
    cudaEvent_t e = log.pool.back();
    log.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}

// Records the phases of one entry point's launch sequence on one stream (a no-op unless
// timing is enabled).
class PhaseTimer {
 public:
  explicit PhaseTimer(cudaStream_t s) : s_(s) {
    if (!g_timing.load(std::memory_order_relaxed)) return;
    if (cudaGetDevice(&dev_) != cudaSuccess || dev_ < 0 || dev_ >= MAX_DEVICES) return;
    std::lock_guard<std::mutex> lock(g_mutex);
    last_ = take_event(g_phase[dev_]);
    if (last_ && cudaEventRecord(last_, s_) != cudaSuccess) {
      g_phase[dev_].pool.push_back(last_);
      last_ = nullptr;
    }
  }
  void mark(int phase) {
    if (!last_) return;
    std::lock_guard<std::mutex> lock(g_mutex);
    PhaseLog& log = g_phase[dev_];
    cudaEvent_t e = take_event(log);
    if (!e) return;
    if (cudaEventRecord(e, s_) != cudaSuccess) {
      log.pool.push_back(e);
      return;
    }
    log.pending.push_back(PhaseRec{phase, last_, e, first_});
    first_ = false;
    last_ = e;
  }
  ~PhaseTimer() {
    if (last_ && first_) {  // opened but no phase recorded: return the start event
      std::lock_guard<std::mutex> lock(g_mutex);
      g_phase[dev_].pool.push_back(last_);
    }
  }

 private:
  cudaStream_t s_;
  int dev_ = -1;
  cudaEvent_t last_ = nullptr;
  bool first_ = true;
};

// Waits for the pending records of device dev and adds them to its totals (g_mutex held).
bool resolve_phases(PhaseLog& log) {
  bool ok = true;
  for (const PhaseRec& r : log.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      ok = false;
      continue;
    }
    log.ms[r.phase] += ms;
    log.count[r.phase] += 1;
  }
  for (const PhaseRec& r : log.pending) {
    log.pool.push_back(r.b);
    if (r.own_a) log.pool.push_back(r.a);
  }
  log.pending.clear();
  return ok;
}

// Per-device set-up, done once per device with that device current.
pisa_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PISA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PISA_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return PISA_ERR_CUDA;
    st.err = static_cast<uint32_t*>(p);
    st.ready = true;
  }
  *out = &st;
  return PISA_OK;
}

pisa_status host_pipe(DeviceState* st, HostPipe** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  HostPipe& hp = st->pipe;
  if (!hp.ready) {
    if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess) return PISA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess) return PISA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&hp.attn, cudaStreamNonBlocking) != cudaSuccess) return PISA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&hp.pyr, cudaStreamNonBlocking) != cudaSuccess) return PISA_ERR_CUDA;
    for (cudaEvent_t& e : hp.ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return PISA_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return PISA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// level sizes for n tokens (C = 64, g = 2); offsets from the capacity layout
Geometry make_geometry(long long n, long long n_cap) {
  Geometry g{};
  g.L = 0;
  long long m = (n + 63) / 64;
  if (n > 0) {
    g.M[1] = (int)m;
    g.L = 1;
    while (m > 1 && g.L < MAX_LEVELS) {
      m = (m + 1) / 2;
      g.M[++g.L] = (int)m;
    }
  }
  long long mc = (n_cap + 63) / 64, off = 0;
  int l = 1;
  if (n_cap > 0) {
    while (true) {
      g.off[l] = off;
      off += mc;
      if (mc <= 1 || l >= MAX_LEVELS) break;
      mc = (mc + 1) / 2;
      ++l;
    }
  }
  g.nodes = off;
  return g;
}

// Keys [0, x) that the causal selection and attention of queries t < T read, x returned.  The
// level walk reads the child summaries of a level-l candidate (l >= 2: 2^(l+5) keys, starting at
// or before t) only at levels where more than K candidates can be eligible, i.e. where
// ((T - 1) >> (l + 5)) + 1 > K; Stage 2 reads the 128 keys of level-2 nodes that start at or before
// t, and the attention the 64-key blocks that do.  So x is the end of the last eligible node at
// the highest level with more than K of them, or of the last eligible level-2 node.
long long causal_key_prefix(long long T, int Ksel, const Geometry& g, long long N) {
  if (T <= 0) return 0;
  long long x = (((T - 1) >> 7) + 1) << 7;
  for (int l = 2; l <= g.L - 1; ++l) {  // the levels the walk may score
    const long long cnt = ((T - 1) >> (l + 5)) + 1;
    if (cnt > Ksel) x = std::max(x, cnt << (l + 5));
  }
  return std::min(x, N);
}

pisa_status check_params(const pisa_shape& s, const pisa_params& pr, Problem* p) {
  if (s.B < 0 || s.N < 0 || s.H_q <= 0 || s.H_kv <= 0 || s.d <= 0) return PISA_ERR_INVALID_ARG;
  if (pr.C != 64 || pr.g != 2 || (s.d != 64 && s.d != 128)) return PISA_ERR_UNSUPPORTED;
  if (pr.K < 1 || pr.K > 32) return PISA_ERR_UNSUPPORTED;  // a query's 2K candidates fit two per lane
  if (pr.causal != 0 && pr.causal != 1) return PISA_ERR_INVALID_ARG;
  if (pr.scoring < 0 || pr.scoring > 2) return PISA_ERR_INVALID_ARG;
  if (s.H_q % s.H_kv != 0) return PISA_ERR_INVALID_ARG;
  const int gq = s.H_q / s.H_kv;
  if (gq != 1 && gq != 2 && gq != 4 && gq != 8 && gq != 16) return PISA_ERR_UNSUPPORTED;
  const long long ncap = s.N_cap == 0 ? s.N : s.N_cap;
  if (ncap < s.N) return PISA_ERR_INVALID_ARG;
  if (ncap >= (1LL << 25)) return PISA_ERR_UNSUPPORTED;                        // entry packing (t << 6)
  if ((long long)s.B * ncap * s.H_q >= (1LL << 31)) return PISA_ERR_UNSUPPORTED;  // TMA coordinates
  if (!(pr.scale == pr.scale)) return PISA_ERR_INVALID_ARG;
  p->B = s.B;
  p->N = s.N;
  p->N_cap = (int)ncap;
  p->H_q = s.H_q;
  p->H_kv = s.H_kv;
  p->d = s.d;
  p->C = pr.C;
  p->g = pr.g;
  p->K = pr.K;
  p->causal = pr.causal;
  p->scoring = pr.scoring;
  p->scale = pr.scale > 0.f ? pr.scale : 1.0f / sqrtf((float)s.d);
  p->GQ = gq;
  p->t_lo = 0;
  p->t_hi = s.N;
  return PISA_OK;
}

struct SelectLayout {
  size_t s2, score, counts, offsets, tile_off, block_sums, entries, tiles, totals, total_bytes;
  ClusterBuffers cb;  // sizes only; pointers filled by carve()
};

SelectLayout select_layout(const Problem& p) {
  SelectLayout L{};
  const long long total = (long long)p.B * p.H_kv * p.N;
  const Geometry g = make_geometry(p.N, p.N);
  const int rpq = p.GQ < 8 ? 8 : p.GQ;
  ClusterBuffers& cb = L.cb;
  cb.qt = 128 / rpq;
  long long win = (32LL << 20) / ((long long)p.GQ * p.d * 2);
  win = win / 64 * 64;
  if (win < 64) win = 64;
  if (win > p.N) win = p.N > 0 ? p.N : 1;
  cb.win = (int)win;
  cb.nwin = p.N > 0 ? (int)((p.N + win - 1) / win) : 1;
  cb.M2 = g.L >= 2 ? g.M[2] : 1;
  cb.nkeys = (long long)p.B * p.H_kv * cb.nwin * cb.M2;
  cb.nblocks = (int)((cb.nkeys + 4095) / 4096);
  if (cb.nblocks < 1) cb.nblocks = 1;
  cb.max_tiles = total * p.K / cb.qt + cb.nkeys + 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  L.s2 = take(sizeof(int32_t) * total * p.K);
  L.score = take(sizeof(float) * total * 2 * p.K);
  L.counts = take(sizeof(int32_t) * (cb.nkeys + 1));  // the histogram, then Stage 1's item counter
  L.offsets = take(sizeof(int32_t) * cb.nkeys);
  L.tile_off = take(sizeof(int32_t) * cb.nkeys);
  L.block_sums = take(sizeof(int32_t) * 2 * cb.nblocks);
  L.entries = take(sizeof(int32_t) * total * p.K);
  L.tiles = take(sizeof(int4) * cb.max_tiles);
  L.totals = take(sizeof(int32_t) * 4);
  L.total_bytes = o;
  return L;
}

pisa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PISA_OK : PISA_ERR_CUDA; }

// The selection's clustering lists and the backward's block -> queries lists hold up to
// B * H_kv * N * K entries and address them with 32-bit offsets; the selection's tile
// offsets are 32-bit as well.
bool entry_lists_fit(const Problem& p) {
  if ((long long)p.B * p.H_kv * p.N * p.K >= (1LL << 31)) return false;
  return select_layout(p).cb.max_tiles < (1LL << 31);
}

// counts_zero: the scratch's histogram and Stage 1's item counter are zero already (Stage 2 of a
// selection over the same scratch leaves them so), and the memset before Stage 1 is skipped.
pisa_status run_select(const uint16_t* Q, const uint16_t* K, const uint16_t* P, int32_t* idx, float* leaf_score,
                       int32_t* s2, void* ws, size_t ws_bytes, const Problem& p, DeviceState* st, cudaStream_t s,
                       bool counts_zero = false) {
  if (!entry_lists_fit(p)) return PISA_ERR_UNSUPPORTED;
  SelectLayout L = select_layout(p);
  if (ws_bytes < L.total_bytes) return PISA_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* S2 = s2 ? s2 : reinterpret_cast<int32_t*>(w + L.s2);
  float* score = leaf_score ? leaf_score : reinterpret_cast<float*>(w + L.score);
  ClusterBuffers cb = L.cb;
  cb.counts = reinterpret_cast<int32_t*>(w + L.counts);
  cb.sched = cb.counts + cb.nkeys;
  cb.rank = reinterpret_cast<int32_t*>(score);  // list places, until Stage 2 writes the scores
  cb.offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  cb.tile_off = reinterpret_cast<int32_t*>(w + L.tile_off);
  cb.block_sums = reinterpret_cast<int32_t*>(w + L.block_sums);
  cb.entries = reinterpret_cast<int32_t*>(w + L.entries);
  cb.tiles = reinterpret_cast<int4*>(w + L.tiles);
  cb.totals = reinterpret_cast<int32_t*>(w + L.totals);
  const Geometry geo = make_geometry(p.N, p.N);
  PhaseTimer tm(s);
  if (!counts_zero && cudaMemsetAsync(cb.counts, 0, sizeof(int32_t) * (cb.nkeys + 1), s) != cudaSuccess)
    return PISA_ERR_CUDA;
  if (launch_stage1(Q, P, S2, cb, p, geo, st->num_sms, st->err, s) != cudaSuccess) return PISA_ERR_CUDA;
  tm.mark(PH_STAGE1);
  if (launch_cluster(S2, cb, p, s) != cudaSuccess) return PISA_ERR_CUDA;
  tm.mark(PH_CLUSTER);
  if (launch_leaf_lse(Q, K, cb, score, p, geo, st->num_sms, st->err, s) != cudaSuccess) return PISA_ERR_CUDA;
  tm.mark(PH_LEAF_LSE);
  if (launch_topk(S2, score, idx, p, geo, st->num_sms, s) != cudaSuccess) return PISA_ERR_CUDA;
  tm.mark(PH_TOPK);
  return PISA_OK;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pisa

using namespace pisa;

extern "C" {

int pisa_pyramid_levels(long long N, int C, int g) {
  if (N <= 0 || C <= 0 || g < 2) return 0;
  long long m = (N + C - 1) / C;
  int L = 1;
  while (m > 1) {
    m = (m + g - 1) / g;
    ++L;
  }
  return L;
}

long long pisa_pyramid_nodes(long long N, int C, int g) {
  if (N <= 0 || C <= 0 || g < 2) return 0;
  long long m = (N + C - 1) / C, s = m;
  while (m > 1) {
    m = (m + g - 1) / g;
    s += m;
  }
  return s;
}

size_t pisa_select_workspace_bytes(pisa_shape shape, pisa_params params) {
  Problem p;
  if (check_params(shape, params, &p) != PISA_OK || !entry_lists_fit(p)) return 0;
  return select_layout(p).total_bytes;
}

pisa_status pisa_build_pyramid(const uint16_t* K, uint16_t* P, pisa_shape shape, pisa_params params,
                               pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!K || !P || !aligned16(K) || !aligned16(P)) return PISA_ERR_INVALID_ARG;
  const Geometry geo = make_geometry(p.N, p.N_cap);
  PhaseTimer tm(static_cast<cudaStream_t>(stream));
  const cudaError_t e = launch_pyramid(K, P, p, geo, static_cast<cudaStream_t>(stream));
  tm.mark(PH_PYRAMID);
  return cuda_status(e);
}

pisa_status pisa_select_prefill(const uint16_t* Q, const uint16_t* K, const uint16_t* P, int32_t* idx,
                                float* leaf_score, int32_t* s2, void* ws, size_t ws_bytes, pisa_shape shape,
                                pisa_params params, pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.N_cap != p.N) return PISA_ERR_INVALID_ARG;
  if (!entry_lists_fit(p)) return PISA_ERR_UNSUPPORTED;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!Q || !K || !P || !idx || !ws) return PISA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(P) || (reinterpret_cast<uintptr_t>(ws) & 255u)) return PISA_ERR_INVALID_ARG;
  if ((leaf_score && !aligned16(leaf_score)) || (s2 && !aligned16(s2)) || !aligned16(idx)) return PISA_ERR_INVALID_ARG;
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  return run_select(Q, K, P, idx, leaf_score, s2, ws, ws_bytes, p, st, static_cast<cudaStream_t>(stream));
}

pisa_status pisa_sparse_attn_prefill(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                     uint16_t* O, float* LSE, pisa_shape shape, pisa_params params,
                                     pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!Q || !K || !V || !idx || !O) return PISA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(idx)) return PISA_ERR_INVALID_ARG;
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  PhaseTimer tm(static_cast<cudaStream_t>(stream));
  const cudaError_t e = launch_sparse_attn(Q, K, V, idx, O, LSE, p, st->num_sms, st->err, static_cast<cudaStream_t>(stream));
  tm.mark(PH_ATTN);
  return cuda_status(e);
}

// The BSA selection's query parts are addressed with 32-bit TMA row coordinates
// (B * H_kv * 2 * N rows) and the summary rows likewise (B * H_kv * nodes).
bool bsa_fits(const Problem& p) {
  const long long bh = (long long)p.B * p.H_kv;
  return bh * 2 * p.N < (1LL << 31) && bh * pisa_pyramid_nodes(p.N, 64, 2) < (1LL << 31);
}

size_t pisa_select_bsa_workspace_bytes(pisa_shape shape, pisa_params params) {
  Problem p;
  if (check_params(shape, params, &p) != PISA_OK || !bsa_fits(p)) return 0;
  return round_up(bsa_workspace_bytes(p), 256);
}

pisa_status pisa_select_bsa(const uint16_t* Q, const uint16_t* P, int32_t* idx, void* ws, size_t ws_bytes,
                            pisa_shape shape, pisa_params params, pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.N_cap != p.N) return PISA_ERR_INVALID_ARG;
  if (!bsa_fits(p)) return PISA_ERR_UNSUPPORTED;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!Q || !P || !idx || !ws) return PISA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(P) || !aligned16(idx) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return PISA_ERR_INVALID_ARG;
  if (ws_bytes < bsa_workspace_bytes(p)) return PISA_ERR_WORKSPACE;
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  const Geometry geo = make_geometry(p.N, p.N);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PhaseTimer tm(s);
  const cudaError_t e = launch_bsa_select(Q, P, idx, ws, p, geo, st->num_sms, st->err, s);
  tm.mark(PH_BSA);
  return cuda_status(e);
}

size_t pisa_attn_backward_workspace_bytes(pisa_shape shape, pisa_params params) {
  Problem p;
  if (check_params(shape, params, &p) != PISA_OK || !entry_lists_fit(p)) return 0;
  return attn_backward_workspace_bytes(p, true);
}

size_t pisa_attn_backward_min_workspace_bytes(pisa_shape shape, pisa_params params) {
  Problem p;
  if (check_params(shape, params, &p) != PISA_OK || !entry_lists_fit(p)) return 0;
  return attn_backward_workspace_bytes(p, false);
}

pisa_status pisa_sparse_attn_backward(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                                      const uint16_t* O, const float* LSE, const uint16_t* dO, float* dQ, float* dK,
                                      float* dV, void* ws, size_t ws_bytes, pisa_shape shape, pisa_params params,
                                      pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (!entry_lists_fit(p)) return PISA_ERR_UNSUPPORTED;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!Q || !K || !V || !idx || !O || !LSE || !dO || !dQ || !dK || !dV || !ws) return PISA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV) || ((uintptr_t)ws & 255))
    return PISA_ERR_INVALID_ARG;
  if (ws_bytes < attn_backward_workspace_bytes(p, false)) return PISA_ERR_WORKSPACE;
  const bool with_ds = ws_bytes >= attn_backward_workspace_bytes(p, true);
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  PhaseTimer tm(static_cast<cudaStream_t>(stream));
  const cudaError_t e = launch_attn_backward(Q, K, V, idx, O, LSE, dO, dQ, dK, dV, ws, with_ds, p, st->num_sms,
                                             st->err, static_cast<cudaStream_t>(stream));
  tm.mark(PH_BACKWARD);
  return cuda_status(e);
}

int pisa_prefill_host_chunks(long long N, long long* bounds, int max_bounds) {
  if (!bounds || N < 0) return -1;
  long long b[PIPE_MAX_CHUNKS + 1];
  const int n = plan_chunks(N, b);
  if (max_bounds < n + 1) return -1;
  for (int i = 0; i <= n; ++i) bounds[i] = b[i];
  return n;
}

size_t pisa_prefill_host_workspace_bytes(pisa_shape shape, pisa_params params) {
  Problem p;
  if (check_params(shape, params, &p) != PISA_OK || !entry_lists_fit(p)) return 0;
  const size_t q = (size_t)p.B * p.N * p.H_q * p.d * 2;
  const size_t kv = (size_t)p.B * p.H_kv * p.N * p.d * 2;
  const size_t pyr = (size_t)p.B * p.H_kv * pisa_pyramid_nodes(p.N, 64, 2) * p.d * 2;
  const size_t idx = (size_t)p.B * p.H_kv * p.N * p.K * 4;
  const size_t lse = (size_t)p.B * p.H_q * p.N * 4;
  return round_up(q, 256) * 2 + round_up(kv, 256) * 2 + round_up(pyr, 256) + round_up(idx, 256) + round_up(lse, 256) +
         select_layout(p).total_bytes;
}

pisa_status pisa_prefill_host(const uint16_t* Q_host, const uint16_t* K_host, const uint16_t* V_host,
                              uint16_t* O_host, float* LSE_host, int32_t* idx_host, void* dev_ws, size_t ws_bytes,
                              pisa_shape shape, pisa_params params, pisa_stream stream) {
  Problem p;
  pisa_status rc = check_params(shape, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.N_cap != p.N) return PISA_ERR_INVALID_ARG;
  if (!entry_lists_fit(p)) return PISA_ERR_UNSUPPORTED;
  if (p.B == 0 || p.N == 0) return PISA_OK;
  if (!Q_host || !K_host || !V_host || !O_host || !dev_ws) return PISA_ERR_INVALID_ARG;
  if (ws_bytes < pisa_prefill_host_workspace_bytes(shape, params)) return PISA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(dev_ws) & 255u) return PISA_ERR_INVALID_ARG;
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  HostPipe* hp;
  if ((rc = host_pipe(st, &hp)) != PISA_OK) return rc;
  std::lock_guard<std::mutex> hold(hp->run);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t q = (size_t)p.B * p.N * p.H_q * p.d * 2;
  const size_t kv = (size_t)p.B * p.H_kv * p.N * p.d * 2;
  const size_t pyr = (size_t)p.B * p.H_kv * pisa_pyramid_nodes(p.N, 64, 2) * p.d * 2;
  const size_t idxb = (size_t)p.B * p.H_kv * p.N * p.K * 4;
  const size_t lseb = (size_t)p.B * p.H_q * p.N * 4;
  uint8_t* w = static_cast<uint8_t*>(dev_ws);
  uint16_t* dQ = reinterpret_cast<uint16_t*>(w);
  w += round_up(q, 256);
  uint16_t* dO = reinterpret_cast<uint16_t*>(w);
  w += round_up(q, 256);
  uint16_t* dK = reinterpret_cast<uint16_t*>(w);
  w += round_up(kv, 256);
  uint16_t* dV = reinterpret_cast<uint16_t*>(w);
  w += round_up(kv, 256);
  uint16_t* dP = reinterpret_cast<uint16_t*>(w);
  w += round_up(pyr, 256);
  int32_t* dIdx = reinterpret_cast<int32_t*>(w);
  w += round_up(idxb, 256);
  float* dL = reinterpret_cast<float*>(w);
  w += round_up(lseb, 256);
  const size_t sel_bytes = select_layout(p).total_bytes;

  // Query chunks: selection and attention of chunk j need Q rows of chunk j only (plus K, and
  // V up to the chunk's last position when causal), so the copy-in of chunk j+1 and the
  // copy-out of chunk j-1 overlap the compute of chunk j; attention of chunk j (its own
  // stream) also overlaps selection of chunk j+1, which fills the tail of each persistent
  // kernel with the next one's CTAs.  When causal, each chunk's K rows come first: those below
  // the prefix its selection reads (causal_key_prefix; the last chunk's slice ends at N), and a
  // fourth stream builds the pyramid nodes that meet the slice while the chunks before are
  // computed (none of them reads those nodes: each meets keys past their prefixes); then the
  // chunk's Q rows and the V rows up to the end of the 64-key block that holds its last
  // position (the attention of chunk j reads V rows of blocks that start at or before its
  // positions, and no further).  Without causality every node is eligible: K goes whole and
  // first, the pyramid follows on `stream`, and V goes whole after Q0.
  // The two share only idx, whose rows of different chunks are disjoint; selection scratch
  // is reused from chunk to chunk in the order of `stream`.  Q and O are [B][N][H_q][d]: a
  // chunk is one row band per sequence.
  long long bounds[PIPE_MAX_CHUNKS + 1];
  const int nchunks = plan_chunks(p.N, bounds);
  cudaEvent_t* ev = hp->ev;
  cudaEvent_t e_start = ev[0], e_k = ev[1], e_v = ev[2], e_end = ev[3];
  cudaEvent_t* e_q = ev + 4;
  cudaEvent_t* e_sel = ev + 4 + PIPE_MAX_CHUNKS;
  cudaEvent_t* e_attn = ev + 4 + 2 * PIPE_MAX_CHUNKS;
  cudaEvent_t* e_vs = ev + 4 + 3 * PIPE_MAX_CHUNKS;  // V rows of chunks 0..j in place (causal)
  cudaEvent_t* e_ks = ev + 4 + 4 * PIPE_MAX_CHUNKS;  // K rows below kpre[j + 1] in place (causal)
  cudaEvent_t* e_py = ev + 4 + 5 * PIPE_MAX_CHUNKS;  // pyramid nodes below kpre[j + 1] exact (causal)
  const Geometry geo = make_geometry(p.N, p.N);
  long long kpre[PIPE_MAX_CHUNKS + 1];  // chunk j reads keys [0, kpre[j + 1])
  kpre[0] = 0;
  for (int j = 0; j < nchunks; ++j)
    kpre[j + 1] = j + 1 == nchunks ? p.N : std::max(kpre[j], causal_key_prefix(bounds[j + 1], p.K, geo, p.N));
  const size_t q_row = (size_t)p.H_q * p.d * 2;  // bytes of one query position, all heads
  auto copy_q = [&](int j) {
    const long long lo = bounds[j], hi = bounds[j + 1];
    return cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(dQ) + lo * q_row, p.N * q_row,
                             reinterpret_cast<const uint8_t*>(Q_host) + lo * q_row, p.N * q_row, (hi - lo) * q_row, p.B,
                             cudaMemcpyHostToDevice, hp->in);
  };
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // the library's streams start after whatever the caller queued on `stream` before this call
  chk(cudaEventRecord(e_start, s));
  chk(cudaStreamWaitEvent(hp->in, e_start, 0));
  chk(cudaStreamWaitEvent(hp->attn, e_start, 0));
  chk(cudaStreamWaitEvent(hp->pyr, e_start, 0));
  const size_t kv_row = (size_t)p.d * 2;  // bytes of one key position of one KV head
  auto copy_v = [&](long long lo, long long hi) {  // positions lo .. hi - 1 of every (b, h_kv)
    return cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(dV) + lo * kv_row, p.N * kv_row,
                             reinterpret_cast<const uint8_t*>(V_host) + lo * kv_row, p.N * kv_row, (hi - lo) * kv_row,
                             (size_t)p.B * p.H_kv, cudaMemcpyHostToDevice, hp->in);
  };
  auto copy_k = [&](long long lo, long long hi) {  // positions lo .. hi - 1 of every (b, h_kv)
    return cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(dK) + lo * kv_row, p.N * kv_row,
                             reinterpret_cast<const uint8_t*>(K_host) + lo * kv_row, p.N * kv_row, (hi - lo) * kv_row,
                             (size_t)p.B * p.H_kv, cudaMemcpyHostToDevice, hp->in);
  };
  if (!p.causal) {
    chk(cudaMemcpyAsync(dK, K_host, kv, cudaMemcpyHostToDevice, hp->in));
    chk(cudaEventRecord(e_k, hp->in));
  }
  for (int j = 0; j < nchunks && ok; ++j) {
    if (p.causal) {
      if (kpre[j + 1] > kpre[j]) chk(copy_k(kpre[j], kpre[j + 1]));
      chk(cudaEventRecord(e_ks[j], hp->in));
    }
    chk(copy_q(j));
    chk(cudaEventRecord(e_q[j], hp->in));
    if (p.causal) {
      auto block_end = [&](long long t) { return std::min<long long>((long long)p.N, (t + 63) / 64 * 64); };
      chk(copy_v(block_end(bounds[j]), block_end(bounds[j + 1])));
      chk(cudaEventRecord(e_vs[j], hp->in));
    } else if (j == 0) {
      chk(cudaMemcpyAsync(dV, V_host, kv, cudaMemcpyHostToDevice, hp->in));
      chk(cudaEventRecord(e_v, hp->in));
    }
  }
  if (p.causal) {
    for (int j = 0; j < nchunks && ok; ++j) {
      chk(cudaStreamWaitEvent(hp->pyr, e_ks[j], 0));
      if (ok) chk(launch_pyramid_range(dK, dP, p, geo, kpre[j], kpre[j + 1], hp->pyr));
      chk(cudaEventRecord(e_py[j], hp->pyr));
    }
  } else {
    chk(cudaStreamWaitEvent(s, e_k, 0));
    if (ok) chk(launch_pyramid(dK, dP, p, geo, s));
  }
  if (!p.causal) chk(cudaStreamWaitEvent(hp->attn, e_v, 0));
  for (int j = 0; j < nchunks && ok; ++j) {
    Problem pc = p;
    pc.t_lo = (int)bounds[j];
    pc.t_hi = (int)bounds[j + 1];
    if (p.causal) chk(cudaStreamWaitEvent(s, e_py[j], 0));
    chk(cudaStreamWaitEvent(s, e_q[j], 0));
    if (!ok) break;
    // after the first chunk the histogram is zero: the previous chunk's Stage 2 left it so
    if ((rc = run_select(dQ, dK, dP, dIdx, nullptr, nullptr, w, sel_bytes, pc, st, s, j > 0)) != PISA_OK) {
      ok = false;
      break;
    }
    chk(cudaEventRecord(e_sel[j], s));
    chk(cudaStreamWaitEvent(hp->attn, e_sel[j], 0));
    if (p.causal) chk(cudaStreamWaitEvent(hp->attn, e_vs[j], 0));
    if (ok) chk(launch_sparse_attn(dQ, dK, dV, dIdx, dO, dL, pc, st->num_sms, st->err, hp->attn));
    chk(cudaEventRecord(e_attn[j], hp->attn));
    // copy-out of chunk j: O rows, and the LSE / selection columns of every head
    const size_t nq = (size_t)(pc.t_hi - pc.t_lo), t0 = (size_t)pc.t_lo;
    chk(cudaStreamWaitEvent(hp->out, e_attn[j], 0));
    chk(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(O_host) + t0 * q_row, p.N * q_row,
                          reinterpret_cast<const uint8_t*>(dO) + t0 * q_row, p.N * q_row, nq * q_row, p.B,
                          cudaMemcpyDeviceToHost, hp->out));
    if (LSE_host)
      chk(cudaMemcpy2DAsync(LSE_host + t0, (size_t)p.N * 4, dL + t0, (size_t)p.N * 4, nq * 4, (size_t)p.B * p.H_q,
                            cudaMemcpyDeviceToHost, hp->out));
    if (idx_host)
      chk(cudaMemcpy2DAsync(idx_host + t0 * p.K, (size_t)p.N * p.K * 4, dIdx + t0 * p.K, (size_t)p.N * p.K * 4,
                            nq * p.K * 4, (size_t)p.B * p.H_kv, cudaMemcpyDeviceToHost, hp->out));
  }
  // the call returns once all four streams are idle (also after an error, so that no copy
  // is still writing into the caller's buffers)
  const cudaError_t e_rec = cudaEventRecord(e_end, hp->out);
  if (e_rec == cudaSuccess) cudaStreamWaitEvent(s, e_end, 0);
  const cudaError_t e_in = cudaStreamSynchronize(hp->in), e_at = cudaStreamSynchronize(hp->attn);
  const cudaError_t e_py_sync = cudaStreamSynchronize(hp->pyr);
  const cudaError_t e_out = cudaStreamSynchronize(hp->out), e_s = cudaStreamSynchronize(s);
  if (rc != PISA_OK) return rc;
  if (!ok || e_rec != cudaSuccess || e_in != cudaSuccess || e_at != cudaSuccess || e_out != cudaSuccess ||
      e_s != cudaSuccess || e_py_sync != cudaSuccess)
    return PISA_ERR_CUDA;
  return PISA_OK;
}

size_t pisa_decode_workspace_bytes(pisa_shape shape, pisa_params params) {
  pisa_shape sh = shape;
  if (sh.N_cap <= 0) return 0;
  sh.N = 0;
  Problem p;
  if (check_params(sh, params, &p) != PISA_OK || p.causal != 1) return 0;
  return decode_logits_bytes(p);
}

pisa_status pisa_decode_step(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                             uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out,
                             pisa_shape shape, pisa_params params, pisa_stream stream) {
  return pisa_decode_step_ws(q, k, v, Kc, Vc, Pc, seq_len, o, lse, idx_out, nullptr, 0, shape, params, stream);
}

pisa_status pisa_decode_step_ws(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* Kc, uint16_t* Vc,
                                uint16_t* Pc, int32_t* seq_len, uint16_t* o, float* lse, int32_t* idx_out, void* ws,
                                size_t ws_bytes, pisa_shape shape, pisa_params params, pisa_stream stream) {
  pisa_shape sh = shape;
  if (sh.N_cap <= 0) return PISA_ERR_INVALID_ARG;
  sh.N = 0;
  Problem p;
  pisa_status rc = check_params(sh, params, &p);
  if (rc != PISA_OK) return rc;
  if (p.causal != 1) return PISA_ERR_UNSUPPORTED;
  if (p.B == 0) return PISA_OK;
  if (ws) {
    if (ws_bytes < decode_logits_bytes(p)) return PISA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return PISA_ERR_INVALID_ARG;
  }
  if (!q || !k || !v || !Kc || !Vc || !Pc || !seq_len || !o) return PISA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(Pc) ||
      !aligned16(o))
    return PISA_ERR_INVALID_ARG;
  DeviceState* st;
  if ((rc = device_state(&st)) != PISA_OK) return rc;
  const Geometry geo_cap = make_geometry(p.N_cap, p.N_cap);
  PhaseTimer tm(static_cast<cudaStream_t>(stream));
  const cudaError_t e =
      launch_decode(q, k, v, Kc, Vc, Pc, seq_len, o, lse, idx_out, static_cast<float*>(ws), p, geo_cap, st->err,
                    static_cast<cudaStream_t>(stream));
  tm.mark(PH_DECODE);
  return cuda_status(e);
}

pisa_status pisa_check_wait_timeout(unsigned long long limit_ns, pisa_stream stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return PISA_ERR_INVALID_ARG;
  DeviceState* st;
  pisa_status rc = device_state(&st);
  if (rc != PISA_OK) return rc;
  return cuda_status(launch_wait_check(limit_ns, st->err, static_cast<cudaStream_t>(stream)));
}

const char* pisa_status_string(pisa_status status) {
  switch (status) {
    case PISA_OK: return "ok";
    case PISA_ERR_INVALID_ARG: return "invalid argument";
    case PISA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case PISA_ERR_CUDA: return "CUDA runtime error";
    case PISA_ERR_TIMEOUT: return "a bounded device wait timed out";
    case PISA_ERR_BAD_INDEX: return "a selected block index was out of range";
    case PISA_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

pisa_status pisa_get_last_device_error(pisa_stream stream) {
  DeviceState* st;
  pisa_status rc = device_state(&st);
  if (rc != PISA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&word, g_device_error, sizeof(word), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PISA_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PISA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PISA_ERR_CUDA;
  if (word & ERR_TIMEOUT) return PISA_ERR_TIMEOUT;
  if (word & ERR_BAD_INDEX) return PISA_ERR_BAD_INDEX;
  return PISA_OK;
}

pisa_status pisa_phase_timing(int enable) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PISA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  PhaseLog& log = g_phase[dev];
  const bool ok = resolve_phases(log);
  for (int i = 0; i < NPHASE; ++i) {
    log.ms[i] = 0.0;
    log.count[i] = 0;
  }
  g_timing.store(enable != 0);
  return ok ? PISA_OK : PISA_ERR_CUDA;
}

int pisa_phase_times(double* ms, long long* count, int n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1;
  std::lock_guard<std::mutex> lock(g_mutex);
  PhaseLog& log = g_phase[dev];
  if (!resolve_phases(log)) return -1;
  for (int i = 0; i < n && i < NPHASE; ++i) {
    if (ms) ms[i] = log.ms[i];
    if (count) count[i] = log.count[i];
  }
  return NPHASE;
}

const char* pisa_phase_name(int phase) { return phase >= 0 && phase < NPHASE ? PHASE_NAMES[phase] : nullptr; }

const char* pisa_version(void) { return "pisa-gb300 0.1 (sm_103a)"; }

}  // extern "C"
