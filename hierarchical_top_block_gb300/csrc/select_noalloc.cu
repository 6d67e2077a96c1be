// Block selection for callers that cannot allocate device memory.
//
// pisa_select_prefill needs a scratch buffer (candidate lists, leaf scores, clustering
// lists and tiles) that the caller allocates.  Some callers cannot do that: code running
// under a memory pool they do not own, plugins of a host that hands out no allocator, or
// code that must not call cudaMalloc between setup and a latency-critical loop.  For them
// this file keeps one scratch array in device global memory, of fixed size (32 MiB) and
// reserved when the module loads on a device, and runs the same selection kernels on it.
//
// Facts a caller has to know:
//   - The array is SCRATCH_BYTES (32 MiB) on every GPU that loads this library, held until
//     the process exits.  Problems whose selection scratch is larger are rejected with
//     PISA_ERR_WORKSPACE before anything is launched (pisa_select_workspace_bytes gives
//     the size a shape needs; about 18 bytes per (b, h_kv, t, K) entry plus small tables).
//   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
//     with that device current; make that first call before any stream capture.
//   - Every call uses the same array and leaves its contents behind; the selection clears
//     the parts that must start at zero itself.  Calls whose work overlaps on the GPU (two
//     streams, or two host threads without ordering) race on the array: serialise them.
//   - Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <mutex>

#include "../../include/pisa.h"
#include "kernels.cuh"

namespace {

constexpr size_t SCRATCH_BYTES = size_t(32) << 20;
constexpr int MAX_DEVICES = 64;

// The name is only a host-side stand-in; kernels get the address looked up below.
static __device__ __align__(256) uint8_t g_select_scratch[SCRATCH_BYTES];

std::mutex g_lock;
void* g_scratch_addr[MAX_DEVICES] = {};

pisa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PISA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_lock);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return PISA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PISA_OK;
}

}  // namespace

extern "C" pisa_status pisa_select_prefill_noalloc(const uint16_t* Q, const uint16_t* K, const uint16_t* P,
                                                   int32_t* idx, float* leaf_score, int32_t* s2, pisa_shape shape,
                                                   pisa_params params, pisa_stream stream) {
  const size_t need = pisa_select_workspace_bytes(shape, params);
  // no workspace size (an argument the selection refuses: it returns its own status before
  // launching anything) or an empty problem (a no-op that touches no device)
  if (need == 0 || (long long)shape.B * shape.N <= 0) return pisa_select_prefill(Q, K, P, idx, leaf_score, s2, nullptr, 0, shape, params, stream);
  if (need > SCRATCH_BYTES) return PISA_ERR_WORKSPACE;
  void* ws = nullptr;
  pisa_status rc = scratch_address(&ws);
  if (rc != PISA_OK) return rc;
  return pisa_select_prefill(Q, K, P, idx, leaf_score, s2, ws, SCRATCH_BYTES, shape, params, stream);
}
