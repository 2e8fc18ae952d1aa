// kvsel_score_noalloc: the scoring entry point for callers that cannot allocate device
// memory.  Its scratch space is a fixed buffer that lives in the library itself (a
// file-scope __device__ array), so the call needs nothing from the caller beyond the
// inputs and outputs.
//
// Who needs it: processes whose device memory is owned by an arena or caching allocator
// (serving engines commonly reserve nearly all HBM for their KV-cache pool up front, so a
// side cudaMalloc may fail or fragment that pool), and code paths that must not
// allocate because cudaMalloc/cudaFree can synchronise the device and stall pipelines
// that are otherwise fully asynchronous.
//
// Costs and rules: every GPU that loads the library holds KVSEL_NOALLOC_SCRATCH_BYTES of
// device memory for this buffer until the process exits.  All calls share the one buffer
// and it keeps the previous call's contents; each call clears the part that must start at
// zero (the device status word) and fully rewrites the rest before reading it.  Calls whose
// GPU work overlaps (different streams, or different host threads, on one device) race on
// the buffer: serialise them.  The first call on each device looks up the buffer's device
// address with that device current; make that first call before any stream capture.
#include <mutex>

#include "../../include/kvsel.h"
#include "internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KVSEL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device (the host-side symbol is
// only a stand-in and must never be handed to a kernel).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVSEL_ECUDA;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVSEL_ECUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return KVSEL_OK;
}

}  // namespace

extern "C" int kvsel_score_noalloc(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o,
                                   float* s_attn, float* s_val, void* stream) {
  size_t need = 0;
  int rc = kvsel_workspace_size(p, &need);
  if (rc) return rc;
  if (need > KVSEL_NOALLOC_SCRATCH_BYTES) return KVSEL_EWORKSPACE;
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch))) return rc;
  // the status word and the barrier counters start at zero for this call; everything else
  // is rewritten
  if (cudaMemsetAsync(scratch, 0, kvsel::kStatusBytes + kvsel::kCounterBytes, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KVSEL_ECUDA;
  return kvsel_score(p, q, kv, w_o, s_attn, s_val, scratch, KVSEL_NOALLOC_SCRATCH_BYTES, stream);
}
