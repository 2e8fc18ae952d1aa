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
// zero (the device status word and the grid-barrier counters) and fully rewrites the rest
// before reading it.  Calls whose GPU work overlaps (different streams, or different host
// threads, on one device) race on the buffer: serialise them.
//
// The host-side name of the array is only a stand-in, never a device address.  Every call
// made outside stream capture looks the address up with cudaGetSymbolAddress in the
// calling thread's current context and records it for that context; a call under stream
// capture uses the recorded address (one call per context must come before any capture).
// Looking it up again on every uncaptured call keeps the address right after the context
// is destroyed and re-created (cudaDeviceReset), which may give the new context the same
// handle as the old one.
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "../../include/kvsel.h"
#include "internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KVSEL_NOALLOC_SCRATCH_BYTES];

std::mutex g_addr_mutex;
std::map<CUcontext, void*> g_addr;   // device address of the buffer, per context

// The calling thread's current context, through the runtime's driver entry point (the
// library links no libcuda).  nullptr when it cannot be queried.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  CUcontext ctx = nullptr;
  if (fn && fn(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  return ctx;
}

}  // namespace

namespace kvsel {

// Device address of the built-in buffer in the current context (see the file comment).
int noalloc_scratch_address(cudaStream_t st, void** out) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return KVSEL_ECUDA;
  if (cs != cudaStreamCaptureStatusNone) {
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    auto it = g_addr.find(ctx);
    if (it == g_addr.end()) return KVSEL_ECUDA;   // no uncaptured call in this context yet
    *out = it->second;
    return KVSEL_OK;
  }
  // the lookup also initialises the runtime's context on this thread's device
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVSEL_ECUDA;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  g_addr[ctx] = p;
  *out = p;
  return KVSEL_OK;
}

}  // namespace kvsel

extern "C" int kvsel_score_noalloc(const kvsel_params* p, const void* q, const kvsel_kv* kv, const void* w_o,
                                   float* s_attn, float* s_val, void* stream) {
  size_t need = 0;
  int rc = kvsel_workspace_size(p, &need);
  if (rc) return rc;
  if (need > KVSEL_NOALLOC_SCRATCH_BYTES) return KVSEL_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if ((rc = kvsel::noalloc_scratch_address(st, &scratch))) return rc;
  // the status word and the barrier counters start at zero for this call; everything else
  // is rewritten
  if (cudaMemsetAsync(scratch, 0, kvsel::kStatusBytes + kvsel::kCounterBytes, st) != cudaSuccess) return KVSEL_ECUDA;
  return kvsel_score(p, q, kv, w_o, s_attn, s_val, scratch, KVSEL_NOALLOC_SCRATCH_BYTES, stream);
}
