// Throughput of the exponential unit (MUFU ex2.approx.ftz.f32) on this GPU, for the
// benchmark's rooflines: the exponential-bound parts of the path (window scoring, the
// query-agnostic row log-sum-exp) are reported against a measured rate rather than an
// assumed one.  A measurement tool beside bench.py, not part of libkvsel; built into
// libkvsel_ex2probe.so by the package's build step.
//
// One CTA of 512 threads per SM; every thread runs eight independent chains
// x <- -2^x - 1/4, which stay in [-1.25, -0.25], so each step is one ex2 and one FMA and
// the compiler cannot fold any of them.  The rate is the ex2 count over the CTAs' own
// clock64 spans (per clock per SM) and over CUDA-event time (per second, whole device).
#include <cuda_runtime.h>

#include <cstdint>

#include <vector>

namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 8;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kProbeThreads, 1)
    ex2_probe_kernel(int iters, float* sink, unsigned long long* cycles) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = -0.25f - 0.01f * static_cast<float>(c + (threadIdx.x & 7));
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = fmaf(ex2_approx(x[c]), -1.f, -0.25f);
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c];
  if (s == 12345.f) sink[blockIdx.x] = s;   // never true; keeps the chains live
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
}

}  // namespace

// Runs the probe for about a millisecond on the current device's legacy default stream.
//   scratch         device, 16-byte aligned, at least 16 * (number of SMs) bytes
//   per_clk_per_sm  host out: ex2 results per SM clock per SM (the CTAs' cycle counts)
//   per_second      host out: ex2 results per second over the device (CUDA events)
// Returns 0, or -1 for bad arguments, -4 for a short scratch, -5 for a CUDA error.
// Synchronises the device.
extern "C" int kvsel_probe_ex2_rate(void* scratch, size_t scratch_bytes, double* per_clk_per_sm, double* per_second) {
  if (!scratch || !per_clk_per_sm || !per_second || (reinterpret_cast<uintptr_t>(scratch) & 15u)) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return -5;
  if (scratch_bytes < 16u * static_cast<size_t>(sms)) return -4;
  constexpr int kIters = 4096;
  auto* cycles = static_cast<unsigned long long*>(scratch);
  auto* sink = reinterpret_cast<float*>(cycles + sms);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int rc = -5;
  std::vector<unsigned long long> host(static_cast<size_t>(sms));
  float ms = 0.f;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) goto done;
  ex2_probe_kernel<<<sms, kProbeThreads>>>(kIters / 8, sink, cycles);   // warm-up
  if (cudaGetLastError() != cudaSuccess || cudaEventRecord(e0, nullptr) != cudaSuccess) goto done;
  ex2_probe_kernel<<<sms, kProbeThreads>>>(kIters, sink, cycles);
  if (cudaGetLastError() != cudaSuccess) goto done;
  if (cudaEventRecord(e1, nullptr) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess) goto done;
  if (cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.f) goto done;
  if (cudaMemcpy(host.data(), cycles, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost) != cudaSuccess)
    goto done;
  {
    unsigned long long cmax = 1;
    for (unsigned long long c : host) cmax = c > cmax ? c : cmax;
    const double per_cta = static_cast<double>(kProbeThreads) * kChains * kIters;
    *per_clk_per_sm = per_cta / static_cast<double>(cmax);
    *per_second = per_cta * sms / (static_cast<double>(ms) * 1e-3);
    rc = 0;
  }
done:
  if (rc != 0) cudaGetLastError();
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  return rc;
}
