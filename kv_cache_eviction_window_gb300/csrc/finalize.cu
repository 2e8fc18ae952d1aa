// Pooling along the sequence and the value-aware combination
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 2: maxpooling of
//  the reduced window attention (SnapKV); Algorithm 1: (A + eps) * ||V W^O||_1 with
//  eps = 1e-4, footnote 3).
//
// One thread per score.  Window of key i: [i - k/2, i + k/2] clipped to [0, n); max
// pooling ignores positions outside, average pooling counts them as zeros and divides
// by k.  The data is a few MiB per layer and stays in L2 after the scoring pass.
#include "internal.cuh"

namespace kvsel {
namespace {

__global__ void finalize_kernel(const ReqTable rq, const float* __restrict__ s_raw, const float* __restrict__ nu,
                                float* __restrict__ s_attn, float* __restrict__ s_val, int pool, int kernel,
                                float eps) {
  const int seg = blockIdx.y;
  const int b = seg / rq.H, h = seg - (seg / rq.H) * rq.H;
  const int n = rq.n[b];
  const size_t base = static_cast<size_t>(rq.soff[b]) + static_cast<size_t>(h) * n;
  const int half = kernel / 2;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float p;
    if (pool == 1 && half > 0) {
      p = s_raw[base + i];
      const int lo = max(0, i - half), hi = min(n - 1, i + half);
      for (int j = lo; j <= hi; ++j) p = fmaxf(p, s_raw[base + j]);
    } else if (pool == 2 && half > 0) {
      float acc = 0.f;
      const int lo = max(0, i - half), hi = min(n - 1, i + half);
      for (int j = lo; j <= hi; ++j) acc += s_raw[base + j];
      p = acc / static_cast<float>(kernel);
    } else {
      p = s_raw[base + i];
    }
    s_attn[base + i] = p;
    if (s_val) s_val[base + i] = (p + eps) * nu[base + i];
  }
}

}  // namespace

cudaError_t launch_finalize(const ReqTable& rq, const float* s_raw, const float* nu, float* s_attn, float* s_val,
                            int pool, int pool_kernel, float eps, cudaStream_t st) {
  int nmax = 0;
  for (int b = 0; b < rq.B; ++b) nmax = rq.n[b] > nmax ? rq.n[b] : nmax;
  if (nmax == 0) return cudaSuccess;
  const int threads = 256;
  int gx = (nmax + threads - 1) / threads;
  if (gx > 1024) gx = 1024;
  finalize_kernel<<<dim3(gx, rq.B * rq.H), threads, 0, st>>>(rq, s_raw, nu, s_attn, s_val, pool, pool_kernel, eps);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
