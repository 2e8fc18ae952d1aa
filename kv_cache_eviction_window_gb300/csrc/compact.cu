// Compaction: gather the kept K/V rows of every (request, KV head) segment into dense
// buffers, on the un-replicated KV heads ("KVzip: Query-Agnostic KV Cache Compression
// with Context Reconstruction", §4.2; the result is the per-head variable-length cache
// that a variable-length decode kernel reads, §7.1).
//
// A row is 128 bf16 = 256 B: 16 lanes move one row with 16-byte loads/stores, so a warp
// copies two K rows and two V rows per step.  Sources are the contiguous cache or the
// block pool through the block table.  Copies are bit-exact.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 128;

constexpr int kRowsInFlight = 4;   // rows per 16-lane group per step (loads issued before stores)

__device__ __forceinline__ bool src_row(const CompactArgs& a, int b, int h, int n, int i, const uint4*& ks,
                                        const uint4*& vs) {
  if (i < 0 || i >= n) return false;
  long long e;
  if (!a.src.paged) {
    e = b * a.stride_req + h * a.stride_head + static_cast<long long>(i) * a.stride_tok;
  } else {
    const int bs = a.src.block_size;
    const int pb = __ldg(a.src.block_table + static_cast<size_t>(b) * a.src.max_blocks + i / bs);
    if (pb < 0 || pb >= a.src.num_blocks) return false;
    e = ((static_cast<long long>(pb) * bs + (i % bs)) * a.rq.H + h) * kHeadDim;
  }
  ks = reinterpret_cast<const uint4*>(a.k + e);
  vs = reinterpret_cast<const uint4*>(a.v + e);
  return true;
}

__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
  const int seg = blockIdx.y;
  const int b = seg / a.rq.H, h = seg - (seg / a.rq.H) * a.rq.H;
  const int n = a.rq.n[b];
  const int count = __ldg(a.counts + seg);
  const long long off = __ldg(a.offsets + seg);
  const int grp = threadIdx.x >> 4;         // 16 groups of 16 lanes; a group moves whole rows
  const int part = threadIdx.x & 15;        // 16-byte piece of a 256-byte row
  constexpr int kGroups = kThreads / 16;
  for (int r0 = blockIdx.x * kRowsPerBlock; r0 < count; r0 += gridDim.x * kRowsPerBlock) {
    const int rend = min(count, r0 + kRowsPerBlock);
    for (int rb = r0 + grp * kRowsInFlight; rb < rend; rb += kGroups * kRowsInFlight) {
      uint4 kv[kRowsInFlight], vv[kRowsInFlight];
      bool ok[kRowsInFlight];
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        const int r = rb + u;
        ok[u] = false;
        if (r < rend) {
          const uint4 *ks, *vs;
          ok[u] = src_row(a, b, h, n, __ldg(a.idx + off + r), ks, vs);
          if (ok[u]) {
            kv[u] = __ldcs(ks + part);
            vv[u] = __ldcs(vs + part);
          } else if (a.status && part == 0) {
            atomicOr(a.status, DEV_BAD_INDEX);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        if (ok[u]) {
          const long long o = (off + rb + u) * kHeadDim;
          __stcs(reinterpret_cast<uint4*>(a.k_out + o) + part, kv[u]);
          __stcs(reinterpret_cast<uint4*>(a.v_out + o) + part, vv[u]);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, int max_count, int num_sms, cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  const int segs = a.rq.B * a.rq.H;
  int gx = (max_count + kRowsPerBlock - 1) / kRowsPerBlock;
  // about 8 blocks per SM over all segments
  const int want = (num_sms * 8 + segs - 1) / segs;
  if (gx > want) gx = want > 0 ? want : 1;
  compact_kernel<<<dim3(gx, segs), kThreads, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
