// Partition of every (request, KV head) segment into its kept and evicted positions, with
// the rows of both sides written out bit-exact ("VestigeKV: The NoPE-MLA KV Cache Carries
// Its Own Eviction Signal in a Vestigial Branch", §4.1: eviction moves rows out of the hot
// cache into an archive and deletes nothing, so every position lands in exactly one of
// the two; the kept side is the per-head variable-length cache of "KVzip: Query-Agnostic
// KV Cache Compression with Context Reconstruction", §4.2, §7.1).
//
// One CTA takes 64 consecutive positions [i0, i0 + 64) of one segment.  Its kept entries
// are idx[lo, hi) of the segment's ascending list (two binary searches), so the positions
// before i0 hold lo kept and i0 - lo evicted entries: the tile's kept rows go to the
// contiguous output range starting at kept slot lo, its evicted rows to the one starting
// at evicted slot i0 - lo.  Each thread gathers 16-byte pieces of the tile's K and V rows
// into shared memory with asynchronous copies, placed so that the evicted rows come
// first and the kept rows after them; one bulk copy per side and kind then writes each
// contiguous range.  Every row of the cache is read once and written once.
//
// Checks: counts, offsets and the kept list are range-checked on the device.  A segment
// whose count or offset does not fit its buffers is skipped; a tile whose kept entries
// are not strictly ascending inside it, or whose output ranges would leave the segment's
// (a list that is not sorted), is skipped; both set DEV_BAD_INDEX in the status word.
// Nothing is read or written outside the caller's buffers either way.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;                          // positions per CTA
constexpr int kPerThread = kRows * 32 / kThreads;  // 16-byte pieces per thread (16 of K, 16 of V per row)

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
               "l"(static_cast<unsigned long long>(__cvta_generic_to_global(src)))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// First j in [0, c) with list[j] >= x (c when none), found by one warp: each round its 32
// lanes probe 32 evenly spaced entries of the remaining range and a ballot keeps the
// part that holds the answer, so a list of c entries takes about log32(c) rounds of
// loads.  The range shrinks every round, so the search ends for any list contents.
__device__ __forceinline__ int warp_lower_bound(const int32_t* list, int c, int x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = c;   // the answer lies in [lo, hi]
  while (lo < hi) {
    const int step = (hi - lo + 31) / 32;
    const int pos = lo + lane * step;
    const bool valid = pos < hi;
    const bool below = valid && __ldg(list + pos) < x;
    const unsigned ball = __ballot_sync(0xffffffffu, below);
    const int t = __popc(ball);
    if (t == 0) {
      hi = lo;
    } else {
      const int last = lo + (t - 1) * step;   // list[last] < x
      const int nxt = lo + t * step;           // first probe not below x, if any
      lo = last + 1;
      hi = min(hi, nxt);
    }
  }
  return lo;
}

// element offset of token i of (request b, head h), or -1 when its block is out of range
__device__ __forceinline__ long long row_elem(const PartitionArgs& a, int b, int h, int i) {
  if (!a.src.paged) return b * a.stride_req + h * a.stride_head + static_cast<long long>(i) * a.stride_tok;
  const int bs = a.src.block_size;
  const int lb = i / bs;
  if (lb >= a.src.max_blocks) return -1;
  const int pb = __ldg(a.src.block_table + static_cast<size_t>(b) * a.src.max_blocks + lb);
  if (pb < 0 || pb >= a.src.num_blocks) return -1;
  return ((static_cast<long long>(pb) * bs + (i % bs)) * a.rq.H + h) * kHeadDim;
}

__global__ void __launch_bounds__(kThreads) partition_kernel(const PartitionArgs a) {
  __shared__ __align__(128) uint8_t s_blk[2][kRows * 256];   // [K, V][slot][256 B]
  __shared__ long long s_src[kRows];
  __shared__ int s_slot[kRows];
  __shared__ int s_ok;
  const int seg = blockIdx.y;
  const int b = seg / a.rq.H, h = seg - b * a.rq.H;
  const int n = a.rq.n[b];
  const int i0 = blockIdx.x * kRows;
  const int c = __ldg(a.counts + seg);
  const long long off = __ldg(a.offsets + seg);
  // evicted entries of every earlier segment: the score positions before this segment
  // minus the kept entries before it (offsets is the exclusive prefix sum of counts)
  const long long ev_off = a.rq.soff[b] + static_cast<long long>(h) * n - off;
  const bool seg_ok = c >= 0 && c <= n && off >= 0 && off + c <= a.n_kept && ev_off >= 0 &&
                      ev_off + (n - c) <= a.n_evicted;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (seg_ok) {
      a.ev_counts[seg] = n - c;
      a.ev_offsets[seg] = ev_off;
    } else {
      if (a.status) atomicOr(a.status, DEV_BAD_INDEX);
      a.ev_counts[seg] = 0;
      a.ev_offsets[seg] = 0;
    }
  }
  if (!seg_ok || i0 >= n) return;
  const int m = min(kRows, n - i0);
  const int32_t* list = a.idx + off;
  __shared__ int s_lohi[2];
  __shared__ unsigned s_mask[2];
  const int warp = threadIdx.x >> 5;
  if (warp < 2) {
    const int r = warp_lower_bound(list, c, warp == 0 ? i0 : i0 + m);
    if ((threadIdx.x & 31) == 0) s_lohi[warp] = r;
  }
  if (threadIdx.x == 64) {
    s_ok = 1;
    s_mask[0] = s_mask[1] = 0u;
  }
  __syncthreads();
  const int lo = s_lohi[0], hi = s_lohi[1];
  // the tile's kept entries: at most m, strictly ascending, inside [i0, i0 + m)
  if (hi - lo > m || hi < lo) {
    if (threadIdx.x == 0) s_ok = 0;
  } else if (static_cast<int>(threadIdx.x) < hi - lo) {
    const int j = lo + threadIdx.x;
    const int x = __ldg(list + j);
    const bool asc = j == lo || __ldg(list + j - 1) < x;
    if (!asc || x < i0 || x >= i0 + m)
      s_ok = 0;
    else
      atomicOr(&s_mask[(x - i0) >> 5], 1u << ((x - i0) & 31));
  }
  __syncthreads();
  const unsigned long long kept = (static_cast<unsigned long long>(s_mask[1]) << 32) | s_mask[0];
  const int n_kept_t = __popcll(kept);
  const int n_ev_t = m - n_kept_t;
  // both output ranges of the tile inside the segment's (fails only for an unsorted list)
  if (!s_ok || lo > i0 || lo + n_kept_t > c || (i0 - lo) + n_ev_t > n - c) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, DEV_BAD_INDEX);
    return;
  }
  if (threadIdx.x < kRows) {
    const int p = threadIdx.x;
    long long e = -1;
    int slot = 0;
    if (p < m) {
      const unsigned long long below = kept & ((1ull << p) - 1ull);
      const int kr = __popcll(below);
      const bool is_kept = (kept >> p) & 1ull;
      // evicted rows first, kept rows after them, each in position order
      slot = is_kept ? n_ev_t + kr : p - kr;
      e = row_elem(a, b, h, i0 + p);
      if (e < 0 && a.status) atomicOr(a.status, DEV_BAD_INDEX);
      if (!is_kept) a.ev_idx[ev_off + (i0 - lo) + (p - kr)] = i0 + p;
    }
    s_src[p] = e;
    s_slot[p] = slot;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int pc = u * kThreads + threadIdx.x;
    const int p = pc >> 5, side = (pc >> 4) & 1, piece = pc & 15;
    if (p < m) {
      uint8_t* dst = s_blk[side] + s_slot[p] * 256 + piece * 16;
      const long long e = s_src[p];
      if (e >= 0)
        cp_async16(dst, (side ? a.v : a.k) + e + piece * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  cp_async_wait_all();
  fence_proxy_async_smem();   // this thread's shared writes -> visible to the bulk copies
  __syncthreads();
  if (threadIdx.x == 0) {
    if (n_ev_t > 0) {
      const long long o = (ev_off + (i0 - lo)) * kHeadDim;
      bulk_store(a.k_ev + o, s_blk[0], static_cast<uint32_t>(n_ev_t) * 256u);
      bulk_store(a.v_ev + o, s_blk[1], static_cast<uint32_t>(n_ev_t) * 256u);
    }
    if (n_kept_t > 0 && a.k_kept) {
      const long long o = (off + lo) * kHeadDim;
      bulk_store(a.k_kept + o, s_blk[0] + n_ev_t * 256, static_cast<uint32_t>(n_kept_t) * 256u);
      bulk_store(a.v_kept + o, s_blk[1] + n_ev_t * 256, static_cast<uint32_t>(n_kept_t) * 256u);
    }
    bulk_commit();
    bulk_wait_all();   // the shared block is read before the CTA ends
  }
}

}  // namespace

cudaError_t launch_partition(const PartitionArgs& a, int n_max, cudaStream_t st) {
  const int segs = a.rq.B * a.rq.H;
  const int gx = n_max > 0 ? (n_max + kRows - 1) / kRows : 1;
  if (segs <= 0) return cudaSuccess;
  partition_kernel<<<dim3(gx, segs), kThreads, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
