// Compaction: gather the kept K/V rows of every (request, KV head) segment into dense
// buffers, on the un-replicated KV heads ("KVzip: Query-Agnostic KV Cache Compression
// with Context Reconstruction", §4.2; the result is the per-head variable-length cache
// that a variable-length decode kernel reads, §7.1).
//
// A row is 128 bf16 = 256 B.  A CTA moves 64 kept rows of one segment: every thread issues
// eight 16-byte asynchronous copies (global -> shared, no registers held while in flight),
// consecutive threads covering consecutive 16-byte pieces of a K row and then of its V
// row, so the shared block is laid out exactly like the destination.  The 64 output rows
// of K (and of V) are contiguous, so one bulk copy per side writes them from shared
// memory.  Sources are the contiguous cache or the block pool through the block table.
// Copies are bit-exact; a row whose index is out of range (or whose block-table entry is)
// is written as zeros and flagged in the status word, and a segment whose count and offset
// would place rows outside the outputs is skipped and flagged.
#include "internal.cuh"

namespace kvsel {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;                          // kept rows per CTA
constexpr int kPieces = kRows * 32;                // 16-byte pieces: 16 of K and 16 of V per row
constexpr int kPerThread = kPieces / kThreads;     // 8
constexpr int kSideBytes = kRows * 256;            // one side (K or V) of the block

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
               "l"(static_cast<unsigned long long>(__cvta_generic_to_global(src)))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// shared -> global bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// element offset of token i of (request b, head h), or -1 when i or its block is out of range
__device__ __forceinline__ long long src_elem(const CompactArgs& a, int b, int h, int n, int i) {
  if (i < 0 || i >= n) return -1;
  if (!a.src.paged) return b * a.stride_req + h * a.stride_head + static_cast<long long>(i) * a.stride_tok;
  const int bs = a.src.block_size;
  const int pb = __ldg(a.src.block_table + static_cast<size_t>(b) * a.src.max_blocks + i / bs);
  if (pb < 0 || pb >= a.src.num_blocks) return -1;
  return ((static_cast<long long>(pb) * bs + (i % bs)) * a.rq.H + h) * kHeadDim;
}

__global__ void __launch_bounds__(kThreads) compact_kernel(const CompactArgs a) {
  __shared__ __align__(128) uint8_t s_blk[2][kSideBytes];   // [K, V][64 rows][256 B]
  __shared__ long long s_src[kRows];
  const int seg = blockIdx.y;
  const int b = seg / a.rq.H, h = seg - (seg / a.rq.H) * a.rq.H;
  const int n = a.rq.n[b];
  int count = __ldg(a.counts + seg);
  const long long off = __ldg(a.offsets + seg);
  // the segment's output rows must lie inside the outputs (counts / offsets from the caller)
  if (count > 0 && (off < 0 || off + count > a.n_kept)) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, DEV_BAD_INDEX);
    count = 0;
  }
  for (int r0 = blockIdx.x * kRows; r0 < count; r0 += gridDim.x * kRows) {
    const int rows = min(kRows, count - r0);
    if (threadIdx.x < kRows) {
      long long e = -1;
      if (static_cast<int>(threadIdx.x) < rows) {
        e = src_elem(a, b, h, n, __ldg(a.idx + off + r0 + threadIdx.x));
        if (e < 0 && a.status) atomicOr(a.status, DEV_BAD_INDEX);
      }
      s_src[threadIdx.x] = e;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int pc = u * kThreads + threadIdx.x;
      const int row = pc >> 5, side = (pc >> 4) & 1, piece = pc & 15;
      if (row < rows) {
        uint8_t* dst = s_blk[side] + row * 256 + piece * 16;
        const long long e = s_src[row];
        if (e >= 0) {
          cp_async16(dst, (side ? a.v : a.k) + e + piece * 8);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();   // this thread's shared writes -> visible to the bulk copy
    __syncthreads();
    if (threadIdx.x == 0) {
      const long long o = (off + r0) * kHeadDim;
      bulk_store(a.k_out + o, s_blk[0], static_cast<uint32_t>(rows) * 256u);
      bulk_store(a.v_out + o, s_blk[1], static_cast<uint32_t>(rows) * 256u);
      bulk_commit();
      bulk_wait_all();   // the block is written before its buffer is refilled or the CTA ends
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_compact(const CompactArgs& a, int max_count, int num_sms, cudaStream_t st) {
  if (max_count <= 0) return cudaSuccess;
  (void)num_sms;
  const int segs = a.rq.B * a.rq.H;
  int gx = (max_count + kRows - 1) / kRows;
  if (gx > 65535) gx = 65535;
  compact_kernel<<<dim3(gx, segs), kThreads, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace kvsel
