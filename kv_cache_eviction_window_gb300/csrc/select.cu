// Top-B selection with forced entries, on one thread-block cluster per segment
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 1 (two stages:
//  b' = floor(alpha*b) by attention, the rest by the value-aware criterion) and
//  Algorithm 2 (Top_k of the pooled score); "KVzip: Query-Agnostic KV Cache Compression
//  with Context Reconstruction", §4.2 (top r% across all heads of a layer)).
//
// A segment is one (request, KV head) in per-head mode, or all heads of one request
// flattened head-major in per-layer mode.  The CTAs of a cluster split the segment into
// contiguous chunks held in shared memory as order-preserving 32-bit keys (forced
// entries get the largest key).  The B-th largest key T is found by a four-pass radix
// select (8-bit digits): each pass builds per-CTA histograms of the candidates,
// the cluster reduces them through distributed shared memory, and every CTA finds the
// same digit.  Entries with key > T, and the first (B - #greater) entries equal to T in
// index order, are kept; a cluster-wide exclusive scan of per-CTA counts plus a block
// scan gives each kept entry its output slot, so indices come out ascending.
#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <tuple>

#include "internal.cuh"

namespace cgx = cooperative_groups;

namespace kvsel {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;        // 8-bit digits, four passes
constexpr uint32_t kKeyMax = 0xFFFFFFFFu;
constexpr int kMaxHeads = 64;
constexpr int kMaxHalo = 64;   // room for 2 * (pool_kernel / 2) staged neighbours of a chunk
static_assert(kBins <= kThreads && kBins % 32 == 0, "digit search: one bin per thread");

__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
  uint32_t whist[kWarps][kBins];  // per-warp histograms of the current pass (no cross-warp atomics)
  uint32_t merged[3][kBins];      // cluster-wide histogram, pushed by every CTA; one buffer per pass mod 3
  uint32_t cnt[2][16][2];     // (greater, equal) counts of every CTA, pushed by each; one buffer per selection mod 2
  uint32_t res_prefix, res_krem, res_bin;
  uint32_t wsum_gt[kWarps], wsum_eq[kWarps];
  uint32_t head_cnt[kMaxHeads];
};

// Address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void red_add_cluster(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// The two halves of a cluster barrier, so that independent work can run between them.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// 4-byte global -> shared copy that does not hold a register while in flight
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
               "l"(static_cast<unsigned long long>(__cvta_generic_to_global(src)))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int kBatch = 8;   // entries per thread whose global loads are issued together

// Block-wide exclusive scan of two counters (one pair per thread).
__device__ __forceinline__ void block_excl_scan2(SelShared& S, uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb,
                                                 uint32_t& ta, uint32_t& tb) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o);
    const uint32_t xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) {
    S.wsum_gt[w] = ia;
    S.wsum_eq[w] = ib;
  }
  __syncthreads();
  uint32_t pa = 0, pb = 0, sa = 0, sb = 0;
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) {
      pa += S.wsum_gt[i];
      pb += S.wsum_eq[i];
    }
    sa += S.wsum_gt[i];
    sb += S.wsum_eq[i];
  }
  ea = pa + ia - a;
  eb = pb + ib - b;
  ta = sa;
  tb = sb;
  __syncthreads();
}

// Per-kernel pass / selection counters (identical in every CTA of the cluster), used to
// rotate the shared-memory buffers that other CTAs write or read.
struct SelState {
  int pass = 0;
  int sel = 0;
};

// Key T of the K-th largest candidate among keys[0, cnt_local) of every CTA, and the
// number of keys equal to T that are taken (krem).  Each pass: per-warp histograms of the
// keys that match the digits found so far (plain shared atomics, contention only inside a
// warp), summed per bin; every CTA adds its non-empty bins into every CTA's copy of the
// cluster histogram with cluster-scope reductions (at most 256 per CTA and pass); after
// one cluster barrier each CTA finds the same digit in its own shared memory.
__device__ void radix_select(cgx::cluster_group& cl, SelShared& S, SelState& st, const uint32_t* keys,
                             int cnt_local, uint32_t K, uint32_t& T, uint32_t& krem_out) {
  const unsigned CS = cl.num_blocks();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t prefix = 0, mask = 0, krem = K;
  if (K == 0) {   // nothing to take (same in every CTA of the cluster)
    T = kKeyMax;
    krem_out = 0;
    return;
  }
  uint32_t* my_hist = S.whist[w];
  // S.whist is all zero on entry and on exit: the thread that sums a bin clears it
  for (int pass = 0; pass < 4; ++pass, ++st.pass) {
    const int buf = st.pass % 3, nxt = (st.pass + 1) % 3;
    const int sh = 24 - 8 * pass;
    // kBatch keys loaded before their atomics, so the loads overlap
    for (int e0 = 0; e0 < cnt_local; e0 += kBatch * kThreads) {
      uint32_t k[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads + threadIdx.x;
        k[u] = e < cnt_local ? keys[e] : 0u;   // out-of-range slots are skipped below
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads + threadIdx.x;
        if (e < cnt_local && (k[u] & mask) == prefix) atomicAdd(&my_hist[(k[u] >> sh) & 0xFFu], 1u);
      }
    }
    __syncthreads();
    if (threadIdx.x < kBins) {
      uint32_t c = 0;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        c += S.whist[ww][threadIdx.x];
        S.whist[ww][threadIdx.x] = 0;
      }
      // the next pass's cluster buffer was last read two cluster barriers ago; remote
      // CTAs add into it only after the barrier below
      S.merged[nxt][threadIdx.x] = 0;
      if (c)
        for (unsigned r = 0; r < CS; ++r) red_add_cluster(cluster_addr(&S.merged[buf][threadIdx.x], r), c);
    }
    cl.sync();
    if (w == 0) {
      // one warp finds the digit: lane l holds bins [8l, 8l + 8); bins of higher lanes and
      // higher slots hold larger keys
      const uint4 b0 = *reinterpret_cast<const uint4*>(&S.merged[buf][8 * lane]);
      const uint4 b1 = *reinterpret_cast<const uint4*>(&S.merged[buf][8 * lane + 4]);
      const uint32_t v[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      uint32_t tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) tot += v[j];
      uint32_t incl = tot;   // keys in the bins of lanes [lane, 32)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += x;
      }
      uint32_t above = incl - tot;   // keys in bins above this lane's
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        if (above < krem && krem <= above + v[j]) {   // exactly one (lane, j) holds the krem-th largest
          S.res_prefix = prefix | (static_cast<uint32_t>(8 * lane + j) << sh);
          S.res_krem = krem - above;
          S.res_bin = v[j];
        }
        above += v[j];
      }
    }
    __syncthreads();
    prefix = S.res_prefix;
    krem = S.res_krem;
    mask |= 0xFFu << sh;
    if (krem == S.res_bin && prefix != 0u) {
      // every key of the threshold bin is taken (after the last pass: every key equal to
      // the threshold): the selection is all keys >= prefix, i.e. keys > prefix - 1 with
      // no ties to resolve (the same decision in every CTA)
      ++st.pass;
      T = prefix - 1u;
      krem_out = 0;
      return;
    }
  }
  T = prefix;
  krem_out = krem;
}

// Walk the local chunk [lo_local, hi_local) in index order and visit every kept entry
// with its slot in the segment-wide ascending order: `visit(e_local, slot)`.  Each warp
// owns a contiguous run of the chunk and reads it lane-interleaved; ranks come from
// ballots, so shared-memory reads are conflict-free and slots are assigned in order.
template <typename Visit>
__device__ void apply_selection(cgx::cluster_group& cl, SelShared& S, SelState& st, const uint32_t* keys,
                                int lo_local, int hi_local, uint32_t T, uint32_t krem, Visit visit) {
  const unsigned CS = cl.num_blocks();
  const unsigned rank = cl.block_rank();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int sb = st.sel & 1;
  ++st.sel;
  const int cnt = max(hi_local - lo_local, 0);
  const int per_w = ((cnt + kWarps - 1) / kWarps + 31) & ~31;
  const int wa = lo_local + min(cnt, w * per_w);
  const int wb = lo_local + min(cnt, (w + 1) * per_w);
  uint32_t ngt = 0, neq = 0;
  for (int e0 = wa; e0 < wb; e0 += 32 * kBatch) {
    uint32_t k[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + 32 * u + lane;
      k[u] = e < wb ? keys[e] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + 32 * u + lane;
      ngt += __popc(__ballot_sync(0xffffffffu, e < wb && k[u] > T));
      neq += __popc(__ballot_sync(0xffffffffu, e < wb && k[u] == T));
    }
  }
  // per-warp totals -> exclusive prefix over warps (lane 0 of each warp contributes)
  uint32_t egt, eeq, tgt, teq;
  block_excl_scan2(S, lane == 0 ? ngt : 0u, lane == 0 ? neq : 0u, egt, eeq, tgt, teq);
  egt = __shfl_sync(0xffffffffu, egt, 0);
  eeq = __shfl_sync(0xffffffffu, eeq, 0);
  if (threadIdx.x < CS) {
    st_cluster(cluster_addr(&S.cnt[sb][rank][0], threadIdx.x), tgt);
    st_cluster(cluster_addr(&S.cnt[sb][rank][1], threadIdx.x), teq);
  }
  cl.sync();
  // exclusive prefix over lower-ranked CTAs (lane c holds CTA c's counts)
  uint32_t g = 0, q = 0;
  if (lane < static_cast<int>(rank)) {
    g = S.cnt[sb][lane][0];
    q = S.cnt[sb][lane][1];
  }
  uint32_t qincl = q;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, qincl, o);
    if (lane >= o) qincl += x;
  }
  const uint32_t qexcl = qincl - q;
  const uint32_t avail = krem > qexcl ? krem - qexcl : 0u;
  uint32_t sel = g + (q < avail ? q : avail);
  uint32_t qs = q;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sel += __shfl_xor_sync(0xffffffffu, sel, o);
    qs += __shfl_xor_sync(0xffffffffu, qs, o);
  }
  (void)CS;
  // equals of earlier CTAs and earlier warps come first
  uint32_t eq_rank = qs + eeq;
  const uint32_t avail_w = krem > qs ? krem - qs : 0u;
  uint32_t slot = sel + egt + (eeq < avail_w ? eeq : avail_w);
  for (int e0 = wa; e0 < wb; e0 += 32 * kBatch) {
    uint32_t k[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + 32 * u + lane;
      k[u] = e < wb ? keys[e] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + 32 * u + lane;
      const bool gt = e < wb && k[u] > T;
      const bool eq = e < wb && k[u] == T;
      const unsigned meq = __ballot_sync(0xffffffffu, eq);
      const bool take = gt || (eq && eq_rank + __popc(meq & lt) < krem);
      const unsigned mtake = __ballot_sync(0xffffffffu, take);
      if (take) visit(e, slot + __popc(mtake & lt));
      slot += __popc(mtake);
      eq_rank += __popc(meq);
    }
  }
  __syncthreads();   // visits (flags, counters) are complete before the caller reads them
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const SelectArgs a, int chunk_cap) {
  cgx::cluster_group cl = cgx::this_cluster();
  extern __shared__ uint8_t smem_raw[];
  SelShared& S = *reinterpret_cast<SelShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(SelShared) + 15) & ~static_cast<size_t>(15)));
  uint8_t* flag = reinterpret_cast<uint8_t*>(keys + chunk_cap + kMaxHalo);

  const unsigned CS = cl.num_blocks();
  const unsigned rank = cl.block_rank();
  const int seg = blockIdx.y;
  const int H = a.rq.H;
  const bool per_layer = (a.mode == 1);
  const int b = per_layer ? seg : seg / H;
  const int h0 = per_layer ? 0 : seg % H;
  const int n = a.rq.n[b];
  const int L = per_layer ? H * n : n;
  const long long sbase = a.rq.soff[b] + (per_layer ? 0 : static_cast<long long>(h0) * n);
  const int cl_len = (L + static_cast<int>(CS) - 1) / static_cast<int>(CS);
  const int c_lo = min(L, static_cast<int>(rank) * cl_len);
  const int c_hi = min(L, c_lo + cl_len);
  const int cnt = c_hi - c_lo;
  const int ns = a.n_sink, nr = a.n_recent;
  const int nforced = min(n, ns + nr);

  // the buffers other CTAs add into are zeroed first; the matching wait comes after the
  // pooling below, so the cluster barrier's latency hides behind it
  if (threadIdx.x < kMaxHeads) S.head_cnt[threadIdx.x] = 0;
  for (int i = threadIdx.x; i < 3 * kBins; i += kThreads) (&S.merged[0][0])[i] = 0;
  for (int i = threadIdx.x; i < kWarps * kBins; i += kThreads) (&S.whist[0][0])[i] = 0;
  cluster_arrive_release();

  const bool pool_mode = a.raw != nullptr;
  // stage-2 scores: the value-aware score this kernel writes, or the caller's array
  // (value-aware scores computed earlier, or the anchors' random keys)
  const float* s2 = (pool_mode && a.out_val) ? a.out_val : a.s2;
  // when a thread owns at most kBatch entries, its stage-2 keys stay in registers
  const bool k2_reg = a.two_stage && cnt <= kBatch * kThreads;
  uint32_t k2[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) k2[u] = 0u;
  if (pool_mode) {
    // stage the raw scores of positions [c_lo - half, c_hi + half) at index
    // (position - c_lo + half), every copy in flight at once.  Then each thread pools its
    // kBatch entries of a round (entry e = r0 + u*kThreads + tid) in registers, all window
    // taps interleaved; a round reads staged indices [r0, r0 + R + 2*half) and, after a
    // barrier, writes the keys [r0, r0 + R), which no later round reads.
    const int half = a.pool != 0 ? a.pool_kernel / 2 : 0;
    const int lo = max(0, c_lo - half), hi = min(L, c_hi + half);
    float* stage = reinterpret_cast<float*>(keys);
    for (int x = lo + static_cast<int>(threadIdx.x); x < hi; x += kThreads)
      cp_async4(stage + (x - c_lo + half), a.raw + sbase + x);
    cp_async_wait_all();
    __syncthreads();
    for (int r0 = 0; r0 < cnt; r0 += kBatch * kThreads) {
      float nuv[kBatch], p[kBatch];
      int wlo[kBatch], whi[kBatch], pos[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = r0 + u * kThreads + static_cast<int>(threadIdx.x);
        const int g = c_lo + e;
        int i = g;
        if (per_layer) i = g % n;
        pos[u] = i;
        // window offsets inside the entry's own head; an empty window past the chunk
        wlo[u] = e < cnt ? max(0, i - half) - i : 1;
        whi[u] = e < cnt ? min(n - 1, i + half) - i : 0;
        // nu for the value-aware score, else the caller's stage-2 score
        nuv[u] = (e < cnt && (a.out_val || k2_reg)) ? __ldg((a.out_val ? a.nu : a.s2) + sbase + g) : 0.f;
        p[u] = (a.pool == 1) ? -INFINITY : 0.f;
      }
      if (a.pool == 0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = r0 + u * kThreads + static_cast<int>(threadIdx.x);
          if (e < cnt) p[u] = stage[e + half];
        }
      } else {
        for (int d = -half; d <= half; ++d) {
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int e = r0 + u * kThreads + static_cast<int>(threadIdx.x);
            if (d >= wlo[u] && d <= whi[u]) {
              const float x = stage[e + half + d];
              p[u] = (a.pool == 1) ? fmaxf(p[u], x) : p[u] + x;
            }
          }
        }
        if (a.pool == 2) {
#pragma unroll
          for (int u = 0; u < kBatch; ++u) p[u] = p[u] / static_cast<float>(a.pool_kernel);
        }
      }
      uint32_t key[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = r0 + u * kThreads + static_cast<int>(threadIdx.x);
        key[u] = 0u;
        if (e < cnt) {
          const int g = c_lo + e;
          a.out_attn[sbase + g] = p[u];
          if (a.out_val) {
            const float sv = (p[u] + a.eps) * nuv[u];
            a.out_val[sbase + g] = sv;
            k2[u] = f2key(sv);
          } else if (k2_reg) {
            k2[u] = f2key(nuv[u]);
          }
          const bool forced = (pos[u] < ns) || (pos[u] >= n - nr);
          key[u] = forced ? kKeyMax : f2key(p[u]);
        }
      }
      __syncthreads();   // this round's staged values are read
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = r0 + u * kThreads + static_cast<int>(threadIdx.x);
        if (e < cnt) {
          keys[e] = key[u];
          flag[e] = 0;
        }
      }
    }
  } else {
    for (int e0 = 0; e0 < cnt; e0 += kBatch * kThreads) {
      float v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads + static_cast<int>(threadIdx.x);
        v[u] = e < cnt ? __ldg(a.s1 + sbase + c_lo + e) : 0.f;
        if (k2_reg) k2[u] = e < cnt ? f2key(__ldg(s2 + sbase + c_lo + e)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads + static_cast<int>(threadIdx.x);
        if (e < cnt) {
          const int g = c_lo + e;
          int i = g;
          if (per_layer) i = g % n;
          const bool forced = (i < ns) || (i >= n - nr);
          keys[e] = forced ? kKeyMax : f2key(v[u]);
          flag[e] = 0;
        }
      }
    }
  }

  SelState sst;
  cluster_wait_acquire();   // every CTA's buffers are zero before any remote reduction lands
  __syncthreads();          // the keys built above are visible to every thread

  uint32_t T, krem;
  if (!per_layer) {
    // the segment's budget: fixed per request, or set on the device by an earlier
    // per-layer selection (its per-head counts and offsets)
    uint32_t B = static_cast<uint32_t>(a.budget[b]);
    uint32_t B1 = static_cast<uint32_t>(a.budget1[b]);
    long long out0 = a.seg_out[b] + static_cast<long long>(h0) * B;
    if (a.dev_counts) {
      const int c = __ldg(a.dev_counts + seg);
      B = static_cast<uint32_t>(min(max(c, 0), n));
      out0 = __ldg(a.dev_offsets + seg);
      long long b1 = static_cast<long long>(floor(static_cast<double>(a.alpha) * static_cast<double>(B)));
      B1 = static_cast<uint32_t>(max(b1, static_cast<long long>(nforced)));
    }
    if (a.two_stage) {
      // stage 1: b' = max(floor(alpha*B), |F|) entries by the attention score.  Without
      // ties to resolve (krem == 0, the usual case) the picks are exactly the keys above T
      // and need no ordered pass; otherwise they are flagged in index order.
      radix_select(cl, S, sst, keys, cnt, B1, T, krem);
      const bool by_threshold = (krem == 0u);
      if (!by_threshold)
        apply_selection(cl, S, sst, keys, 0, cnt, T, krem, [&](int e, uint32_t) { flag[e] = 1; });
      // stage 2: the remaining B - b' by the value-aware score, stage-1 picks forced in
      if (k2_reg) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = u * kThreads + static_cast<int>(threadIdx.x);
          if (e < cnt) keys[e] = (by_threshold ? keys[e] > T : flag[e] != 0) ? kKeyMax : k2[u];
        }
      } else {
        // each thread reads back only values it wrote itself, so plain loads see them
        for (int e0 = 0; e0 < cnt; e0 += kBatch * kThreads) {
          float v[kBatch];
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kThreads + threadIdx.x;
            v[u] = e < cnt ? (pool_mode ? s2[sbase + c_lo + e] : __ldg(s2 + sbase + c_lo + e)) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + u * kThreads + threadIdx.x;
            if (e < cnt) keys[e] = (by_threshold ? keys[e] > T : flag[e] != 0) ? kKeyMax : f2key(v[u]);
          }
        }
      }
      __syncthreads();
    }
    radix_select(cl, S, sst, keys, cnt, B, T, krem);
    apply_selection(cl, S, sst, keys, 0, cnt, T, krem, [&](int e, uint32_t slot) {
      if (slot < B) a.idx[out0 + slot] = c_lo + e;
    });
    if (rank == 0 && threadIdx.x == 0 && !a.dev_counts) {
      a.counts[seg] = static_cast<int32_t>(B);
      a.offsets[seg] = out0;
    }
  } else {
    // per-head floors: every head first keeps its forced entries plus its own top
    // entries up to the floor; those picks are then forced into the layer-wide top.
    const int fh = min(n, max(a.floor_h[b], nforced));
    if (fh > nforced) {
      for (int hh = 0; hh < H; ++hh) {
        const int lo = min(max(hh * n - c_lo, 0), cnt);
        const int hi = min(max((hh + 1) * n - c_lo, 0), cnt);
        radix_select(cl, S, sst, keys + lo, hi - lo, static_cast<uint32_t>(fh), T, krem);
        apply_selection(cl, S, sst, keys, lo, hi, T, krem, [&](int e, uint32_t) { flag[e] = 1; });
      }
      for (int e = threadIdx.x; e < cnt; e += kThreads)
        if (flag[e]) keys[e] = kKeyMax;
      __syncthreads();
    }
    const uint32_t BL = static_cast<uint32_t>(a.budget[b]);
    radix_select(cl, S, sst, keys, cnt, BL, T, krem);
    const long long out0 = a.seg_out[b];
    int cur_h = -1;
    uint32_t cur_c = 0;
    apply_selection(cl, S, sst, keys, 0, cnt, T, krem, [&](int e, uint32_t slot) {
      const int g = c_lo + e;
      const int hh = g / n;
      if (slot < BL) a.idx[out0 + slot] = g - hh * n;
      if (hh != cur_h) {
        if (cur_c) atomicAdd(&S.head_cnt[cur_h], cur_c);
        cur_h = hh;
        cur_c = 0;
      }
      ++cur_c;
    });
    if (cur_c) atomicAdd(&S.head_cnt[cur_h], cur_c);
    __syncthreads();
    cl.sync();
    if (rank == 0 && threadIdx.x == 0) {
      long long off = out0;
      for (int hh = 0; hh < H; ++hh) {
        uint32_t c = 0;
        for (unsigned r = 0; r < CS; ++r) c += cl.map_shared_rank(&S.head_cnt[0], r)[hh];
        a.counts[b * H + hh] = static_cast<int32_t>(c);
        a.offsets[b * H + hh] = off;
        off += c;
      }
    }
  }
  // per-layer mode: rank 0 has just read the other CTAs' head counts, so no CTA leaves
  // before it is done.  Per-head mode makes no remote access after the apply step's own
  // cluster barrier, so its CTAs may leave at once.
  if (per_layer) cl.sync();
}

size_t select_smem(int chunk_cap) {
  return ((sizeof(SelShared) + 15) & ~static_cast<size_t>(15)) + static_cast<size_t>(chunk_cap + kMaxHalo) * 5 + 16;
}

}  // namespace

// Cluster size for `segments` segments of at most `max_len` entries.  Alone on the
// device (min_cs = 0): the largest of 16 / 8 CTAs whose clusters all fit on the device
// at once (a cluster must sit inside one GPC), else the one that keeps the most CTAs busy
// in the first wave.  Beside other work (min_cs = 2 or 4): the smallest of min_cs,
// 2 min_cs, ... 16 CTAs whose staging fits in shared memory.  A cluster spends most of its
// time in cluster barriers, so with other calls in flight fewer, longer-running CTAs leave
// more SMs to them: a 4-CTA cluster per head holds half the SM time of an 8-CTA one for
// about 17% more latency.
int select_cluster_size_uncached(int max_len, int segments, int min_cs, int* chunk_cap);

int select_cluster_size(int max_len, int segments, int min_cs, int* chunk_cap) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, std::pair<int, int>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, max_len, segments, min_cs);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *chunk_cap = it->second.second;
      return it->second.first;
    }
  }
  int cap = 0;
  const int cs = select_cluster_size_uncached(max_len, segments, min_cs, &cap);
  if (cs > 0) {
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = std::make_pair(cs, cap);
    *chunk_cap = cap;
  }
  return cs;
}

int select_cluster_size_uncached(int max_len, int segments, int min_cs, int* chunk_cap) {
  const size_t limit = 232448 - 1024;
  int best_cs = -1, best_cap = 0;
  long long best_busy = -1;
  const bool small = min_cs > 0;
  int order[4] = {16, 8, 0, 0};
  int n_order = 2;
  if (small) {
    n_order = 0;
    for (int cs = min_cs; cs <= 16; cs *= 2) order[n_order++] = cs;
  }
  for (int i = 0; i < n_order; ++i) {
    const int cs = order[i];
    const int cap = (max_len + cs - 1) / cs;
    const int cap16 = ((cap + 15) & ~15) > 16 ? ((cap + 15) & ~15) : 16;
    const size_t smem = select_smem(cap16);
    if (smem > limit) continue;
    // raise (never lower) the kernel's shared-memory limit through the shared cache: a
    // lower limit set here would fail later launches that the cache thinks are covered
    if (ensure_smem(reinterpret_cast<const void*>(select_kernel), smem) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    if (cs > 8 && cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      continue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, select_kernel, &cfg) != cudaSuccess || active < 1) {
      cudaGetLastError();
      continue;
    }
    if (small || active >= segments) {   // the first that fits (small), or all segments at once
      *chunk_cap = cap16;
      return cs;
    }
    const long long busy = static_cast<long long>(active) * cs;
    if (busy > best_busy) {
      best_busy = busy;
      best_cs = cs;
      best_cap = cap16;
    }
  }
  if (best_cs > 0) *chunk_cap = best_cap;
  return best_cs;
}

cudaError_t launch_select(const SelectArgs& a, int cluster, int chunk_cap, cudaStream_t st) {
  const size_t smem = select_smem(chunk_cap);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  const int segs = (a.mode == 1) ? a.rq.B : a.rq.B * a.rq.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, segs, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, select_kernel, a, chunk_cap);
  if (e == cudaSuccess) note_launch();
  return e;
}

}  // namespace kvsel
