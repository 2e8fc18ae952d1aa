// Top-B selection with forced entries, on one thread-block cluster per segment
// ("CriticalKV: 출력 섭동 관점에서 KV 캐시 축출을 최적화하기", §3.4 Algorithm 1 (two stages:
//  b' = floor(alpha*b) by attention, the rest by the value-aware criterion) and
//  Algorithm 2 (Top_k of the pooled score); "KVzip: Query-Agnostic KV Cache Compression
//  with Context Reconstruction", §4.2 (top r% across all heads of a layer)).
//
// A segment is one (request, KV head) in per-head mode, or all heads of one request
// flattened head-major in per-layer mode.  The CTAs of a cluster split the segment into
// contiguous chunks held in shared memory as order-preserving 32-bit keys (forced
// entries get the largest key).  The B-th largest key T is found by a three-pass radix
// select (11/11/10-bit digits): each pass builds per-CTA histograms of the candidates,
// the cluster reduces them through distributed shared memory, and every CTA finds the
// same digit.  Entries with key > T, and the first (B - #greater) entries equal to T in
// index order, are kept; a cluster-wide exclusive scan of per-CTA counts plus a block
// scan gives each kept entry its output slot, so indices come out ascending.
#include <cooperative_groups.h>

#include "internal.cuh"

namespace cgx = cooperative_groups;

namespace kvsel {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr uint32_t kKeyMax = 0xFFFFFFFFu;
constexpr int kMaxHeads = 64;

__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
  uint32_t hist[kBins];       // local histogram of the current pass
  uint32_t mslice[kBins];     // merged bins owned by this CTA (first kBins / cluster)
  uint32_t slice_total;
  uint32_t cnt_gt, cnt_eq;    // local counts for the current selection
  uint32_t res_prefix, res_krem;
  uint32_t wsum_gt[kWarps], wsum_eq[kWarps];
  uint32_t head_cnt[kMaxHeads];
};

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

// Find the key T of the K-th largest candidate among elements [lo, hi) of the segment
// (local chunk positions given by my_lo/my_hi, already intersected), and how many keys
// equal to T are taken (krem).  Candidates: keys[] in shared memory.
__device__ void radix_select(cgx::cluster_group& cl, SelShared& S, const uint32_t* keys, int cnt_local, uint32_t K,
                            uint32_t& T, uint32_t& krem_out) {
  const unsigned CS = cl.num_blocks();
  const unsigned rank = cl.block_rank();
  const int slice = kBins / static_cast<int>(CS);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t prefix = 0, mask = 0, krem = K;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    for (int i = threadIdx.x; i < kBins; i += kThreads) S.hist[i] = 0;
    __syncthreads();
    const int trips = (cnt_local + kThreads - 1) / kThreads;
    for (int j = 0; j < trips; ++j) {
      const int e = j * kThreads + threadIdx.x;
      uint32_t dig = 0xFFFFFFFFu;
      if (e < cnt_local) {
        const uint32_t k = keys[e];
        if ((k & mask) == prefix) dig = (k >> sh) & dmask;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, dig);
      if (dig != 0xFFFFFFFFu && lane == __ffs(peers) - 1) atomicAdd(&S.hist[dig], static_cast<uint32_t>(__popc(peers)));
    }
    cl.sync();
    // reduce my slice of bins over the cluster
    uint32_t my_tot = 0;
    for (int i = threadIdx.x; i < slice; i += kThreads) {
      const int bin = static_cast<int>(rank) * slice + i;
      uint32_t s = 0;
      for (unsigned c = 0; c < CS; ++c) s += cl.map_shared_rank(&S.hist[0], c)[bin];
      S.mslice[i] = s;
      my_tot += s;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my_tot += __shfl_xor_sync(0xffffffffu, my_tot, o);
    if (threadIdx.x == 0) S.slice_total = 0;
    __syncthreads();
    if (lane == 0 && my_tot) atomicAdd(&S.slice_total, my_tot);
    cl.sync();
    // every CTA locates the digit (warp 0)
    if (w == 0) {
      // slice totals, highest slice first
      uint32_t tot = (lane < static_cast<int>(CS)) ? cl.map_shared_rank(&S.slice_total, lane)[0] : 0u;
      // suffix sums over slices: sum of totals of slices > lane
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += x;
      }
      const uint32_t above = incl - tot;  // sum over slices with index > lane
      const bool hit = (lane < static_cast<int>(CS)) && above < krem && krem <= incl;
      const unsigned hm = __ballot_sync(0xffffffffu, hit);
      const int cs = __ffs(hm) - 1;       // exactly one slice qualifies
      const uint32_t above_s = __shfl_sync(0xffffffffu, above, cs < 0 ? 0 : cs);
      uint32_t kr = krem - above_s;
      // bins of slice cs, highest first: lane l holds bins [l*per, (l+1)*per)
      const int per = slice / 32;
      const uint32_t* rb = cl.map_shared_rank(&S.mslice[0], cs < 0 ? 0 : cs);
      uint32_t loc[8];
      uint32_t lsum = 0;
      for (int i = 0; i < per; ++i) {
        loc[i] = rb[lane * per + i];
        lsum += loc[i];
      }
      uint32_t lincl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_down_sync(0xffffffffu, lincl, o);
        if (lane + o < 32) lincl += x;
      }
      const uint32_t labove = lincl - lsum;
      const bool lhit = labove < kr && kr <= lincl;
      const unsigned lm = __ballot_sync(0xffffffffu, lhit);
      const int ls = __ffs(lm) - 1;
      if (lane == ls) {
        uint32_t cum = labove;
        int digit = lane * per;
        for (int i = per - 1; i >= 0; --i) {
          if (cum + loc[i] >= kr) {
            digit = lane * per + i;
            break;
          }
          cum += loc[i];
        }
        S.res_prefix = prefix | (static_cast<uint32_t>(cs * slice + digit) << sh);
        S.res_krem = kr - cum;
      }
    }
    __syncthreads();
    prefix = S.res_prefix;
    krem = S.res_krem;
    mask |= dmask << sh;
    __syncthreads();
  }
  T = prefix;
  krem_out = krem;
}

// Walk the local chunk in index order and visit every kept entry with its slot in the
// segment-wide ascending order.  Returns nothing; `visit(e_local, slot)`.
template <typename Visit>
__device__ void apply_selection(cgx::cluster_group& cl, SelShared& S, const uint32_t* keys, int lo_local,
                                int hi_local, uint32_t T, uint32_t krem, Visit visit) {
  const unsigned CS = cl.num_blocks();
  const unsigned rank = cl.block_rank();
  const int lane = threadIdx.x & 31;
  const int cnt = hi_local - lo_local;
  const int per = cnt > 0 ? (cnt + kThreads - 1) / kThreads : 0;
  const int a = lo_local + min(cnt, static_cast<int>(threadIdx.x) * per);
  const int b = lo_local + min(cnt, static_cast<int>(threadIdx.x + 1) * per);
  uint32_t ngt = 0, neq = 0;
  for (int e = a; e < b; ++e) {
    const uint32_t k = keys[e];
    ngt += (k > T);
    neq += (k == T);
  }
  uint32_t egt, eeq, tgt, teq;
  block_excl_scan2(S, ngt, neq, egt, eeq, tgt, teq);
  if (threadIdx.x == 0) {
    S.cnt_gt = tgt;
    S.cnt_eq = teq;
  }
  cl.sync();
  // cluster exclusive prefix over CTA ranks
  uint32_t base_out = 0, eq_base = 0;
  {
    uint32_t g = 0, q = 0;
    if (lane < static_cast<int>(CS) && lane < static_cast<int>(rank)) {
      g = cl.map_shared_rank(&S.cnt_gt, lane)[0];
      q = cl.map_shared_rank(&S.cnt_eq, lane)[0];
    }
    // eq_base of each lower CTA is needed to know how many of its equals were taken;
    // compute prefix of q across lanes
    uint32_t qincl = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, qincl, o);
      if (lane >= o) qincl += x;
    }
    const uint32_t qexcl = qincl - q;
    const uint32_t avail = krem > qexcl ? krem - qexcl : 0u;
    const uint32_t take = q < avail ? q : avail;
    uint32_t sel = g + take;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, o);
    uint32_t qs = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
    base_out = sel;
    eq_base = qs;
  }
  // equals taken before this thread
  const uint32_t avail_cta = krem > eq_base ? krem - eq_base : 0u;
  const uint32_t taken_before = eeq < avail_cta ? eeq : avail_cta;
  uint32_t slot = base_out + egt + taken_before;
  uint32_t eq_rank = eq_base + eeq;
  for (int e = a; e < b; ++e) {
    const uint32_t k = keys[e];
    bool take = false;
    if (k > T) {
      take = true;
    } else if (k == T) {
      take = eq_rank < krem;
      ++eq_rank;
    }
    if (take) visit(e, slot++);
  }
  cl.sync();   // counters are reused by the next selection
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const SelectArgs a, int chunk_cap) {
  cgx::cluster_group cl = cgx::this_cluster();
  extern __shared__ uint8_t smem_raw[];
  SelShared& S = *reinterpret_cast<SelShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(SelShared) + 15) & ~static_cast<size_t>(15)));
  uint8_t* flag = reinterpret_cast<uint8_t*>(keys + chunk_cap);

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

  // stage-1 keys (forced entries at the top)
  for (int e = threadIdx.x; e < cnt; e += kThreads) {
    const int g = c_lo + e;
    const int i = per_layer ? g % n : g;
    const bool forced = (i < ns) || (i >= n - nr);
    keys[e] = forced ? kKeyMax : f2key(__ldg(a.s1 + sbase + g));
    flag[e] = 0;
  }
  if (threadIdx.x < kMaxHeads) S.head_cnt[threadIdx.x] = 0;
  __syncthreads();

  uint32_t T, krem;
  if (!per_layer) {
    const uint32_t B = static_cast<uint32_t>(a.budget[b]);
    if (a.two_stage) {
      // stage 1: b' = max(floor(alpha*B), |F|) entries by the attention score
      radix_select(cl, S, keys, cnt, static_cast<uint32_t>(a.budget1[b]), T, krem);
      apply_selection(cl, S, keys, 0, cnt, T, krem, [&](int e, uint32_t) { flag[e] = 1; });
      // stage 2: the remaining B - b' by the value-aware score, stage-1 picks forced in
      for (int e = threadIdx.x; e < cnt; e += kThreads)
        keys[e] = flag[e] ? kKeyMax : f2key(__ldg(a.s2 + sbase + c_lo + e));
      __syncthreads();
    }
    radix_select(cl, S, keys, cnt, B, T, krem);
    const long long out0 = a.seg_out[b] + static_cast<long long>(h0) * B;
    apply_selection(cl, S, keys, 0, cnt, T, krem, [&](int e, uint32_t slot) {
      if (slot < B) a.idx[out0 + slot] = c_lo + e;
    });
    if (rank == 0 && threadIdx.x == 0) {
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
        radix_select(cl, S, keys + lo, hi - lo, static_cast<uint32_t>(fh), T, krem);
        apply_selection(cl, S, keys, lo, hi, T, krem, [&](int e, uint32_t) { flag[e] = 1; });
      }
      for (int e = threadIdx.x; e < cnt; e += kThreads)
        if (flag[e]) keys[e] = kKeyMax;
      __syncthreads();
    }
    const uint32_t BL = static_cast<uint32_t>(a.budget[b]);
    radix_select(cl, S, keys, cnt, BL, T, krem);
    const long long out0 = a.seg_out[b];
    int cur_h = -1;
    uint32_t cur_c = 0;
    apply_selection(cl, S, keys, 0, cnt, T, krem, [&](int e, uint32_t slot) {
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
  cl.sync();   // no CTA leaves while others may still read its shared memory
}

size_t select_smem(int chunk_cap) {
  return ((sizeof(SelShared) + 15) & ~static_cast<size_t>(15)) + static_cast<size_t>(chunk_cap) * 5 + 16;
}

}  // namespace

int select_cluster_size(int max_len, int* chunk_cap) {
  const size_t limit = 232448 - 1024;
  for (int cs = 16; cs >= 8; cs >>= 1) {
    const int cap = (max_len + cs - 1) / cs;
    const int cap16 = ((cap + 15) & ~15) > 16 ? ((cap + 15) & ~15) : 16;
    const size_t smem = select_smem(cap16);
    if (smem > limit) continue;
    // the cluster must be schedulable on this device with that much shared memory
    if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      continue;
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
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, select_kernel, &cfg) != cudaSuccess || nclusters < 1) {
      cudaGetLastError();
      continue;
    }
    *chunk_cap = cap16;
    return cs;
  }
  return -1;
}

cudaError_t launch_select(const SelectArgs& a, int cluster, int chunk_cap, cudaStream_t st) {
  const size_t smem = select_smem(chunk_cap);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
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
  return e;
}

}  // namespace kvsel
